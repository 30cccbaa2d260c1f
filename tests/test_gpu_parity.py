"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

Packed codes, zero points, scales, sparse entries and the fp16 window must be
bit-identical to the oracle's (exported in the canonical layout); decode
attention must be within a max relative error of 2e-3 (per query head,
||o - o*||_inf / ||o*||_inf) of the oracle's fp64 attention over its own,
bit-identical cache.  Cases are oracle-sized versions of the five workloads
(several pages, a ragged window) plus edge cases.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _kvq():
    import bit_asymmetric_kv_kvq_gb300 as kvq
    return kvq


def compare_stores(cache, units, b, kvh, where=""):
    got = cache.export_unit(b, kvh)
    ref = units[(b, kvh)].stores()
    for key in ref:
        assert got[key].shape == ref[key].shape, (where, key, got[key].shape, ref[key].shape)
        if not np.array_equal(got[key], ref[key]):
            bad = np.argwhere(got[key] != ref[key])
            raise AssertionError(f"{where}: {key} differs at {bad[:5].tolist()} ({len(bad)} entries)")


def check_attention(w, units, q, out, where=""):
    out = out.float().cpu().numpy().astype(np.float64)
    worst = 0.0
    for (b, kvh), u in units.items():
        hs = slice(kvh * w.group_q, (kvh + 1) * w.group_q)
        ref = u.attention(q[b, hs], w.softmax_scale)
        err = oracle.max_rel_err(out[b, hs], ref)
        worst = max(worst, err)
        assert err <= TOL, f"{where}: unit ({b},{kvh}) attention error {err:.3e}"
    return worst


def run_case(w, steps, check_every=1, splits=0, sample_units=None):
    """Prefill, then `steps` x (append, decode), checking stores and outputs against the oracle."""
    kvq = _kvq()
    K = synth.keys(w)
    V = synth.values(w)
    T0 = w.prefill_tokens
    cache = kvq.KVCache.for_workload(w)
    if splits:
        cache.set_splits(splits)
    cache.prefill_quantize(_dev(K[:, :, :T0]), _dev(V[:, :, :T0]))
    all_units = [(b, h) for b in range(w.batch) for h in range(w.kv_heads)]
    sel = all_units if sample_units is None else sample_units
    units = {}
    for (b, h) in sel:
        u = oracle.OracleUnit.for_workload(w)
        u.prefill(K[b, h, :T0], V[b, h, :T0])
        units[(b, h)] = u
    assert cache.state() == (T0, oracle.quantized_tokens(T0, w.residual), T0 - oracle.quantized_tokens(T0, w.residual))
    for (b, h) in sel:
        compare_stores(cache, units, b, h, "prefill")
    worst = 0.0
    for step in range(steps):
        t = T0 + step
        cache.append(_dev(K[:, :, t]), _dev(V[:, :, t]))
        for (b, h) in sel:
            units[(b, h)].append(K[b, h, t], V[b, h, t])
        q = synth.queries(w, step)
        out = cache.decode_attention(_dev(q))
        assert cache.sync_status() == 0
        if step % check_every == 0 or step == steps - 1:
            for (b, h) in sel:
                compare_stores(cache, units, b, h, f"step {step}")
            worst = max(worst, check_attention(w, units, q, out, f"step {step}"))
    cache.close()
    return worst


# oracle-sized versions of the five workloads: several pages, a ragged window, a flush mid-run
CASES = {
    "tiny-mha-2bit": (synth.WORKLOADS[0], 1),
    "llama2-7b-shape": (synth.WORKLOADS[1].scaled(batch=2, kv_heads=4, q_heads=4, prefill_tokens=1000,
                                                  decode_steps=40), 40),
    "llama2-13b-k4v2-peaked": (synth.WORKLOADS[2].scaled(batch=2, kv_heads=3, q_heads=3, prefill_tokens=700,
                                                         decode_steps=3), 3),
    "llama3-8b-gqa": (synth.WORKLOADS[3].scaled(batch=2, kv_heads=2, q_heads=8, prefill_tokens=1500,
                                                decode_steps=2), 2),
    "long-ctx-rope-sparse-k3v3": (synth.WORKLOADS[4].scaled(batch=1, kv_heads=2, q_heads=8, prefill_tokens=2100,
                                                            decode_steps=2), 2),
}


@pytest.mark.parametrize("name", list(CASES))
def test_workload_parity(name):
    w, steps = CASES[name]
    worst = run_case(w, steps, check_every=8)
    print(f"{name}: worst attention error {worst:.2e}")


@pytest.mark.parametrize("T0", [1, 31, 127, 128, 129, 256, 257])
def test_window_edges(T0):
    """Window-only caches, exactly full windows, and one token past a page boundary."""
    w = synth.WORKLOADS[0].scaled(batch=1, kv_heads=2, q_heads=2, prefill_tokens=T0, decode_steps=3)
    run_case(w, 3)


@pytest.mark.parametrize("hg,bk,bv", [(1, 4, 4), (2, 2, 2), (2, 4, 2), (4, 4, 4), (1, 3, 3), (2, 3, 3)])
def test_other_bit_widths_and_groups(hg, bk, bv):
    w = synth.WORKLOADS[1].scaled(batch=1, kv_heads=2, q_heads=2 * hg, prefill_tokens=600, decode_steps=2,
                                  k_bits=bk, v_bits=bv)
    run_case(w, 2)


@pytest.mark.parametrize("G,nsp,rope", [(64, 0, 0), (64, 1, 0), (32, 2, 0), (32, 4, 1), (64, 0, 1)])
def test_group_sparse_rope_variants(G, nsp, rope):
    w = synth.WORKLOADS[4].scaled(batch=1, kv_heads=2, q_heads=2, prefill_tokens=900, decode_steps=2,
                                  group=G, k_sparse=nsp, rope=rope, k_bits=2, v_bits=2)
    run_case(w, 2)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 1000])
def test_split_counts_agree(splits):
    """Any split count (including more splits than pages) gives the same answer within tolerance."""
    w = synth.WORKLOADS[3].scaled(batch=1, kv_heads=2, q_heads=8, prefill_tokens=1300, decode_steps=1)
    run_case(w, 1, splits=splits)


@pytest.mark.parametrize("bits,q_heads", [((2, 2), 4), ((4, 2), 4), ((4, 4), 1)],
                         ids=["k2v2-4heads-13-stages", "k4v2-4heads-10-stages", "k4v4-1head-10-stages"])
def test_page_ring_wraps_many_times(bits, q_heads):
    """One CTA streams the 100 pages of one unit through its page ring: the ring's stage counts that
    are not powers of two (13 stages of 12 KB pages beside four query heads' buffers, 10 of 16 KB or
    20 KB pages) wrap around seven to ten times within one launch."""
    w = synth.WORKLOADS[3].scaled(batch=1, kv_heads=1, q_heads=q_heads, prefill_tokens=100 * 128 + 3,
                                  decode_steps=1, k_bits=bits[0], v_bits=bits[1])
    run_case(w, 1, splits=1)


def test_capacity_and_state_errors():
    kvq = _kvq()
    w = synth.WORKLOADS[0].scaled(batch=1, kv_heads=1, q_heads=1, prefill_tokens=5, decode_steps=1)  # capacity 6
    K = _dev(synth.keys(w))
    V = _dev(synth.values(w))
    q = _dev(synth.queries(w, 0))
    cache = kvq.KVCache.for_workload(w)
    with pytest.raises(kvq.KVQError) as e:
        cache.decode_attention(q)  # nothing cached yet
    assert e.value.status == kvq.kvq.KVQ_ERR_STATE
    cache.prefill_quantize(K[:, :, :5].contiguous(), V[:, :, :5].contiguous())
    with pytest.raises(kvq.KVQError) as e:
        cache.prefill_quantize(K[:, :, :5].contiguous(), V[:, :, :5].contiguous())
    assert e.value.status == kvq.kvq.KVQ_ERR_STATE
    cache.append(K[:, :, 5].contiguous(), V[:, :, 5].contiguous())
    with pytest.raises(kvq.KVQError) as e:
        cache.append(K[:, :, 5].contiguous(), V[:, :, 5].contiguous())
    assert e.value.status == kvq.kvq.KVQ_ERR_CAPACITY
    assert cache.state() == (6, 0, 6)
    # a misaligned device pointer is refused before any launch
    flat = torch.zeros(2 * 128 + 8, dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_decode_attention(cache.handle, flat.data_ptr() + 2, flat.data_ptr())
    assert e.value.status == kvq.kvq.KVQ_ERR_INVALID_ARG
    assert cache.sync_status() == 0
    cache.close()
    small = kvq.KVCache.for_workload(w, max_tokens=4)
    with pytest.raises(kvq.KVQError) as e:
        small.prefill_quantize(K[:, :, :5].contiguous(), V[:, :, :5].contiguous())
    assert e.value.status == kvq.kvq.KVQ_ERR_CAPACITY
    assert small.state() == (0, 0, 0)
    small.close()


def test_append_on_empty_cache_acts_as_prefill():
    kvq = _kvq()
    w = synth.WORKLOADS[0].scaled(batch=2, kv_heads=2, q_heads=2, prefill_tokens=0, decode_steps=200)
    K = synth.keys(w)
    V = synth.values(w)
    cache = kvq.KVCache.for_workload(w)
    units = {(b, h): oracle.OracleUnit.for_workload(w) for b in range(2) for h in range(2)}
    for t in range(200):
        cache.append(_dev(K[:, :, t]), _dev(V[:, :, t]))
        for (b, h), u in units.items():
            if t == 0:
                u.prefill(K[b, h, :1], V[b, h, :1])
            else:
                u.append(K[b, h, t], V[b, h, t])
        if t in (0, 127, 128, 129, 199):
            q = synth.queries(w, t)
            out = cache.decode_attention(_dev(q))
            for (b, h) in units:
                compare_stores(cache, units, b, h, f"t={t}")
            check_attention(w, units, q, out, f"t={t}")
    assert cache.state() == (200, 128, 72)
    cache.close()


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_quantizer_rounding_ties(bits):
    """Values exactly on half steps, and one fp16 ulp either side, quantize as the oracle's true division."""
    kvq = _kvq()
    L = 2 ** bits - 1
    D, R, G = 128, 128, 32
    T = R + 1
    rng = np.random.default_rng(bits)
    K = np.zeros((T, D), np.float64)
    V = np.zeros((T, D), np.float64)
    for c in range(D):
        z = float(rng.integers(-64, 64)) * 0.25
        s = [1.0, 0.5, 2.0, 0.125][c % 4]
        k = rng.integers(0, L, T)
        vals = z + s * (k + 0.5)                       # exact ties
        nudge = rng.integers(-1, 2, T)                 # -1, 0, +1 ulp
        vals = np.where(nudge == 0, vals, np.nextafter(vals.astype(np.float16), np.where(nudge > 0, np.inf, -np.inf)
                                                       ).astype(np.float64))
        vals[::G] = z                                  # every group holds its min and max
        vals[1::G] = z + s * L
        K[:, c] = vals
    for t in range(T):
        z = float(rng.integers(-64, 64)) * 0.25
        s = [1.0, 0.5, 0.25, 2.0][t % 4]
        k = rng.integers(0, L, D)
        vals = z + s * (k + 0.5)
        vals[::G] = z
        vals[1::G] = z + s * L
        V[t] = vals
    K16 = K.astype(np.float16).reshape(1, 1, T, D)
    V16 = V.astype(np.float16).reshape(1, 1, T, D)
    w = synth.WORKLOADS[0].scaled(batch=1, kv_heads=1, q_heads=1, prefill_tokens=T, decode_steps=1,
                                  k_bits=bits, v_bits=bits)
    cache = kvq.KVCache.for_workload(w)
    cache.prefill_quantize(_dev(K16), _dev(V16))
    u = oracle.OracleUnit.for_workload(w)
    u.prefill(K16[0, 0], V16[0, 0])
    compare_stores(cache, {(0, 0): u}, 0, 0, f"ties {bits}-bit")
    # the crafted values really do sit on ties: the oracle's codes are even there
    assert cache.sync_status() == 0
    cache.close()
