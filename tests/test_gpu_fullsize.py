"""Parity at the workloads' full sizes, in the launch configuration the bench uses.

The whole cache is built on the GPU (automatic split count, as bench.py runs
it); the oracle recomputes a sample of (batch, kv head) units one by one from
the same host inputs.  Sampled units must match bit for bit (codes, zero
points, scales, sparse entries, window) and their query heads' attention must
be within 2e-3.  Units are sampled at both ends of the batch and head ranges.
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


def _check_unit(cache, w, K, V, b, kvh, T, q_list, outs, label):
    """Oracle for unit (b, kvh): prefill, then the appends; compare stores and every checked output."""
    T0 = w.prefill_tokens
    u = oracle.OracleUnit.for_workload(w)
    u.prefill(K[b, kvh, :T0], V[b, kvh, :T0])
    hs = slice(kvh * w.group_q, (kvh + 1) * w.group_q)
    worst = 0.0
    for step in range(T - T0):
        u.append(K[b, kvh, T0 + step], V[b, kvh, T0 + step])
        if step in outs:
            ref = u.attention(q_list[step][b, hs], w.softmax_scale)
            err = oracle.max_rel_err(outs[step][b, hs].astype(np.float64), ref)
            worst = max(worst, err)
            assert err <= TOL, f"{label} unit ({b},{kvh}) step {step}: attention error {err:.3e}"
    got = cache.export_unit(b, kvh)
    ref = u.stores()
    for key in ref:
        assert got[key].shape == ref[key].shape, (label, key)
        assert np.array_equal(got[key], ref[key]), f"{label} unit ({b},{kvh}): {key} differs"
    return worst


def _run(widx, steps, check_steps, units):
    import bit_asymmetric_kv_kvq_gb300 as kvq
    w = synth.WORKLOADS[widx]
    T0 = w.prefill_tokens
    K = synth.keys(w)
    V = synth.values(w)
    cache = kvq.KVCache.for_workload(w)
    cache.prefill_quantize(_dev(K[:, :, :T0]), _dev(V[:, :, :T0]))
    q_list, outs = [], {}
    for step in range(steps):
        cache.append(_dev(K[:, :, T0 + step]), _dev(V[:, :, T0 + step]))
        if w.queries == "peaked":
            q = synth.queries(w, step, keys_of=lambda b, h: K[b, h, :T0 + step + 1])
        else:
            q = synth.queries(w, step)
        q_list.append(q)
        out = cache.decode_attention(_dev(q))
        if step in check_steps:
            outs[step] = out.cpu().numpy()
    assert cache.sync_status() == 0
    worst = 0.0
    for (b, kvh) in units:
        worst = max(worst, _check_unit(cache, w, K, V, b, kvh, T0 + steps, q_list, outs, f"workload {widx}"))
    print(f"workload {widx}: splits {cache.splits()}, worst sampled attention error {worst:.2e}")
    cache.close()


def test_llama2_7b_shape_full():
    w = synth.WORKLOADS[1]
    _run(1, w.decode_steps, {0, 1, 31, 63}, [(0, 0), (3, 17), (w.batch - 1, w.kv_heads - 1)])


def test_llama2_13b_k4v2_full():
    w = synth.WORKLOADS[2]
    _run(2, 1, {0}, [(0, 0), (w.batch - 1, w.kv_heads - 1)])


def test_llama3_8b_gqa_full():
    w = synth.WORKLOADS[3]
    _run(3, 1, {0}, [(0, 0), (17, 5), (w.batch - 1, w.kv_heads - 1)])


def test_long_context_rope_sparse_full():
    w = synth.WORKLOADS[4]
    _run(4, 1, {0}, [(0, w.kv_heads - 1)])
