"""GPU parity of codebook caches (non-uniform levels, the nuqX datatype without its calibration).

KVQuant review, "Proposed method".  Stores (codes, zero points, scales, sparse entries, window)
must equal the oracle's bit for bit after the prefill and after every decode step, and the
attention must be within 2e-3 of the oracle's fp64 attention over its own cache, for every
configuration the codebook kernels serve (including pre-RoPE keys with sparse outliers), through
both the fused decode step and append + decode.  Host-side rules of kvq_set_codebooks are checked
too.
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


def levels(bits, kind):
    """Strictly increasing levels from 0 to L: denser near the ends ("edge") or the middle ("mid")."""
    L = (1 << bits) - 1
    u = np.arange(L + 1) / L
    if kind == "edge":
        f = 0.5 - 0.5 * np.cos(np.pi * u)
    else:
        f = 0.5 + 0.5 * np.sign(2 * u - 1) * np.abs(2 * u - 1) ** 1.7
    lev = (L * f).astype(np.float32)
    lev[0], lev[-1] = 0.0, float(L)
    assert np.all(np.diff(lev) > 0)
    return lev


CASES = [
    (1, dict(batch=2, kv_heads=4, q_heads=4, prefill_tokens=260), 5),                                  # K2V2, MHA
    (3, dict(batch=1, kv_heads=2, q_heads=8, prefill_tokens=300, k_bits=3, v_bits=3), 4),              # 3/3 GQA
    (2, dict(batch=2, kv_heads=2, q_heads=2, prefill_tokens=255, k_bits=4, v_bits=4, queries="normal"), 3),
    (2, dict(batch=1, kv_heads=2, q_heads=8, prefill_tokens=129, queries="normal"), 3),                # K4V2 GQA
    (4, dict(batch=1, kv_heads=2, q_heads=8, prefill_tokens=383), 4),                                  # pre-RoPE, sparse
]


@pytest.mark.parametrize("widx,kw,steps", CASES)
@pytest.mark.parametrize("kind", ["edge", "mid"])
def test_codebook_parity(widx, kw, steps, kind):
    import bit_asymmetric_kv_kvq_gb300 as kvq
    w = synth.WORKLOADS[widx].scaled(decode_steps=steps, **kw)
    kl, vl = levels(w.k_bits, kind), levels(w.v_bits, kind)
    K = synth.keys(w)
    V = synth.values(w)
    T0 = w.prefill_tokens
    cache = kvq.KVCache(w.batch, w.kv_heads, w.q_heads, w.head_dim, w.max_tokens, w.k_bits, w.v_bits, w.group,
                        w.residual, w.k_sparse, w.rope, w.rope_base, w.softmax_scale, 0, 0, kl, vl)
    cache.prefill_quantize(_dev(K[:, :, :T0]), _dev(V[:, :, :T0]))
    units = {}
    for b in range(w.batch):
        for h in range(w.kv_heads):
            u = oracle.OracleUnit(w.head_dim, w.k_bits, w.v_bits, w.group, w.residual, w.k_sparse, w.rope,
                                  w.rope_base, 0, kl, vl)
            u.prefill(K[b, h, :T0], V[b, h, :T0])
            units[(b, h)] = u

    def check(where, out=None, qn=None):
        for (b, h), u in units.items():
            got, ref = cache.export_unit(b, h), u.stores()
            for key in ref:
                assert np.array_equal(got[key], ref[key]), (where, b, h, key)
            if out is not None:
                hs = slice(h * w.group_q, (h + 1) * w.group_q)
                err = oracle.max_rel_err(out[b, hs], u.attention(qn[b, hs], w.softmax_scale))
                assert err <= TOL, (where, b, h, err)

    check("prefill")
    for step in range(steps):
        t = T0 + step
        qn = synth.queries(w, step)
        if step % 2 == 0:
            out = cache.decode_step(_dev(K[:, :, t]), _dev(V[:, :, t]), _dev(qn))
        else:
            cache.append(_dev(K[:, :, t]), _dev(V[:, :, t]))
            out = cache.decode_attention(_dev(qn))
        for (b, h), u in units.items():
            u.append(K[b, h, t], V[b, h, t])
        check(f"step {step}", out.cpu().numpy().astype(np.float64), qn)
    assert cache.sync_status() == 0
    cache.close()


def test_set_codebooks_rules():
    import bit_asymmetric_kv_kvq_gb300 as kvq
    from bit_asymmetric_kv_kvq_gb300.kvq import KVQ_ERR_INVALID_ARG, KVQ_ERR_STATE, KVQ_ERR_UNSUPPORTED
    w = synth.WORKLOADS[0].scaled(prefill_tokens=64, decode_steps=1)
    good = levels(2, "edge")

    def make(cb=1, **kw):
        cfg = kvq.make_config(1, 4, 4, 128, 65, 2, 2, 32, 128, codebook=cb, **kw)
        return kvq.kvq_create(cfg, 0)

    h = make()
    K = _dev(synth.keys(w)[:, :, :64])
    V = _dev(synth.values(w)[:, :, :64])
    with pytest.raises(kvq.KVQError) as e:  # no codebooks yet
        kvq.kvq_prefill_quantize(h, K, V, 64)
    assert e.value.status == KVQ_ERR_STATE
    for bad in ([0, 1, 1, 3], [0.5, 1, 2, 3], [0, 1, 2, 2.5], [0, 2, 1, 3]):
        with pytest.raises(kvq.KVQError) as e:
            kvq.kvq_set_codebooks(h, bad, good)
        assert e.value.status == KVQ_ERR_INVALID_ARG
    kvq.kvq_set_codebooks(h, good, good)
    kvq.kvq_prefill_quantize(h, K, V, 64)
    with pytest.raises(kvq.KVQError) as e:  # after the prefill
        kvq.kvq_set_codebooks(h, good, good)
    assert e.value.status == KVQ_ERR_STATE
    kvq.kvq_destroy(h)
    h = make(cb=0)
    with pytest.raises(kvq.KVQError) as e:  # a uniform cache
        kvq.kvq_set_codebooks(h, good, good)
    assert e.value.status == KVQ_ERR_INVALID_ARG
    kvq.kvq_destroy(h)
    with pytest.raises(kvq.KVQError) as e:  # 3-bit keys with 2-bit values: no codebook kernel
        kvq.kvq_create(kvq.make_config(1, 4, 4, 128, 65, 3, 2, 32, 128, codebook=1), 0)
    assert e.value.status == KVQ_ERR_UNSUPPORTED
