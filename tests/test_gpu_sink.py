"""GPU parity of the attention-sink tokens (the first S tokens kept fp16 beside the window).

unite.ai page and dothoosh.com page, research-direction sections (InnerQ).  Every case checks,
after the prefill and after every decode step, the exported stores of every unit (packed codes,
scales, zero points, sparse entries, window and sink rows) bit for bit against the oracle, and the
attention of every unit within 2e-3 of the oracle's fp64 attention.  Cases cover both decode
kernels (tensor-core pages; the CUDA-core kernel with pre-RoPE keys or 3-bit codes), prefills
shorter than the sink, a sink of R tokens (two fp16 items per unit), flushes, and both the fused
decode step and append + decode.
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


CASES = [
    # (workload, sizes and sink, decode steps)
    (1, dict(batch=2, kv_heads=4, q_heads=4, prefill_tokens=260, sink=4), 6),      # flush on the first step
    (3, dict(batch=1, kv_heads=2, q_heads=8, prefill_tokens=3, sink=8), 40),       # prefill shorter than the sink
    (0, dict(batch=1, kv_heads=4, q_heads=4, prefill_tokens=700, sink=128), 3),    # S = R: 2 fp16 items
    (4, dict(batch=1, kv_heads=2, q_heads=8, prefill_tokens=300, sink=4), 4),      # pre-RoPE, sparse, 3-bit
    (4, dict(batch=1, kv_heads=2, q_heads=8, prefill_tokens=520, sink=100, rope=0, k_sparse=0), 3),  # 3-bit
    (2, dict(batch=1, kv_heads=2, q_heads=2, prefill_tokens=33, sink=33), 2),      # K4V2, sink exactly full
]


@pytest.mark.parametrize("widx,kw,steps", CASES)
@pytest.mark.parametrize("fused", [True, False])
def test_sink_parity(widx, kw, steps, fused):
    import bit_asymmetric_kv_kvq_gb300 as kvq
    w = synth.WORKLOADS[widx].scaled(decode_steps=steps, **kw)
    K = synth.keys(w)
    V = synth.values(w)
    T0 = w.prefill_tokens
    cache = kvq.KVCache.for_workload(w)
    cache.prefill_quantize(_dev(K[:, :, :T0]), _dev(V[:, :, :T0]))
    units = {}
    for b in range(w.batch):
        for h in range(w.kv_heads):
            u = oracle.OracleUnit.for_workload(w)
            u.prefill(K[b, h, :T0], V[b, h, :T0])
            units[(b, h)] = u

    def check(where, out=None, qn=None):
        u0 = units[(0, 0)]
        assert cache.state() == (u0.T, u0.Tq, u0.n_r), where
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
        if fused:
            out = cache.decode_step(_dev(K[:, :, t]), _dev(V[:, :, t]), _dev(qn))
        else:
            cache.append(_dev(K[:, :, t]), _dev(V[:, :, t]))
            out = cache.decode_attention(_dev(qn))
        for (b, h), u in units.items():
            u.append(K[b, h, t], V[b, h, t])
        check(f"step {step}", out.cpu().numpy().astype(np.float64), qn)
    assert cache.sync_status() == 0
    cache.close()
