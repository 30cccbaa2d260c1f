"""kvq_decode_step against kvq_append followed by kvq_decode_attention.

The fused step must leave the same cache (bit for bit, checked through the export) and the same
attention, across a flush (the window full before the step) and for both decode kernels
(tensor-core pages and the rotated-key CUDA-core path).  Decode outputs are not bitwise
reproducible from launch to launch: warps claim partial slots as they finish and the merge sums
the slots in that order, so the two outputs are compared within 1e-3 (max relative error over a
head) and each is checked against the oracle's fp64 attention within 2e-3.
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


@pytest.mark.parametrize("widx,batch,kvh,qh,T0,steps", [
    (1, 2, 4, 4, 254, 5),    # 2-bit MHA, fragment-ordered pages: window 126 -> flush after 2 steps
    (3, 2, 2, 8, 255, 3),    # 4-way GQA: flush on the second step
    (4, 1, 2, 8, 383, 4),    # pre-RoPE 3-bit keys with sparse outliers (CUDA-core kernel)
])
def test_decode_step_equals_append_then_decode(widx, batch, kvh, qh, T0, steps):
    import bit_asymmetric_kv_kvq_gb300 as kvq
    w = synth.WORKLOADS[widx].scaled(batch=batch, kv_heads=kvh, q_heads=qh, prefill_tokens=T0, decode_steps=steps)
    K = synth.keys(w)
    V = synth.values(w)
    a = kvq.KVCache.for_workload(w)
    b = kvq.KVCache.for_workload(w)
    for c in (a, b):
        c.prefill_quantize(_dev(K[:, :, :T0]), _dev(V[:, :, :T0]))
    units = {}
    for bb in range(batch):
        for h in range(kvh):
            units[(bb, h)] = oracle.OracleUnit.for_workload(w)
            units[(bb, h)].prefill(K[bb, h, :T0], V[bb, h, :T0])
    for step in range(steps):
        k, v = _dev(K[:, :, T0 + step]), _dev(V[:, :, T0 + step])
        qn = synth.queries(w, step)
        q = _dev(qn)
        a.append(k, v)
        ref = a.decode_attention(q)
        got = b.decode_step(k, v, q)
        torch.cuda.synchronize()
        assert a.state() == b.state()
        ref = ref.cpu().numpy().astype(np.float64)
        got = got.cpu().numpy().astype(np.float64)
        for (bb, h), u in units.items():
            u.append(K[bb, h, T0 + step], V[bb, h, T0 + step])
            hs = slice(h * w.group_q, (h + 1) * w.group_q)
            o = u.attention(qn[bb, hs], w.softmax_scale)
            assert oracle.max_rel_err(got[bb, hs], o) <= TOL, (widx, step, bb, h, "fused")
            assert oracle.max_rel_err(ref[bb, hs], o) <= TOL, (widx, step, bb, h, "separate")
            assert oracle.max_rel_err(got[bb, hs], ref[bb, hs]) <= 1e-3, (widx, step, bb, h)
    for bb in range(batch):
        for h in range(kvh):
            ea, eb = a.export_unit(bb, h), b.export_unit(bb, h)
            for key in ea:
                assert np.array_equal(ea[key], eb[key]), (widx, bb, h, key)
    assert a.sync_status() == 0 and b.sync_status() == 0
    a.close()
    b.close()


def test_decode_step_capacity_and_launches():
    import bit_asymmetric_kv_kvq_gb300 as kvq
    w = synth.WORKLOADS[0].scaled(prefill_tokens=1023, decode_steps=1)
    K = synth.keys(w)
    V = synth.values(w)
    cache = kvq.KVCache.for_workload(w)  # max_tokens = 1024
    cache.prefill_quantize(_dev(K[:, :, :1023]), _dev(V[:, :, :1023]))
    n0 = cache.launch_count()
    q = _dev(synth.queries(w, 0))
    cache.decode_step(_dev(K[:, :, 1023]), _dev(V[:, :, 1023]), q)
    assert cache.launch_count() - n0 == 2  # no flush: the decode kernel and the merge of its partials
    with pytest.raises(kvq.KVQError) as e:
        cache.decode_step(_dev(K[:, :, 1023]), _dev(V[:, :, 1023]), q)
    assert e.value.status == kvq.kvq.KVQ_ERR_CAPACITY
    assert cache.state() == (1024, 896, 128)
    cache.close()
