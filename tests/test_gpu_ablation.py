"""GPU axis ablation against the oracle and numpy.

Quantization along either axis must give the oracle's codes, zero points and scales bit for bit
(keys per channel = oracle.quantize_keys, per token = oracle.quantize_values, and the same two for
values); dequantization must equal z + s*code rounded once to fp32; the fp32 attention kernel must
match numpy's fp64 softmax attention over the same rows within 1e-5.  The harness must reproduce
the ordering the unite.ai page states for keys ("Keys" section): on keys with outlier channels,
per-channel groups give a lower score error than per-token groups at every bit width.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

RNG = np.random.default_rng(2468)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _inputs(U, T, D=128):
    w = synth.WORKLOADS[1].scaled(batch=1, kv_heads=U, q_heads=U, prefill_tokens=T, decode_steps=1)
    K = synth.keys(w)[0, :, :T].copy()
    V = synth.values(w)[0, :, :T].copy()
    K[0, :64, :] = np.float16(1.5)          # constant groups: zero range, codes 0
    K[1, 3, 5] = np.float16(-0.0)
    V[-1, 7, :] = np.float16(-2.25)
    return K, V


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("axis", ["tokens", "channels"])
def test_axis_quantize_matches_oracle(bits, group, axis):
    from bit_asymmetric_kv_kvq_gb300 import ablation
    from bit_asymmetric_kv_kvq_gb300.kvq import KVQ_AXIS_CHANNELS, KVQ_AXIS_TOKENS
    ax = KVQ_AXIS_TOKENS if axis == "tokens" else KVQ_AXIS_CHANNELS
    K, V = _inputs(3, 256)
    for X in (K, V):
        codes, z, s = ablation.quantize(_dev(X), bits, group, ax)
        deq = ablation.dequantize(codes, z, s, group, ax)
        torch.cuda.synchronize()
        codes, deq = codes.cpu().numpy(), deq.cpu().numpy()
        z, s = z.cpu().numpy().view(np.uint16), s.cpu().numpy().view(np.uint16)
        for u in range(X.shape[0]):
            if axis == "tokens":
                rc, rz, rs, _, _ = oracle.quantize_keys(X[u], group, bits)
                zz = oracle.bits_f64(rz).repeat(group, axis=0)
                ss = oracle.bits_f64(rs).repeat(group, axis=0)
            else:
                rc, rz, rs = oracle.quantize_values(X[u], group, bits)
                zz = oracle.bits_f64(rz).repeat(group, axis=1)
                ss = oracle.bits_f64(rs).repeat(group, axis=1)
            assert np.array_equal(codes[u], rc), (u, "codes")
            assert np.array_equal(z[u], rz), (u, "zero")
            assert np.array_equal(s[u], rs), (u, "scale")
            want = (zz + ss * rc).astype(np.float32)  # exact in fp64, then one rounding
            assert np.array_equal(deq[u], want), (u, "dequant")


@pytest.mark.parametrize("hg", [1, 4])
@pytest.mark.parametrize("f32", [True, False])
def test_axis_attention_matches_numpy(hg, f32):
    from bit_asymmetric_kv_kvq_gb300 import ablation
    U, T, D = 3, 301, 128
    K = (RNG.standard_normal((U, T, D)) * 2).astype(np.float32 if f32 else np.float16)
    V = RNG.standard_normal((U, T, D)).astype(np.float32 if f32 else np.float16)
    Q = RNG.standard_normal((U, hg, D)).astype(np.float16)
    scale = float(np.float32(1 / np.sqrt(D)))
    out, sc = ablation.attention(_dev(K), _dev(V), _dev(Q), scale, with_scores=True)
    torch.cuda.synchronize()
    out, sc = out.cpu().numpy(), sc.cpu().numpy()
    for u in range(U):
        q = Q[u].astype(np.float64)
        s = scale * (q @ K[u].astype(np.float64).T)
        assert np.abs(sc[u] - s).max() <= 1e-5 * np.abs(s).max()
        p = np.exp(s - s.max(axis=1, keepdims=True))
        ref = (p / p.sum(axis=1, keepdims=True)) @ V[u].astype(np.float64)
        assert oracle.max_rel_err(out[u], ref) <= 1e-5


def test_harness_orders_key_axes_like_the_pages():
    from bit_asymmetric_kv_kvq_gb300 import ablation
    U, T = 8, 1024
    w = synth.WORKLOADS[1].scaled(batch=1, kv_heads=U, q_heads=U, prefill_tokens=T, decode_steps=1)
    K = _dev(synth.keys(w)[0, :, :T])
    V = _dev(synth.values(w)[0, :, :T])
    Q = _dev(synth.queries(w, 0)[0].reshape(U, 1, -1))
    for bits in (2, 3, 4):
        e = ablation.axis_errors(K, V, Q, bits, 32, w.softmax_scale)
        for va in ("channel", "token"):
            assert e[("channel", va)]["score_rel_fro"] < e[("token", va)]["score_rel_fro"], (bits, va, e)
        # the score error depends on the keys only
        assert e[("channel", "channel")]["score_rel_fro"] == e[("channel", "token")]["score_rel_fro"]
