"""Pins of the oracle's attention-sink tokens (the first S tokens kept fp16 beside the window).

unite.ai page and dothoosh.com page, research-direction sections (InnerQ keeps high-precision
windows for both the recent tokens and the attention-sink tokens).  The references here are
independent of the oracle's sink code: the plain cache (S = 0) on the sequence without its first
S tokens, numpy softmax attention, explicit rotation matrices at absolute positions, and the
state machine's counts written out.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(4242)


def textbook_attention(q, K, V, scale):
    s = scale * (q @ K.T)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    return p @ V


def rot_matrix(D, t, base):
    h = D // 2
    M = np.zeros((D, D))
    for i in range(h):
        a = t * base ** (-2.0 * i / D)
        c, s = np.cos(a), np.sin(a)
        M[i, i], M[i, i + h] = c, -s
        M[i + h, i], M[i + h, i + h] = s, c
    return M


def _seq(T, D, scale=3.0):
    K = (RNG.standard_normal((T, D)) * scale).astype(np.float16)
    V = RNG.standard_normal((T, D)).astype(np.float16)
    return K, V


@pytest.mark.parametrize("rope", [0, 1])
def test_sink_only_is_exact_attention(rope):
    """T <= S: every token stays fp16 in the sink; attention is the textbook one."""
    D, S = 16, 8
    K, V = _seq(S, D)
    u = oracle.OracleUnit(D, 2, 2, 8, 16, 0, rope, 100.0, sink=S)
    u.prefill(K[:5], V[:5])
    for t in range(5, S):
        u.append(K[t], V[t])
    assert (u.n_s, u.Tq, u.n_r) == (S, 0, 0)
    Kd = K.astype(np.float64)
    if rope:
        Kd = np.stack([rot_matrix(D, t, 100.0) @ Kd[t] for t in range(S)])
    q = RNG.standard_normal((3, D)).astype(np.float16)
    got = u.attention(q, 0.3)
    ref = textbook_attention(q.astype(np.float64), Kd, V.astype(np.float64), np.float64(np.float32(0.3)))
    assert np.abs(got - ref).max() < 1e-12


@pytest.mark.parametrize("S", [1, 3, 16])
def test_stores_after_the_sink_equal_the_plain_cache_of_the_shifted_sequence(S):
    """Quantization starts at token S: the packed stores and the window are those of a cache
    without sinks fed tokens S.., and the sink holds tokens 0..S exactly."""
    D, G, R = 32, 8, 16
    for T in [S + 1, S + R, S + R + 1, S + 3 * R + 5]:
        K, V = _seq(T, D)
        u = oracle.OracleUnit(D, 3, 2, G, R, 1, 0, 10000.0, sink=S)
        u.prefill(K, V)
        plain = oracle.OracleUnit(D, 3, 2, G, R, 1, 0, 10000.0)
        plain.prefill(K[S:], V[S:])
        got, ref = u.stores(), plain.stores()
        for key in ref:
            if key in ("sk", "sv"):
                continue
            assert np.array_equal(got[key], ref[key]), (S, T, key)
        assert np.array_equal(got["sk"], K[:S].view(np.uint16))
        assert np.array_equal(got["sv"], V[:S].view(np.uint16))
        assert (u.n_s, u.Tq, u.n_r) == (S, R * ((T - S - 1) // R), T - S - R * ((T - S - 1) // R))


@pytest.mark.parametrize("rope", [0, 1])
def test_brute_force_with_sink(rope):
    """Attention over sink + quantized + window == numpy attention over the tokens as the decoder
    sees them, each (when RoPE applies) rotated at its absolute position."""
    D, G, R, S, base = 8, 8, 16, 3, 100.0
    for T in [1, 2, 3, 4, 19, 20, 36, 70]:
        K, V = _seq(T, D)
        u = oracle.OracleUnit(D, 3, 3, G, R, 1, rope, base, sink=S)
        u.prefill(K, V)
        ns = min(T, S)
        assert u.n_s == ns
        Kd = np.zeros((T, D))
        Vd = np.zeros((T, D))
        for t in range(T):
            j = t - ns
            if t < ns:
                k, v = K[t].astype(np.float64), V[t].astype(np.float64)
            elif j < u.Tq:
                g = j // G
                k = oracle.bits_f64(u.kz[g]) + oracle.bits_f64(u.ks[g]) * u.kcodes[j]
                k[u.sp_idx[j, 0]] = oracle.bits_f64(u.sp_val[j, 0])
                v = oracle.bits_f64(u.vz[j]).repeat(G) + oracle.bits_f64(u.vs[j]).repeat(G) * u.vcodes[j]
            else:
                k, v = K[t].astype(np.float64), V[t].astype(np.float64)
            if rope:
                k = rot_matrix(D, t, base) @ k
            Kd[t], Vd[t] = k, v
        q = RNG.standard_normal((2, D)).astype(np.float16)
        got = u.attention(q, 0.35)
        ref = textbook_attention(q.astype(np.float64), Kd, Vd, np.float64(np.float32(0.35)))
        assert np.abs(got - ref).max() < 1e-12, T


def test_prefill_and_appends_reach_the_same_state_with_sink():
    """state(prefill(T)) == state(prefill(T0) + appends) for every T0, also T0 < S."""
    D, G, R, S = 16, 8, 16, 5
    T = S + 2 * R + 7
    K, V = _seq(T, D)
    ref = oracle.OracleUnit(D, 2, 4, G, R, 0, 0, 10000.0, sink=S)
    ref.prefill(K, V)
    want = ref.stores()
    for T0 in [1, 2, S - 1, S, S + 1, S + R, S + R + 1, T - 1]:
        u = oracle.OracleUnit(D, 2, 4, G, R, 0, 0, 10000.0, sink=S)
        u.prefill(K[:T0], V[:T0])
        for t in range(T0, T):
            u.append(K[t], V[t])
        got = u.stores()
        for key in want:
            assert np.array_equal(got[key], want[key]), (T0, key)
