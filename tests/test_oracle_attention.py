"""Pins of the oracle's decode attention, RoPE, split merge and cache state machine.

References used here are independent of the oracle: numpy's fp64 softmax
attention written as matrix products, explicit 2x2 rotation matrices, closed
forms (T = 1, q = 0, one-hot scores) and the directional claim of the
unite.ai page ("Keys" section): on keys with fixed outlier channels, grouping
per channel gives a lower attention-score error than grouping per token.
"""
import numpy as np
import pytest

import oracle
import synth

RNG = np.random.default_rng(777)


def textbook_attention(q, K, V, scale):
    """softmax(scale * q K^T) V in fp64, numpy."""
    s = scale * (q @ K.T)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    return p @ V


def rot_matrix(D, t, base):
    """Block rotation of the rotate-half layout: pairs (i, i + D/2)."""
    h = D // 2
    M = np.zeros((D, D))
    for i in range(h):
        a = t * base ** (-2.0 * i / D)
        c, s = np.cos(a), np.sin(a)
        M[i, i], M[i, i + h] = c, -s
        M[i + h, i], M[i + h, i + h] = s, c
    return M


def _unit(D=16, bk=2, bv=2, G=32, R=64, nsp=0, rope=0):
    return oracle.OracleUnit(D, bk, bv, G, R, nsp, rope, 10000.0)


def test_window_only_equals_textbook():
    """T <= R keeps everything fp16: plain softmax attention."""
    D, T = 16, 50
    u = _unit(D=D)
    K = RNG.standard_normal((T, D)).astype(np.float16)
    V = RNG.standard_normal((T, D)).astype(np.float16)
    u.prefill(K, V)
    assert u.Tq == 0 and u.n_r == T
    q = RNG.standard_normal((3, D)).astype(np.float16)
    got = u.attention(q, 0.25)
    ref = textbook_attention(q.astype(np.float64), K.astype(np.float64), V.astype(np.float64),
                             np.float64(np.float32(0.25)))
    assert np.abs(got - ref).max() < 1e-12


def test_single_token_returns_its_value():
    D = 16
    u = _unit(D=D)
    K = RNG.standard_normal((1, D)).astype(np.float16)
    V = RNG.standard_normal((1, D)).astype(np.float16)
    u.prefill(K, V)
    got = u.attention(RNG.standard_normal((2, D)).astype(np.float16), 0.3)
    assert np.array_equal(got, np.tile(V.astype(np.float64), (2, 1)))


def test_zero_query_averages_dequantized_values():
    D, G, R = 16, 16, 32
    u = oracle.OracleUnit(D, 2, 2, G, R)
    T = 3 * R + 5
    K = RNG.standard_normal((T, D)).astype(np.float16)
    V = RNG.standard_normal((T, D)).astype(np.float16)
    u.prefill(K, V)
    assert u.Tq == 3 * R
    vhat = np.stack([u.dequant(t)[1] for t in range(T)])
    got = u.attention(np.zeros((1, D), np.float16), 1.0)
    assert np.abs(got[0] - vhat.mean(axis=0)).max() < 1e-13
    # the quantized values are the stored grid: z + s*code, per token per channel group
    t = 7
    z = oracle.bits_f64(u.vz[t]).repeat(G)
    s = oracle.bits_f64(u.vs[t]).repeat(G)
    assert np.array_equal(vhat[t], z + s * u.vcodes[t])


def test_one_hot_scores_pick_one_token():
    D, T = 16, 40
    u = _unit(D=D)
    K = np.zeros((T, D), np.float16)
    K[17, 0] = 8.0
    V = RNG.standard_normal((T, D)).astype(np.float16)
    u.prefill(K, V)
    q = np.zeros((1, D), np.float16)
    q[0, 0] = 8.0  # score gap 64
    got = u.attention(q, 1.0)
    assert np.abs(got[0] - V[17].astype(np.float64)).max() < 1e-20 + 1e-25 * T


@pytest.mark.parametrize("bk,bv,G,nsp,rope", [(2, 2, 8, 0, 0), (4, 2, 8, 0, 0), (3, 3, 8, 1, 1)])
def test_brute_force_tiny_shapes(bk, bv, G, nsp, rope):
    """Oracle attention == numpy attention over the dequantized (and rotated) keys."""
    D, R = 8, 16
    for T in [1, 15, 16, 17, 33, 70]:
        u = oracle.OracleUnit(D, bk, bv, G, R, nsp, rope, 100.0)
        K = (RNG.standard_normal((T, D)) * 3).astype(np.float16)
        V = RNG.standard_normal((T, D)).astype(np.float16)
        u.prefill(K, V)
        Kd = np.zeros((T, D))
        Vd = np.zeros((T, D))
        for t in range(T):
            if t < u.Tq:
                g = t // G
                k = oracle.bits_f64(u.kz[g]) + oracle.bits_f64(u.ks[g]) * u.kcodes[t]
                for j in range(nsp):
                    k[u.sp_idx[t, j]] = oracle.bits_f64(u.sp_val[t, j])
                zv = oracle.bits_f64(u.vz[t]).repeat(G)
                sv = oracle.bits_f64(u.vs[t]).repeat(G)
                v = zv + sv * u.vcodes[t]
            else:
                k = K[t].astype(np.float64)
                v = V[t].astype(np.float64)
            if rope:
                k = rot_matrix(D, t, 100.0) @ k
            Kd[t], Vd[t] = k, v
        q = RNG.standard_normal((2, D)).astype(np.float16)
        scale = np.float32(0.35)
        got = u.attention(q, float(scale))
        ref = textbook_attention(q.astype(np.float64), Kd, Vd, np.float64(scale))
        assert np.abs(got - ref).max() < 1e-12, T


def test_rope_properties():
    D, base = 16, 10000.0
    k = RNG.standard_normal(D)
    q = RNG.standard_normal(D)
    assert np.array_equal(oracle.rope(k, 0, base), k)
    for t in [1, 5, 1000, 1048576]:
        assert abs(np.linalg.norm(oracle.rope(k, t, base)) - np.linalg.norm(k)) < 1e-12
        assert np.abs(oracle.rope(k, t, base) - rot_matrix(D, t, base) @ k).max() < 1e-9
    for m, n in [(3, 10), (100, 107), (1000000, 1000007)]:
        a = oracle.rope(q, m, base) @ oracle.rope(k, n, base)
        b = oracle.rope(q, 0, base) @ oracle.rope(k, n - m, base)
        assert abs(a - b) < 1e-8
    # sign convention: (1, 0) in the first pair turns toward +sin in channel D/2
    e = np.zeros(D)
    e[0] = 1
    r = oracle.rope(e, 0.5, base)
    assert abs(r[0] - np.cos(0.5)) < 1e-15 and abs(r[D // 2] - np.sin(0.5)) < 1e-15


def test_split_merge_is_associative():
    D, G, R = 16, 16, 32
    u = oracle.OracleUnit(D, 2, 2, G, R)
    T = 200
    K = (RNG.standard_normal((T, D)) * 2).astype(np.float16)
    V = RNG.standard_normal((T, D)).astype(np.float16)
    u.prefill(K, V)
    q = RNG.standard_normal((1, D)).astype(np.float16)
    full = u.attention(q, 0.5)[0]
    for _ in range(20):
        cuts = np.sort(RNG.choice(np.arange(1, T), size=int(RNG.integers(1, 8)), replace=False))
        edges = [0, *cuts.tolist(), T]
        ms, ls, accs = [], [], []
        for a, b in zip(edges[:-1], edges[1:]):
            m, l, acc = u.attention_partial(q, 0.5, a, b)
            ms.append(m[0]); ls.append(l[0]); accs.append(acc[0])
        # an empty split is allowed and ignored
        m, l, acc = u.attention_partial(q, 0.5, 5, 5)
        ms.append(m[0]); ls.append(l[0]); accs.append(acc[0])
        got = oracle.combine(ms, ls, np.array(accs))
        assert np.abs(got - full).max() < 1e-12


# ------------------------------------------------------------------ state machine

@pytest.mark.parametrize("T,R,Tq", [(0, 128, 0), (1, 128, 0), (128, 128, 0), (129, 128, 128), (1024, 128, 896),
                                    (1025, 128, 1024), (4096, 128, 3968), (1048577, 128, 1048576)])
def test_quantized_token_count(T, R, Tq):
    assert oracle.quantized_tokens(T, R) == Tq


@pytest.mark.parametrize("T0", [1, 31, 32, 64, 65, 100])
def test_flush_equivalence(T0):
    """prefill(T0) + appends up to T gives the same stores as prefill(T), bit for bit."""
    w = synth.WORKLOADS[4].scaled(batch=1, kv_heads=1, q_heads=2, head_dim=32, prefill_tokens=T0,
                                  decode_steps=150 - T0, group=16, residual=32, k_sparse=1)
    K = synth.keys(w)[0, 0]
    V = synth.values(w)[0, 0]
    inc = oracle.OracleUnit.for_workload(w)
    inc.prefill(K[:T0], V[:T0])
    for T in range(T0 + 1, 151):
        inc.append(K[T - 1], V[T - 1])
        assert 1 <= inc.n_r <= w.residual
        if T in (T0 + 1, 97, 128, 129, 150):
            direct = oracle.unit_from_sequence(w, K[:T], V[:T])
            a, b = inc.stores(), direct.stores()
            for key in a:
                assert np.array_equal(a[key], b[key]), (T, key)


@pytest.mark.parametrize("bits,G,nsp", [(2, 32, 0), (4, 32, 0), (3, 64, 2)])
def test_unit_stores_reconstruct_the_input(bits, G, nsp):
    """The cache state's stores, dequantized by hand, stay within half a step of the original tokens."""
    D, R, T = 64, 64, 200
    w = synth.WORKLOADS[4].scaled(batch=1, kv_heads=1, q_heads=1, head_dim=D, prefill_tokens=T - 5, decode_steps=5,
                                  group=G, residual=R, k_sparse=nsp, k_bits=bits, v_bits=bits)
    K = synth.keys(w)[0, 0]
    V = synth.values(w)[0, 0]
    u = oracle.OracleUnit.for_workload(w)
    u.prefill(K[:T - 5], V[:T - 5])
    for t in range(T - 5, T):
        u.append(K[t], V[t])
    st = u.stores()
    Tq = u.Tq
    assert Tq == oracle.quantized_tokens(T, R) == 192 and u.n_r == T - Tq
    L = 2 ** bits - 1
    kc = np.stack([oracle.unpack(st["kcodes"][t], D, bits) for t in range(Tq)]).astype(np.float64)
    vc = np.stack([oracle.unpack(st["vcodes"][t], D, bits) for t in range(Tq)]).astype(np.float64)
    kz = oracle.bits_f64(st["kz"]).repeat(G, axis=0)
    ks = oracle.bits_f64(st["ks"]).repeat(G, axis=0)
    khat = kz + ks * kc
    for t in range(Tq):
        for j in range(nsp):
            khat[t, st["sp_idx"][t, j]] = oracle.bits_f64(st["sp_val"][t, j])
    vz = oracle.bits_f64(st["vz"]).repeat(G, axis=1)
    vs = oracle.bits_f64(st["vs"]).repeat(G, axis=1)
    vhat = vz + vs * vc
    Kd, Vd = K[:Tq].astype(np.float64), V[:Tq].astype(np.float64)
    # half a step plus the fp16 rounding of the step (per group)
    assert np.all(np.abs(khat - Kd) <= ks * (0.5 + L * 2.0 ** -11) + 1e-6)
    assert np.all(np.abs(vhat - Vd) <= vs * (0.5 + L * 2.0 ** -11) + 1e-6)
    # sparse entries are exact, the window is the input verbatim
    for t in range(Tq):
        for j in range(nsp):
            assert khat[t, st["sp_idx"][t, j]] == Kd[t, st["sp_idx"][t, j]]
    assert np.array_equal(st["wk"], K[Tq:T].view(np.uint16)) and np.array_equal(st["wv"], V[Tq:T].view(np.uint16))


def test_prefill_twice_is_rejected():
    u = _unit()
    u.prefill(np.zeros((3, 16), np.float16), np.zeros((3, 16), np.float16))
    with pytest.raises(RuntimeError):
        u.prefill(np.zeros((3, 16), np.float16), np.zeros((3, 16), np.float16))


# ------------------------------------------------------------------ directional claims

def _score_error(Kq_fn, K, q, scale):
    Kd = K.astype(np.float64)
    return np.abs(scale * (Kq_fn - Kd) @ q).mean()


def test_per_channel_keys_beat_per_token_keys_on_outlier_channels():
    """Gate (unite.ai page, "Keys"): per-channel K gives lower score error than per-token K."""
    w = synth.WORKLOADS[0]
    K = synth.keys(w, nt=1024)[0]
    q = synth.queries(w, 0)[0].astype(np.float64)
    G, B, D = w.group, w.k_bits, w.head_dim
    for h in range(w.kv_heads):
        Kh = K[h]
        codes, z, s, _, _ = oracle.quantize_keys(Kh, G, B)
        per_channel = oracle.bits_f64(z).repeat(G, axis=0) + oracle.bits_f64(s).repeat(G, axis=0) * codes
        tc, tz, ts = oracle.quantize_values(Kh, G, B)  # same quantizer along the other axis
        per_token = oracle.bits_f64(tz).repeat(G, axis=1) + oracle.bits_f64(ts).repeat(G, axis=1) * tc
        e_ch = _score_error(per_channel, Kh, q[h], w.softmax_scale)
        e_tok = _score_error(per_token, Kh, q[h], w.softmax_scale)
        assert e_ch < e_tok, (h, e_ch, e_tok)
        # reconstruction error tells the same story for keys
        Kd = Kh.astype(np.float64)
        assert np.abs(per_channel - Kd).mean() < np.abs(per_token - Kd).mean()
