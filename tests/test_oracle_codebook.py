"""Pins of the oracle's codebook (non-uniform level) quantizer.

KVQuant review, "Proposed method" (the nuqX datatype, here with caller-supplied levels).  The
references are independent of the oracle's level search: the uniform quantizer (levels c = c must
give the same codes away from exact ties), a brute-force nearest-level search in fp64 on the same
fp32 quotient, monotonicity, and numpy softmax attention over values rebuilt from the stores.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(97531)


def _quotients(x16, z_bits, s_bits):
    """The fp32 quotient (x - z) / s the quantizer rounds, as numpy computes it (IEEE fp32)."""
    z = np.float32(oracle.half_to_double(z_bits))
    s = np.float32(oracle.half_to_double(s_bits))
    return (x16.astype(np.float32) - z) / s


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_identity_levels_give_the_uniform_codes_away_from_ties(bits):
    lev = np.arange(1 << bits, dtype=np.float32)
    for _ in range(200):
        x = (RNG.standard_normal(32) * RNG.uniform(0.1, 30)).astype(np.float16)
        zu, su, cu = oracle.quantize_group(x, bits)
        zl, sl, cl = oracle.quantize_group(x, bits, levels=lev)
        assert (zu, su) == (zl, sl)
        y = _quotients(x, zu, su)
        tie = np.abs(y - np.floor(y) - 0.5) == 0
        assert np.array_equal(cu[~tie], cl[~tie])
        # on an exact tie the level search takes the lower level, rint the even one
        assert np.all(cl[tie] == np.floor(y[tie]))


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_nearest_level_by_brute_force(bits):
    L = (1 << bits) - 1
    for _ in range(200):
        inner = np.sort(RNG.uniform(0, L, L - 1))
        lev = np.concatenate([[0.0], inner, [float(L)]]).astype(np.float32)
        if np.any(np.diff(lev) <= 0):
            continue
        x = (RNG.standard_normal(64) * 5).astype(np.float16)
        z, s, codes = oracle.quantize_group(x, bits, levels=lev)
        y = _quotients(x, z, s).astype(np.float64)
        dist = np.abs(y[:, None] - lev[None, :].astype(np.float64))
        near = dist.argmin(axis=1)
        thr = ((lev[:-1] + lev[1:]).astype(np.float32) * np.float32(0.5)).astype(np.float64)
        clear = np.min(np.abs(y[:, None] - thr[None, :]), axis=1) > 1e-6
        assert np.array_equal(codes[clear], near[clear])
        # the group's minimum and maximum stay exact
        assert codes[np.argmin(x.astype(np.float32))] == 0 and codes[np.argmax(x.astype(np.float32))] == L


def test_codes_are_monotone_in_the_value():
    lev = np.array([0, 0.4, 1.1, 1.5, 2.9, 3.2, 5.0, 7.0], np.float32)
    x = np.sort((RNG.standard_normal(64) * 3).astype(np.float16))
    _, _, codes = oracle.quantize_group(x, 3, levels=lev)
    assert np.all(np.diff(codes.astype(int)) >= 0)


def test_codebook_unit_attention_is_textbook_attention_over_its_levels():
    D, G, R = 16, 8, 16
    klev = np.array([0, 0.7, 1.9, 3.0], np.float32)
    vlev = np.array([0, 0.25, 0.5, 1.0, 2.0, 3.5, 5.0, 6.0, 7.0, 8.0, 9.5, 11.0, 12.0, 13.0, 14.5, 15.0], np.float32)
    T = 3 * R + 5
    K = (RNG.standard_normal((T, D)) * 2).astype(np.float16)
    V = RNG.standard_normal((T, D)).astype(np.float16)
    u = oracle.OracleUnit(D, 2, 4, G, R, 0, 0, 10000.0, k_levels=klev, v_levels=vlev)
    u.prefill(K, V)
    Kd = K.astype(np.float64).copy()
    Vd = V.astype(np.float64).copy()
    for t in range(u.Tq):
        g = t // G
        Kd[t] = oracle.bits_f64(u.kz[g]) + oracle.bits_f64(u.ks[g]) * klev[u.kcodes[t]].astype(np.float64)
        Vd[t] = (oracle.bits_f64(u.vz[t]).repeat(G) + oracle.bits_f64(u.vs[t]).repeat(G)
                 * vlev[u.vcodes[t]].astype(np.float64))
    q = RNG.standard_normal((2, D)).astype(np.float16)
    sc = np.float64(np.float32(0.3)) * (q.astype(np.float64) @ Kd.T)
    p = np.exp(sc - sc.max(axis=1, keepdims=True))
    ref = (p / p.sum(axis=1, keepdims=True)) @ Vd
    assert np.abs(u.attention(q, 0.3) - ref).max() < 1e-12
    # the stores' codes are those of the group quantizer with the same levels
    c2, _, _, _, _ = oracle.quantize_keys(K[:u.Tq], G, 2, 0, klev)
    assert np.array_equal(u.kcodes, c2)


def test_exact_ties_take_the_lower_level():
    # z = 0, s = 1: quotients 0.5, 1.5 and 2.5 lie exactly on the thresholds of the identity levels
    x = np.array([0, 0.5, 1.5, 2.5, 3], np.float16)
    z, s, codes = oracle.quantize_group(x, 2, levels=np.arange(4, dtype=np.float32))
    assert oracle.half_to_double(s) == 1.0 and oracle.half_to_double(z) == 0.0
    assert codes.tolist() == [0, 0, 1, 2, 3]
    _, _, uni = oracle.quantize_group(x, 2)
    assert uni.tolist() == [0, 0, 2, 2, 3]  # rint: half to even
