"""Pins of the oracle's fp16 codec, quantizer, sparse selection and packing.

Each test checks the oracle against something other than itself: numpy's
independent binary16 conversion, the quantizer's closed-form error bound
(element error at most half a step, unite.ai page, "Quantization error in
practice"), exact grid round trips, brute force over every code, and packing
recomputed with Python integers.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(12345)


# ------------------------------------------------------------------ fp16 codec

def test_half_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_double_n(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # sign of zero is kept
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0])


def test_half_encode_roundtrips_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = bits.view(np.float16).astype(np.float32)
    back = oracle.float_to_half_n(f)
    finite = ~np.isnan(f)
    assert np.array_equal(back[finite], bits[finite])
    assert np.all((back[~finite] & 0x7C00) == 0x7C00) and np.all((back[~finite] & 0x3FF) != 0)


def _edge_floats():
    vals = []
    for h in range(0, 0x7C00, 7):  # midpoints between neighbouring halves: exact ties
        a = np.float64(np.uint16(h).view(np.float16))
        b = np.float64(np.uint16(h + 1).view(np.float16))
        mid = (a + b) / 2
        vals += [mid, np.nextafter(mid, 0), np.nextafter(mid, 1e9)]
    vals += [65504.0, 65519.99, 65520.0, 65536.0, 1e9, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001,
             2.0 ** -26, 1e-30, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 6.1e-5]
    vals = np.array(vals, np.float64)
    return np.concatenate([vals, -vals]).astype(np.float32)


def test_float_to_half_matches_numpy_rne():
    f = np.concatenate([
        _edge_floats(),
        (RNG.standard_normal(1_000_000) * 10.0 ** RNG.uniform(-9, 5, 1_000_000)).astype(np.float32),
        RNG.integers(0, 2 ** 32, 1_000_000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    f = f[~np.isnan(f)]
    ours = oracle.float_to_half_n(f)
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(f[i]), hex(ours[i]), hex(ref[i])) for i in bad[:5]]


# ------------------------------------------------------------------ quantizer

def _groups(n_groups, G, scale_range=(-3, 3)):
    """fp16 groups with assorted ranges, offsets and outliers."""
    out = []
    for i in range(n_groups):
        kind = i % 4
        mag = 10.0 ** RNG.uniform(*scale_range)
        x = RNG.standard_normal(G) * mag
        if kind == 1:
            x += RNG.uniform(-100, 100)
        elif kind == 2:
            x[RNG.integers(G)] *= 50
        elif kind == 3:
            x = np.abs(x)
        out.append(np.clip(x, -60000, 60000).astype(np.float16))
    return out


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("G", [32, 64])
def test_error_at_most_half_step(bits, G):
    """|x - x^| <= s/2 (+ the fp16 rounding of the step), for every element."""
    L = 2 ** bits - 1
    for x in _groups(300, G):
        zb, sb, codes = oracle.quantize_group(x, bits)
        xd = x.astype(np.float64)
        z, s = oracle.half_to_double(zb), oracle.half_to_double(sb)
        rng = xd.max() - xd.min()
        s_exact = rng / L
        xhat = z + s * codes.astype(np.float64)
        bound = s / 2 + L * abs(s_exact - s) + 4 * np.spacing(np.float32(np.abs(xd).max()))
        assert np.all(np.abs(xd - xhat) <= bound)
        assert codes.max() <= L
        # zero point is the group minimum, stored exactly
        assert z == xd.min() or (z == 0 and xd.min() == 0)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_codes_are_nearest_step_brute_force(bits):
    """The chosen code is the nearest grid point among all 2^B (ties to even)."""
    L = 2 ** bits - 1
    for x in _groups(200, 32):
        zb, sb, codes = oracle.quantize_group(x, bits)
        z, s = oracle.half_to_double(zb), oracle.half_to_double(sb)
        xd = x.astype(np.float64)
        grid = z + s * np.arange(L + 1)
        err = np.abs(xd[:, None] - grid[None, :])
        best = err.min(axis=1)
        chosen = err[np.arange(xd.size), codes]
        # fp32 rounding of (x - z)/s moves a decision by at most a few ulp of a step
        assert np.all(chosen <= best + 1e-6 * s)
        ties = np.isclose(err, best[:, None], rtol=0, atol=1e-9 * s).sum(axis=1) > 1
        for i in np.nonzero(ties)[0]:
            cands = np.nonzero(np.isclose(err[i], best[i], rtol=0, atol=1e-9 * s))[0]
            assert codes[i] in cands and codes[i] % 2 == 0


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_min_maps_to_zero_and_max_to_top_code(bits):
    L = 2 ** bits - 1
    for x in _groups(200, 32):
        xd = x.astype(np.float64)
        if xd.max() == xd.min():
            continue
        _, _, codes = oracle.quantize_group(x, bits)
        assert codes[np.argmin(xd)] == 0
        assert codes[np.argmax(xd)] == L


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_constant_group_is_exact(bits):
    for v in [0.0, -0.0, 1.5, -3.25, 1000.0, 6e-5]:
        x = np.full(32, v, np.float16)
        zb, sb, codes = oracle.quantize_group(x, bits)
        assert sb == 0 and np.all(codes == 0)
        assert oracle.half_to_double(zb) == np.float64(np.float16(v))
        assert zb != 0x8000  # -0 is stored as +0


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_grid_values_roundtrip_exactly(bits):
    """Values z + k*s (k = 0..L all present) come back with z, s and codes k."""
    L = 2 ** bits - 1
    for _ in range(200):
        e = int(RNG.integers(-8, 4))
        ms = int(RNG.integers(1, 8))
        mz = int(RNG.integers(-200, 200))
        s = ms * 2.0 ** e
        z = mz * 2.0 ** e
        k = RNG.integers(0, L + 1, 32)
        k[0], k[1] = 0, L
        RNG.shuffle(k)
        x = (z + s * k).astype(np.float16)
        assert np.array_equal(x.astype(np.float64), z + s * k)
        zb, sb, codes = oracle.quantize_group(x, bits)
        assert oracle.half_to_double(zb) == z and oracle.half_to_double(sb) == s
        assert np.array_equal(codes, k)


def test_excluded_entries_leave_the_range():
    x = RNG.standard_normal(32).astype(np.float16)
    x[5] = 300.0
    excl = np.zeros(32, np.uint8)
    excl[5] = 1
    zb0, sb0, _ = oracle.quantize_group(x, 2)
    zb1, sb1, codes = oracle.quantize_group(x, 2, excl)
    keep = np.delete(x.astype(np.float64), 5)
    assert oracle.half_to_double(sb1) <= oracle.half_to_double(sb0)
    assert oracle.half_to_double(zb1) == keep.min()
    assert codes[5] == 0
    # every entry excluded -> zero range, codes 0
    zb, sb, codes = oracle.quantize_group(x, 2, np.ones(32, np.uint8))
    assert zb == 0 and sb == 0 and not codes.any()


# ------------------------------------------------------------------ sparse outliers

def test_sparse_select_brute_force():
    for _ in range(500):
        D = 8
        x = RNG.choice(np.array([-3, -2, -1, -0.5, 0, 0.5, 1, 2, 3], np.float16), D)
        nsp = int(RNG.integers(1, 4))
        idx, val = oracle.sparse_select(x, nsp)
        a = np.abs(x.astype(np.float64))
        assert list(idx) == sorted(idx) and len(set(idx)) == nsp
        assert np.array_equal(val, x[idx].view(np.uint16))
        chosen = set(int(i) for i in idx)
        for c in range(D):
            if c in chosen:
                continue
            for i in chosen:
                assert a[i] > a[c] or (a[i] == a[c] and i < c)


def test_keys_sparse_entries_reconstruct_exactly_and_shrink_ranges():
    T, D, G = 64, 16, 32
    K = RNG.standard_normal((T, D)).astype(np.float16)
    K[:, 3] *= 40
    codes, z, s, si, sv = oracle.quantize_keys(K, G, 3, nsp=2)
    _, z0, s0, _, _ = oracle.quantize_keys(K, G, 3, nsp=0)
    assert np.all(oracle.bits_f64(s) <= oracle.bits_f64(s0))
    u = oracle.OracleUnit(D, 3, 3, G, 64, k_sparse=2)
    u.kcodes, u.kz, u.ks, u.sp_idx, u.sp_val = codes, z, s, si, sv
    u.vcodes = np.zeros((T, D), np.uint8)
    u.vz = np.zeros((T, D // G), np.uint16)
    u.vs = np.zeros((T, D // G), np.uint16)
    for t in range(T):
        k, _ = u.dequant(t)
        for j in range(2):
            c = si[t, j]
            assert k[c] == np.float64(K[t, c])
            assert codes[t, c] == 0
        # the largest-|x| entry of each token is always one of the two
        assert np.argmax(np.abs(K[t].astype(np.float64))) in si[t]


# ------------------------------------------------------------------ packing

# Worked examples of the packing reading (code i at bits [B*i, B*i+B) of a
# little-endian bitstream of 32-bit words), worked out by hand:
#   B=2, codes i mod 4:  each byte is 00,01,10,11 from bit 0 up = 0xE4.
#   B=4, codes i mod 16: nibbles 0..7 then 8..15.
#   B=3, codes i mod 8:  word 0 = sum_{i<10} (i mod 8) << 3i  +  (10 mod 8 & 3) << 30.
PACK_EXAMPLES = [
    (2, [i % 4 for i in range(32)], [0xE4E4E4E4, 0xE4E4E4E4]),
    (3, [i % 8 for i in range(32)], [0x88FAC688, 0xC688FAC6, 0xFAC688FA]),
    (3, [(7 - i) % 8 for i in range(32)], [0x77053977, 0x39770539, 0x05397705]),
    (4, [i % 16 for i in range(32)], [0x76543210, 0xFEDCBA98, 0x76543210, 0xFEDCBA98]),
]


@pytest.mark.parametrize("bits,codes,words", PACK_EXAMPLES)
def test_pack_worked_examples(bits, codes, words):
    got = oracle.pack(np.array(codes, np.uint8), bits)
    assert [int(w) for w in got] == words
    assert list(oracle.unpack(got, 32, bits)) == codes


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pack_matches_big_integer_bitstream(bits):
    for _ in range(50):
        n = 128
        codes = RNG.integers(0, 2 ** bits, n).astype(np.uint8)
        big = 0
        for i, c in enumerate(codes):
            big |= int(c) << (bits * i)
        ref = [(big >> (32 * w)) & 0xFFFFFFFF for w in range(n * bits // 32)]
        assert [int(w) for w in oracle.pack(codes, bits)] == ref
        assert np.array_equal(oracle.unpack(oracle.pack(codes, bits), n, bits), codes)
