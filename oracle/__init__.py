"""CPU oracle for the asymmetric low-bit KV cache: TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library's product path never loads
it and shares no code with it.

The arithmetic lives in ``kvq_oracle.c`` (plain scalar C, fp32 quantizer steps
with no FMA contraction, fp64 attention).  This file adds the cache state
machine and the canonical packed stores the CUDA library exports:

  kcodes  uint32 [Tq][D*Bk/32]   key codes, one row per token, channel bitstream
  kz, ks  uint16 [Tq/G][D]        key zero point / scale (fp16 bits), per channel per G-token group
  vcodes  uint32 [Tq][D*Bv/32]   value codes, one row per token
  vz, vs  uint16 [Tq][D/G]        value zero point / scale, per token per G-channel group
  sp_idx  uint8  [Tq][nsp]        sparse key entries: channel, ascending
  sp_val  uint16 [Tq][nsp]        sparse key entries: exact fp16 value
  wk, wv  uint16 [n_r][D]         fp16 residual window (tokens S+Tq .. S+Tq+n_r)
  sk, sv  uint16 [n_s][D]         fp16 attention-sink tokens (tokens 0 .. n_s)

State machine (unite.ai page, "System tax"; KIVI summary page, "Method"):
the most recent tokens stay in an fp16 window of at most R tokens and are
quantized as one block when the window is full.  Reading: an append that
finds the window full first quantizes those R tokens, then stores the new
token, so for T >= 1 tokens the window holds n_r in [1, R] tokens and
Tq = R*floor((T-1)/R).

Codebooks (KVQuant review, "Proposed method": the nuqX non-uniform datatype,
here with caller-supplied levels instead of calibrated ones): a cache may map
codes to non-uniform levels lev[c] (in steps, 0 = lev[0] < ... < lev[L] = L);
a value then takes the nearest level and dequantizes to z + s*lev[c].

Attention sinks (unite.ai page and dothoosh.com page, sections on research
directions, on InnerQ): besides the recent window, the first tokens of the
sequence are kept in fp16 too.  Reading: with S sink tokens, the first
n_s = min(T, S) tokens go to the sink store and are never quantized; the
state machine above runs on the tokens after them (T - n_s of them), so
Tq = R*floor((T-n_s-1)/R).  Positions (for RoPE) stay absolute: sink tokens
0..n_s, quantized tokens n_s..n_s+Tq, window after them.  S = 0 is the plain
cache.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libkvqoracle.so")

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2 -ffp-contract=off, no fast-math)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Unit(ctypes.Structure):
    _fields_ = [("D", _I), ("G", _I), ("nsp", _I), ("rope", _I), ("rope_base", ctypes.c_double),
                ("Tq", _I64), ("n_r", _I64),
                ("kcodes", _P), ("kz", _P), ("ks", _P), ("sp_idx", _P), ("sp_val", _P),
                ("vcodes", _P), ("vz", _P), ("vs", _P), ("wk", _P), ("wv", _P),
                ("n_s", _I64), ("sk", _P), ("sv", _P), ("k_lev", _P), ("v_lev", _P)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.kvqo_half_to_double.restype = ctypes.c_double
            L.kvqo_half_to_double.argtypes = [ctypes.c_uint16]
            L.kvqo_float_to_half.restype = ctypes.c_uint16
            L.kvqo_float_to_half.argtypes = [ctypes.c_float]
            L.kvqo_half_to_double_n.restype = None
            L.kvqo_half_to_double_n.argtypes = [_P, _I64, _P]
            L.kvqo_float_to_half_n.restype = None
            L.kvqo_float_to_half_n.argtypes = [_P, _I64, _P]
            L.kvqo_quantize_group.restype = None
            L.kvqo_quantize_group.argtypes = [_P, _I64, _I, _P, _I64, _I, _P, _P, _P, _I64, _P]
            L.kvqo_sparse_select.restype = None
            L.kvqo_sparse_select.argtypes = [_P, _I, _I, _P, _P]
            L.kvqo_quantize_keys.restype = _I
            L.kvqo_quantize_keys.argtypes = [_P, _I64, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]
            L.kvqo_quantize_values.restype = _I
            L.kvqo_quantize_values.argtypes = [_P, _I64, _I, _I, _I, _P, _P, _P, _P]
            L.kvqo_pack.restype = _I
            L.kvqo_pack.argtypes = [_P, _I64, _I, _P]
            L.kvqo_unpack.restype = _I
            L.kvqo_unpack.argtypes = [_P, _I64, _I, _P]
            L.kvqo_rope.restype = None
            L.kvqo_rope.argtypes = [_P, _I, ctypes.c_double, ctypes.c_double]
            L.kvqo_dequant_token.restype = _I
            L.kvqo_dequant_token.argtypes = [ctypes.POINTER(_Unit), _I64, _P, _P]
            L.kvqo_attention_partial.restype = _I
            L.kvqo_attention_partial.argtypes = [ctypes.POINTER(_Unit), _P, _I, ctypes.c_float, _I64, _I64, _P, _P, _P]
            L.kvqo_combine.restype = _I
            L.kvqo_combine.argtypes = [_I, _I, _P, _P, _P, _P]
            L.kvqo_attention.restype = _I
            L.kvqo_attention.argtypes = [ctypes.POINTER(_Unit), _P, _I, ctypes.c_float, _P]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- fp16 codec

def half_to_double(bits: int) -> float:
    return float(lib().kvqo_half_to_double(int(bits)))


def float_to_half(x) -> int:
    """fp32 -> fp16 bits, round to nearest even (x is first taken to fp32)."""
    return int(lib().kvqo_float_to_half(float(np.float32(x))))


def half_to_double_n(bits) -> np.ndarray:
    b = _c(bits, np.uint16).ravel()
    out = np.zeros(b.size, np.float64)
    lib().kvqo_half_to_double_n(_ptr(b), b.size, _ptr(out))
    return out


def float_to_half_n(x) -> np.ndarray:
    f = _c(x, np.float32).ravel()
    out = np.zeros(f.size, np.uint16)
    lib().kvqo_float_to_half_n(_ptr(f), f.size, _ptr(out))
    return out


def f16_bits(a) -> np.ndarray:
    """fp16 bit patterns of `a`: uint16 arrays are taken as bits already, float16 arrays are viewed,
    anything else is rounded to fp16 first."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a)
    return np.ascontiguousarray(np.asarray(a, np.float16)).view(np.uint16)


def bits_f64(b) -> np.ndarray:
    return np.asarray(b, np.uint16).view(np.float16).astype(np.float64)


# ---------------------------------------------------------------- quantizer

def quantize_group(x16, bits: int, excl=None, levels=None):
    """One group of fp16 values -> (z_bits, s_bits, codes u8); levels: non-uniform levels in steps."""
    lev = _levels(levels, bits)
    x = f16_bits(x16).ravel().copy()
    n = x.size
    ex = None if excl is None else _c(excl, np.uint8).ravel()
    z = np.zeros(1, np.uint16)
    s = np.zeros(1, np.uint16)
    codes = np.zeros(n, np.uint8)
    lib().kvqo_quantize_group(_ptr(x), 1, n, _ptr(ex), 1, bits, _ptr(z), _ptr(s), _ptr(codes), 1, _ptr(lev))
    return int(z[0]), int(s[0]), codes


def sparse_select(x16, nsp: int):
    x = f16_bits(x16).ravel().copy()
    idx = np.zeros(nsp, np.uint8)
    val = np.zeros(nsp, np.uint16)
    lib().kvqo_sparse_select(_ptr(x), x.size, nsp, _ptr(idx), _ptr(val))
    return idx, val


def _levels(levels, bits):
    if levels is None:
        return None
    lev = np.ascontiguousarray(levels, dtype=np.float32)
    if lev.shape != (1 << bits,):
        raise ValueError("need 2^bits levels")
    return lev


def quantize_keys(K16, G: int, bits: int, nsp: int = 0, levels=None):
    """Keys [T][D] fp16 -> codes u8 [T][D], z/s u16 [T/G][D], sp_idx u8 [T][nsp], sp_val u16 [T][nsp]."""
    K = f16_bits(K16)
    T, D = K.shape
    codes = np.zeros((T, D), np.uint8)
    z = np.zeros((T // G, D), np.uint16)
    s = np.zeros((T // G, D), np.uint16)
    si = np.zeros((T, nsp), np.uint8)
    sv = np.zeros((T, nsp), np.uint16)
    lev = _levels(levels, bits)
    rc = lib().kvqo_quantize_keys(_ptr(K), T, D, G, bits, nsp, _ptr(codes), _ptr(z), _ptr(s), _ptr(si), _ptr(sv),
                                  _ptr(lev))
    if rc != 0:
        raise ValueError(f"kvqo_quantize_keys rejected its arguments ({rc})")
    return codes, z, s, si, sv


def quantize_values(V16, G: int, bits: int, levels=None):
    """Values [T][D] fp16 -> codes u8 [T][D], z/s u16 [T][D/G]."""
    V = f16_bits(V16)
    T, D = V.shape
    codes = np.zeros((T, D), np.uint8)
    z = np.zeros((T, D // G), np.uint16)
    s = np.zeros((T, D // G), np.uint16)
    lev = _levels(levels, bits)
    rc = lib().kvqo_quantize_values(_ptr(V), T, D, G, bits, _ptr(codes), _ptr(z), _ptr(s), _ptr(lev))
    if rc != 0:
        raise ValueError(f"kvqo_quantize_values rejected its arguments ({rc})")
    return codes, z, s


def pack_rows(codes, bits: int) -> np.ndarray:
    """Pack each row (token) as its own bitstream.  Rows are a whole number of 32-bit words, so the
    rows laid end to end form one bitstream with the same words."""
    c = _c(codes, np.uint8)
    T, D = c.shape
    if (D * bits) % 32:
        raise ValueError("row length times bits is not a multiple of 32")
    out = np.zeros((T, D * bits // 32), np.uint32)
    if T and lib().kvqo_pack(_ptr(c), T * D, bits, _ptr(out)) != 0:
        raise ValueError("packing failed")
    return out


def pack(codes, bits: int) -> np.ndarray:
    c = _c(codes, np.uint8).ravel()
    out = np.zeros(c.size * bits // 32, np.uint32)
    if lib().kvqo_pack(_ptr(c), c.size, bits, _ptr(out)) != 0:
        raise ValueError("code count times bits is not a multiple of 32")
    return out


def unpack(words, n: int, bits: int) -> np.ndarray:
    w = _c(words, np.uint32).ravel()
    out = np.zeros(n, np.uint8)
    if lib().kvqo_unpack(_ptr(w), n, bits, _ptr(out)) != 0:
        raise ValueError("code count times bits is not a multiple of 32")
    return out


def rope(v, t: float, base: float) -> np.ndarray:
    x = np.array(v, np.float64)
    lib().kvqo_rope(_ptr(x), x.size, float(t), float(base))
    return x


def combine(m, l, acc) -> np.ndarray:
    m = _c(m, np.float64)
    l = _c(l, np.float64)
    acc = _c(acc, np.float64)
    S, D = acc.shape
    out = np.zeros(D, np.float64)
    if lib().kvqo_combine(S, D, _ptr(m), _ptr(l), _ptr(acc), _ptr(out)) != 0:
        raise ValueError("no partial holds a token")
    return out


def quantized_tokens(T: int, R: int) -> int:
    """Tq = R*floor((T-1)/R) for T >= 1 (window holds 1..R tokens), 0 for T = 0."""
    return 0 if T <= 0 else R * ((T - 1) // R)


# ---------------------------------------------------------------- one unit

class OracleUnit:
    """Cache state of one (batch, kv-head) sequence, driven like the library."""

    def __init__(self, head_dim, k_bits, v_bits, group, residual, k_sparse=0, rope=0, rope_base=10000.0, sink=0,
                 k_levels=None, v_levels=None):
        self.D, self.bk, self.bv, self.G, self.R = head_dim, k_bits, v_bits, group, residual
        self.nsp, self.rope, self.rope_base, self.S = k_sparse, rope, rope_base, sink
        self.k_lev, self.v_lev = _levels(k_levels, k_bits), _levels(v_levels, v_bits)
        D = head_dim
        self.kcodes = np.zeros((0, D), np.uint8)
        self.kz = np.zeros((0, D), np.uint16)
        self.ks = np.zeros((0, D), np.uint16)
        self.sp_idx = np.zeros((0, k_sparse), np.uint8)
        self.sp_val = np.zeros((0, k_sparse), np.uint16)
        self.vcodes = np.zeros((0, D), np.uint8)
        self.vz = np.zeros((0, D // group), np.uint16)
        self.vs = np.zeros((0, D // group), np.uint16)
        self.wk = np.zeros((0, D), np.uint16)
        self.wv = np.zeros((0, D), np.uint16)
        self.sk = np.zeros((0, D), np.uint16)
        self.sv = np.zeros((0, D), np.uint16)
        self.prefilled = False

    @classmethod
    def for_workload(cls, w):
        return cls(w.head_dim, w.k_bits, w.v_bits, w.group, w.residual, w.k_sparse, w.rope, w.rope_base,
                   getattr(w, "sink", 0), getattr(w, "k_levels", None) or None, getattr(w, "v_levels", None) or None)

    @property
    def Tq(self):
        return self.kcodes.shape[0]

    @property
    def n_r(self):
        return self.wk.shape[0]

    @property
    def n_s(self):
        return self.sk.shape[0]

    @property
    def T(self):
        return self.n_s + self.Tq + self.n_r

    def _quantize_block(self, K16, V16):
        kc, kz, ks, si, sv = quantize_keys(K16, self.G, self.bk, self.nsp, self.k_lev)
        vc, vz, vs = quantize_values(V16, self.G, self.bv, self.v_lev)
        self.kcodes = np.concatenate([self.kcodes, kc])
        self.kz = np.concatenate([self.kz, kz])
        self.ks = np.concatenate([self.ks, ks])
        self.sp_idx = np.concatenate([self.sp_idx, si])
        self.sp_val = np.concatenate([self.sp_val, sv])
        self.vcodes = np.concatenate([self.vcodes, vc])
        self.vz = np.concatenate([self.vz, vz])
        self.vs = np.concatenate([self.vs, vs])

    def prefill(self, K16, V16):
        """Cache T prompt tokens: the first min(T, S) go to the sink; of the rest, quantize the first
        R*floor((T'-1)/R) and keep the others in the fp16 window."""
        if self.prefilled or self.T:
            raise RuntimeError("prefill is allowed once, on an empty cache")
        K, V = f16_bits(K16), f16_bits(V16)
        ns = min(K.shape[0], self.S)
        self.sk, self.sv = K[:ns].copy(), V[:ns].copy()
        K, V = K[ns:], V[ns:]
        T = K.shape[0]
        Tq = quantized_tokens(T, self.R)
        if Tq:
            self._quantize_block(K[:Tq], V[:Tq])
        self.wk = K[Tq:].copy()
        self.wv = V[Tq:].copy()
        self.prefilled = True

    def append(self, k16, v16):
        """One decode token: into the sink while it has room; otherwise flush a full window as one
        quantized block, then store the token in the window."""
        k = f16_bits(k16).reshape(1, self.D)
        v = f16_bits(v16).reshape(1, self.D)
        if self.n_s < self.S:
            self.sk = np.concatenate([self.sk, k])
            self.sv = np.concatenate([self.sv, v])
            return
        if self.n_r == self.R:
            self._quantize_block(self.wk, self.wv)
            self.wk = np.zeros((0, self.D), np.uint16)
            self.wv = np.zeros((0, self.D), np.uint16)
        self.wk = np.concatenate([self.wk, k])
        self.wv = np.concatenate([self.wv, v])

    def stores(self) -> dict:
        """Canonical packed stores (the layout the library exports)."""
        return dict(kcodes=pack_rows(self.kcodes, self.bk), kz=self.kz.copy(), ks=self.ks.copy(),
                    vcodes=pack_rows(self.vcodes, self.bv), vz=self.vz.copy(), vs=self.vs.copy(),
                    sp_idx=self.sp_idx.copy(), sp_val=self.sp_val.copy(), wk=self.wk.copy(), wv=self.wv.copy(),
                    sk=self.sk.copy(), sv=self.sv.copy())

    def _struct(self):
        keep = [_c(self.kcodes, np.uint8), _c(self.kz, np.uint16), _c(self.ks, np.uint16),
                _c(self.sp_idx, np.uint8), _c(self.sp_val, np.uint16), _c(self.vcodes, np.uint8),
                _c(self.vz, np.uint16), _c(self.vs, np.uint16), _c(self.wk, np.uint16), _c(self.wv, np.uint16)]
        sink = [_c(self.sk, np.uint16), _c(self.sv, np.uint16)]
        u = _Unit(self.D, self.G, self.nsp, self.rope, float(self.rope_base), self.Tq, self.n_r,
                  *[_ptr(a) for a in keep], self.n_s, *[_ptr(a) for a in sink], _ptr(self.k_lev), _ptr(self.v_lev))
        keep += sink
        return u, keep

    def dequant(self, t: int):
        """(k, v) of token t in fp64 as the decoder sees them (k rotated when keys are pre-RoPE)."""
        u, keep = self._struct()
        k = np.zeros(self.D)
        v = np.zeros(self.D)
        if lib().kvqo_dequant_token(ctypes.byref(u), t, _ptr(k), _ptr(v)) != 0:
            raise IndexError(t)
        return k, v

    def attention_partial(self, q16, softmax_scale, t_begin, t_end):
        q = f16_bits(q16).reshape(-1, self.D).copy()
        Hg = q.shape[0]
        m = np.zeros(Hg)
        l = np.zeros(Hg)
        acc = np.zeros((Hg, self.D))
        u, keep = self._struct()
        rc = lib().kvqo_attention_partial(ctypes.byref(u), _ptr(q), Hg, float(softmax_scale), t_begin, t_end,
                                          _ptr(m), _ptr(l), _ptr(acc))
        if rc != 0:
            raise ValueError(f"kvqo_attention_partial failed ({rc})")
        return m, l, acc

    def attention(self, q16, softmax_scale) -> np.ndarray:
        """Decode attention of the Hg query heads q[h][c] (fp16, post-RoPE) over all T tokens, fp64."""
        q = f16_bits(q16).reshape(-1, self.D).copy()
        Hg = q.shape[0]
        out = np.zeros((Hg, self.D))
        u, keep = self._struct()
        rc = lib().kvqo_attention(ctypes.byref(u), _ptr(q), Hg, float(softmax_scale), _ptr(out))
        if rc != 0:
            raise ValueError(f"kvqo_attention failed ({rc})")
        return out


def unit_from_sequence(w, K16, V16) -> OracleUnit:
    """The state after caching the T tokens of K/V, written down directly (no appends)."""
    u = OracleUnit.for_workload(w)
    u.prefill(K16, V16)
    return u


def max_rel_err(out_test, out_ref) -> float:
    """Error metric: max over heads of ||o - o*||_inf / ||o*||_inf (rows are heads)."""
    a = np.asarray(out_test, np.float64).reshape(-1, out_ref.shape[-1])
    b = np.asarray(out_ref, np.float64).reshape(-1, out_ref.shape[-1])
    num = np.abs(a - b).max(axis=1)
    den = np.abs(b).max(axis=1)
    return float((num / den).max())
