"""Seeded synthetic workloads for the asymmetric low-bit KV cache.

This module only draws random inputs: keys, values and queries with the shapes
and value distributions of the five workloads (a tiny MHA case, a Llama-2-7B
shaped layer, a Llama-2-13B shaped mixed-precision layer, a Llama-3-8B shaped
GQA layer and a 1M-token pre-RoPE layer).  It holds none of the quantization or
attention arithmetic; the CPU oracle and the CUDA library both consume the
host arrays produced here.

The pages measure on real models and datasets (CoQA, GSM8K, LongBench,
Wikitext-2); these seeded stand-ins replace them.  Keys carry fixed outlier
channels, which is the structure the per-channel key quantizer is built for
("Keys: fixed channels carry outliers" on the unite.ai page).
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libkvqsynth.so")

TENSOR_K, TENSOR_V, TENSOR_Q, TENSOR_QNOISE, TENSOR_PICK, TENSOR_OUTLIER = 1, 2, 3, 4, 5, 6

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the generator into synth/_lib (plain C, no target-specific flags)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.synth_fill_f16.restype = ctypes.c_int
            lib.synth_fill_f16.argtypes = [ctypes.c_uint64, ctypes.c_uint64] + [ctypes.c_int64] * 7 + [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.synth_stream_base.restype = ctypes.c_uint64
            lib.synth_stream_base.argtypes = [ctypes.c_uint64] * 4
            lib.synth_draw.restype = ctypes.c_uint64
            lib.synth_draw.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_normal.restype = ctypes.c_double
            lib.synth_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            _lib = lib
    return _lib


def stream_base(seed: int, tensor: int, b: int, h: int) -> int:
    return int(_get().synth_stream_base(seed, tensor, b, h))


def draw(base: int, k: int) -> int:
    return int(_get().synth_draw(base, k))


def normal(base: int, i: int) -> float:
    return float(_get().synth_normal(base, i))


def _threads() -> int:
    """Generator threads: KVQ_SYNTH_THREADS when set (a process pinned to one core sets 1), else the cores."""
    env = os.environ.get("KVQ_SYNTH_THREADS")
    if env:
        return max(1, min(64, int(env)))
    return max(1, min(64, os.cpu_count() or 1))


@dataclasses.dataclass(frozen=True)
class Workload:
    """One workload: shapes, method parameters and the input recipe."""
    name: str
    batch: int
    kv_heads: int
    q_heads: int
    head_dim: int
    prefill_tokens: int
    decode_steps: int
    k_bits: int
    v_bits: int
    group: int
    residual: int
    k_sparse: int          # sparse fp16 entries per key vector (0 = dense only)
    rope: int              # 1: keys are stored pre-RoPE and rotated at decode
    rope_base: float
    key_outliers: str      # "per_head4": 4 channels per kv head ~ sign*N(40,5); "layer1pct": 1% of (head, channel) pairs ~ sign*N(50,5)
    queries: str           # "normal": N(0,1); "peaked": biased toward 8 past keys (84% of mass on 5% of tokens)
    seed: int
    sink: int = 0          # attention-sink tokens kept fp16 (0: none)
    k_levels: tuple = ()   # non-uniform codebook levels in steps (empty: uniform codes)
    v_levels: tuple = ()

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def max_tokens(self) -> int:
        return self.prefill_tokens + self.decode_steps

    @property
    def group_q(self) -> int:
        return self.q_heads // self.kv_heads

    def scaled(self, **kw) -> "Workload":
        """Same method parameters and recipe, other sizes (for oracle-sized parity cases)."""
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    0: Workload("tiny 2-bit MHA decode: B=1, 4/4 heads, D=128, T=1024, K2V2, G=32, R=128",
                1, 4, 4, 128, 1024, 1, 2, 2, 32, 128, 0, 0, 10000.0, "per_head4", "normal", 0),
    1: Workload("Llama-2-7B-shaped layer: B=8, 32/32 heads, D=128, T=4096 + 64 decode steps, K2V2, G=32, R=128",
                8, 32, 32, 128, 4096, 64, 2, 2, 32, 128, 0, 0, 10000.0, "per_head4", "normal", 1),
    2: Workload("Llama-2-13B-shaped layer: B=16, 40/40 heads, D=128, T=8192, K4V2, G=32, R=128, peaked queries",
                16, 40, 40, 128, 8192, 1, 4, 2, 32, 128, 0, 0, 10000.0, "layer1pct", "peaked", 2),
    3: Workload("Llama-3-8B-shaped GQA layer: B=32, 8 KV / 32 Q heads, D=128, T=32768, K2V2, G=32, R=128",
                32, 8, 32, 128, 32768, 1, 2, 2, 32, 128, 0, 0, 10000.0, "per_head4", "normal", 3),
    4: Workload("1M-token pre-RoPE layer: B=1, 8 KV / 32 Q heads, D=128, T=1048576, K3V3, G=64, R=128, 1% sparse K",
                1, 8, 32, 128, 1048576, 1, 3, 3, 64, 128, 2, 1, 10000.0, "per_head4", "normal", 4),
}


def key_channel_stats(w: Workload):
    """Per (kv head, channel) mean and std of the keys, with the outlier channels.

    per_head4: in every kv head, 4 distinct seeded channels draw sign*N(40, 5)
    with a seeded sign fixed per (head, channel); the rest draw N(0, 1).
    layer1pct: round(0.01 * Hkv * D) distinct seeded (head, channel) pairs draw
    sign*N(50, 5); the rest N(0, 1).
    """
    H, D = w.kv_heads, w.head_dim
    mean = np.zeros((H, D), np.float64)
    std = np.ones((H, D), np.float64)
    if w.key_outliers == "per_head4":
        for h in range(H):
            base = stream_base(w.seed, TENSOR_OUTLIER, 0, h)
            chosen = []
            k = 0
            while len(chosen) < 4:
                c = draw(base, k) % D
                k += 1
                if c not in chosen:
                    chosen.append(c)
            for c in chosen:
                sign = 1.0 if (draw(base, 1000 + c) & 1) else -1.0
                mean[h, c] = 40.0 * sign
                std[h, c] = 5.0
    elif w.key_outliers == "layer1pct":
        n = int(round(0.01 * H * D))
        base = stream_base(w.seed, TENSOR_OUTLIER, 0, 0)
        chosen = []
        k = 0
        while len(chosen) < n:
            p = draw(base, k) % (H * D)
            k += 1
            if p not in chosen:
                chosen.append(p)
        for p in chosen:
            sign = 1.0 if (draw(base, 100000 + p) & 1) else -1.0
            mean[p // D, p % D] = 50.0 * sign
            std[p // D, p % D] = 5.0
    else:
        raise ValueError(w.key_outliers)
    return mean, std


def _fill(seed, tensor, b0, nb, h0, nh, t0, nt, D, mean, std, out=None):
    mean = np.ascontiguousarray(mean, np.float64)
    std = np.ascontiguousarray(std, np.float64)
    assert mean.shape == (nh, D) and std.shape == (nh, D)
    if out is None:
        out = np.empty((nb, nh, nt, D), np.float16)
    assert out.dtype == np.float16 and out.flags.c_contiguous and out.shape == (nb, nh, nt, D)
    rc = _get().synth_fill_f16(seed, tensor, b0, nb, h0, nh, t0, nt, D,
                               mean.ctypes.data, std.ctypes.data, out.ctypes.data, _threads())
    if rc != 0:
        raise ValueError("synth_fill_f16 rejected its arguments")
    return out


def keys(w: Workload, b0=0, nb=None, h0=0, nh=None, t0=0, nt=None, out=None) -> np.ndarray:
    """Keys K[b][kvh][t][c] for t in [t0, t0+nt); tokens >= prefill_tokens are the appended ones."""
    nb = w.batch - b0 if nb is None else nb
    nh = w.kv_heads - h0 if nh is None else nh
    nt = w.max_tokens - t0 if nt is None else nt
    mean, std = key_channel_stats(w)
    return _fill(w.seed, TENSOR_K, b0, nb, h0, nh, t0, nt, w.head_dim, mean[h0:h0 + nh], std[h0:h0 + nh], out)


def values(w: Workload, b0=0, nb=None, h0=0, nh=None, t0=0, nt=None, out=None) -> np.ndarray:
    """Values V[b][kvh][t][c] ~ N(0, 1)."""
    nb = w.batch - b0 if nb is None else nb
    nh = w.kv_heads - h0 if nh is None else nh
    nt = w.max_tokens - t0 if nt is None else nt
    D = w.head_dim
    return _fill(w.seed, TENSOR_V, b0, nb, h0, nh, t0, nt, D, np.zeros((nh, D)), np.ones((nh, D)), out)


def _normal_rows(seed, tensor, b, h, row, D):
    return _fill(seed, tensor, b, 1, h, 1, row, 1, D, np.zeros((1, D)), np.ones((1, D)))[0, 0, 0].astype(np.float64)


def queries(w: Workload, step: int, keys_of=None) -> np.ndarray:
    """Query q[b][hq][c] (fp16) of decode step `step` (0-based).

    normal: N(0, 1), already rotated (post-RoPE at its own position).
    peaked: q = alpha*u + g, u the normalised sum of 8 seeded past keys of the
    head's kv head, g ~ N(0, 1); alpha is found by bisection so that the top
    ceil(0.05*T) tokens hold 0.84 of the softmax mass over the raw keys (the
    84.3% attention sparsity on the unite.ai page, "Values" section).
    `keys_of(b, kvh)` must return the raw fp16 keys [T][D] of that unit at this
    step (T = prefill_tokens + step + 1); it defaults to regenerating them.
    """
    B, Hq, D = w.batch, w.q_heads, w.head_dim
    if w.queries == "normal":
        return _fill(w.seed, TENSOR_Q, 0, B, 0, Hq, step, 1, D, np.zeros((Hq, D)), np.ones((Hq, D)))[:, :, 0, :].copy()
    if w.queries != "peaked":
        raise ValueError(w.queries)
    T = w.prefill_tokens + step + 1
    out = np.empty((B, Hq, D), np.float16)
    for b in range(B):
        for h in range(Hq):
            kvh = h // w.group_q
            K = keys(w, b, 1, kvh, 1, 0, T)[0, 0] if keys_of is None else keys_of(b, kvh)
            K = np.asarray(K, np.float64)
            base = stream_base(w.seed, TENSOR_PICK, b, h)
            picks = [draw(base, j) % w.prefill_tokens for j in range(8)]
            s = K[picks].sum(axis=0)
            u = s / np.linalg.norm(s)
            g = _normal_rows(w.seed, TENSOR_QNOISE, b, h, step, D)
            alpha = peaked_alpha(K @ u, K @ g, w.softmax_scale, target=0.84)
            out[b, h] = (alpha * u + g).astype(np.float16)
    return out


def top_mass(a, n, alpha, scale, frac=0.05):
    """Share of softmax mass held by the top ceil(frac*T) tokens of scale*(alpha*a + n)."""
    s = scale * (alpha * a + n)
    s = s - s.max()
    p = np.exp(s)
    k = int(math.ceil(frac * len(s)))
    top = np.partition(p, len(p) - k)[len(p) - k:]
    return float(top.sum() / p.sum())


def peaked_alpha(a, n, scale, target=0.84):
    if top_mass(a, n, 0.0, scale) >= target:
        return 0.0
    hi = 1.0
    while top_mass(a, n, hi, scale) < target and hi < 1e6:
        hi *= 2.0
    lo = 0.0
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        if top_mass(a, n, mid, scale) < target:
            lo = mid
        else:
            hi = mid
    return hi
