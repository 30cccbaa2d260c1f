"""Axis ablation: score and attention-output error of quantizing keys and values along either axis.

The comparison at the centre of "KV cache has a geometry problem, not a bit problem" (sections
"Keys" and "Values"): keys carry a few outlier channels, so groups along the tokens of a channel
(per-channel) keep attention scores far better than groups across the channels of a token
(per-token); values are read as weighted sums over tokens.  Every step runs in the library's
kernels (kvq_axis_quantize, kvq_axis_dequantize, kvq_axis_attention); torch only holds device
memory, and the error norms are taken on the host.

    python bench_ablation.py        # (repository root) table for a seeded outlier-key workload
"""
from __future__ import annotations

import numpy as np

from .kvq import KVQ_AXIS_CHANNELS, KVQ_AXIS_TOKENS, kvq_axis_attention, kvq_axis_dequantize, kvq_axis_quantize

AXES = {"channel": KVQ_AXIS_TOKENS, "token": KVQ_AXIS_CHANNELS}  # "per-channel" groups run along tokens


def quantize(x, bits: int, group: int, axis: int, stream=None):
    """x: CUDA fp16 [U][T][D] -> (codes u8 [U][T][D], zero, scale fp16 in the axis' layout)."""
    import torch
    U, T, D = x.shape
    meta = (U, T // group, D) if axis == KVQ_AXIS_TOKENS else (U, T, D // group)
    codes = torch.empty((U, T, D), dtype=torch.uint8, device=x.device)
    z = torch.empty(meta, dtype=torch.float16, device=x.device)
    s = torch.empty(meta, dtype=torch.float16, device=x.device)
    kvq_axis_quantize(x, U, T, D, bits, group, axis, codes, z, s, stream)
    return codes, z, s


def dequantize(codes, z, s, group: int, axis: int, stream=None):
    import torch
    U, T, D = codes.shape
    out = torch.empty((U, T, D), dtype=torch.float32, device=codes.device)
    kvq_axis_dequantize(codes, z, s, U, T, D, group, axis, out, stream)
    return out


def attention(k, v, q, scale: float, with_scores: bool = False, stream=None):
    """k, v: CUDA [U][T][D] fp32 or fp16; q: CUDA fp16 [U][Hg][D] -> (out fp32 [U][Hg][D], scores or None)."""
    import torch
    U, T, D = k.shape
    Hg = q.shape[1]
    out = torch.empty((U, Hg, D), dtype=torch.float32, device=k.device)
    scores = torch.empty((U, Hg, T), dtype=torch.float32, device=k.device) if with_scores else None
    kvq_axis_attention(k, v, 1 if k.dtype == torch.float32 else 0, q, U, Hg, T, D, scale, scores, out, stream)
    return out, scores


def _rel_fro(a, b):
    return float(np.linalg.norm((a - b).ravel()) / np.linalg.norm(b.ravel()))


def _max_rel_inf(a, b):
    a = a.reshape(-1, a.shape[-1])
    b = b.reshape(-1, b.shape[-1])
    return float((np.abs(a - b).max(axis=1) / np.abs(b).max(axis=1)).max())


def axis_errors(K, V, Q, bits: int, group: int, scale: float) -> dict:
    """Errors of the four (key axis, value axis) choices against exact attention over K, V.

    K, V: CUDA fp16 [U][T][D]; Q: CUDA fp16 [U][Hg][D].  Returns {(key_axis, value_axis):
    {"score_rel_fro", "out_rel_fro", "out_max_rel_inf"}} with axes named "channel" / "token"."""
    import torch
    ref_out, ref_sc = attention(K, V, Q, scale, with_scores=True)
    deq = {}
    for name, ax in AXES.items():
        deq[("K", name)] = dequantize(*quantize(K, bits, group, ax), group, ax)
        deq[("V", name)] = dequantize(*quantize(V, bits, group, ax), group, ax)
    torch.cuda.synchronize()
    ref_out, ref_sc = ref_out.cpu().numpy(), ref_sc.cpu().numpy()
    res = {}
    for ka in AXES:
        for va in AXES:
            out, sc = attention(deq[("K", ka)], deq[("V", va)], Q, scale, with_scores=True)
            out, sc = out.cpu().numpy(), sc.cpu().numpy()
            res[(ka, va)] = {"score_rel_fro": _rel_fro(sc, ref_sc), "out_rel_fro": _rel_fro(out, ref_out),
                             "out_max_rel_inf": _max_rel_inf(out, ref_out)}
    return res


def time_kernels(K, V, Q, bits: int, group: int, scale: float, reps: int = 20) -> dict:
    """Mean device time (CUDA events, after a warm-up) and bytes moved per call of each kernel."""
    import torch
    U, T, D = K.shape
    res = {}

    def timed(fn):
        fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e-3

    for name, ax in AXES.items():
        meta = (T // group) * D if ax == KVQ_AXIS_TOKENS else T * (D // group)
        q = quantize(K, bits, group, ax)
        sec = timed(lambda: quantize(K, bits, group, ax))
        res[f"quantize per-{name}"] = {"s": sec, "bytes": U * (T * D * 2 + T * D + 2 * meta * 2)}
        sec = timed(lambda: dequantize(*q, group, ax))
        res[f"dequantize per-{name}"] = {"s": sec, "bytes": U * (T * D + 2 * meta * 2 + T * D * 4)}
    kd = dequantize(*quantize(K, bits, group, KVQ_AXIS_TOKENS), group, KVQ_AXIS_TOKENS)
    vd = dequantize(*quantize(V, bits, group, KVQ_AXIS_CHANNELS), group, KVQ_AXIS_CHANNELS)
    sec = timed(lambda: attention(kd, vd, Q, scale))
    res["attention fp32 rows"] = {"s": sec, "bytes": U * 2 * T * D * 4}
    for r in res.values():
        r["GBps"] = r["bytes"] / r["s"] / 1e9
    return res
