#!/usr/bin/env python
"""Benchmark: decode-attention KV tokens/s on the Llama-2-7B-shaped 2-bit layer.

Workload (one step): for each of L layer caches (default 4) of the
Llama-2-7B-shaped layer (B=8, 32 KV = 32 query heads, D=128, K2V2, G=32,
R=128): prefill 4096 tokens (quantize-and-pack), then 64 fused decode steps
(kvq_decode_step): each appends one token and runs decode attention over the
whole cache in one launch (the first one flushes the full fp16 window into a
page before it).  Layers are visited
in turn inside each decode step, as a model does, so the 101-109 MB cache of
one layer is never L2-resident when it is read again (4 caches > 129 MB L2).

value  = KV tokens attended per second over the whole step (sum over decodes
         of B*T, T = 4097..4160), inputs resident in HBM.
e2e    = the same metric through the public C-ABI calls with the inputs in
         pinned host memory: every step copies its prefill inputs, appended
         tokens and queries host->device and reads every output back.  The
         copies run on streams of their own into one device buffer per layer
         (and one per step for the decode inputs), so the next step's copies
         overlap the current step's compute.
roofline: the dominant kernel (decode attention) against the measured HBM
         copy bandwidth: algorithmic bytes per call (packed codes + scales
         and zero points + fp16 window + q + out + the new token's window
         store) / mean time of the decode steps that do not flush, each timed
         with CUDA events around the whole call (the decode kernel and the
         small kernel that merges its partials, launched back to back).

`--impl reference` times the CPU oracle (the plain fp64/fp32 C reference the
tests check against) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import tempfile
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode-attention KV tokens/s and HBM GB/s (% of GB300 roofline) at 2-bit"
UNIT = "KV tokens/s"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description="Decode-attention throughput of the quantized KV cache (one JSON line).")
    ap.add_argument("--gpus", type=int, default=1, help="GPUs (one process each under torchrun; replicas)")
    ap.add_argument("--steps", type=int, default=100, help="timed steps")
    ap.add_argument("--warmup", type=int, default=3, help="untimed warm-up steps (at least 3)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours",
                    help="the CUDA library, or the CPU oracle on a bounded sample")
    ap.add_argument("--layers", type=int, default=4, help="layer caches visited in turn per step")
    ap.add_argument("--workload", type=int, default=1, help="index into synth.WORKLOADS")
    ap.add_argument("--graph", type=int, default=1, help="replay each step as one CUDA graph (1) or call directly (0)")
    ap.add_argument("--e2e-steps", type=int, default=10, help="steps timed end to end from pinned host buffers")
    ap.add_argument("--timing-steps", type=int, default=3, help="extra direct-call steps timed per decode launch")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi clocks")
    ap.add_argument("--sink", type=int, default=0, help="attention-sink tokens kept fp16 (0: none)")
    ap.add_argument("--codebook", action="store_true",
                    help="non-uniform levels (cosine-spaced, denser at the group's ends) for keys and values")
    return ap.parse_args(argv)


def codebook_levels(bits):
    """Cosine-spaced levels in steps: 0 and L kept, denser near both ends of the group's range."""
    L = (1 << bits) - 1
    lev = (L * (0.5 - 0.5 * np.cos(np.pi * np.arange(L + 1) / L))).astype(np.float32)
    lev[0], lev[-1] = 0.0, float(L)
    return lev


def workload_of(args):
    w = synth.WORKLOADS[args.workload]
    if args.sink:
        w = w.scaled(sink=args.sink)
    if args.codebook:
        w = dataclasses.replace(w, k_levels=tuple(codebook_levels(w.k_bits).tolist()),
                                v_levels=tuple(codebook_levels(w.v_bits).tolist()))
    return w


# ------------------------------------------------------------------ distributed helpers

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend)
            self.pg = dist
            self.backend = backend

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = f"cuda:{self.local_rank}" if self.backend == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        dev = f"cuda:{self.local_rank}" if self.backend == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ workload accounting

def quantized_tokens(T, R):
    return 0 if T <= 0 else R * ((T - 1) // R)


def decode_bytes(w, T):
    """Algorithmic bytes of one decode launch over T cached tokens (all units), plus q and out."""
    D, G = w.head_dim, w.group
    n_s = min(T, w.sink)
    Tq = quantized_tokens(T - n_s, w.residual)
    n_r = T - n_s - Tq
    per_unit = (Tq * D * (w.k_bits + w.v_bits) // 8 + (Tq // G) * D * 4 + Tq * (D // G) * 4
                + Tq * w.k_sparse * 3 + (n_r + n_s) * D * 4)
    return w.batch * w.kv_heads * per_unit + 2 * w.batch * w.q_heads * D * 2


def decode_step_bytes(w, T):
    """decode_bytes plus the store of the new token's key and value into the window (a fused step)."""
    return decode_bytes(w, T) + w.batch * w.kv_heads * w.head_dim * 4


def step_tokens(w, layers):
    T0 = w.prefill_tokens
    return layers * sum(w.batch * (T0 + i) for i in range(1, w.decode_steps + 1))


def workload_config(w, layers, graph, world):
    return {
        "workload": w.name,
        "layers": layers,
        "batch": w.batch, "kv_heads": w.kv_heads, "q_heads": w.q_heads, "head_dim": w.head_dim,
        "prefill_tokens": w.prefill_tokens, "decode_steps": w.decode_steps,
        "k_bits": w.k_bits, "v_bits": w.v_bits, "group": w.group, "residual": w.residual,
        **({"sink_tokens": w.sink} if w.sink else {}),
        **({"codebook": "cosine-spaced levels (non-uniform)"} if w.k_levels else {}),
        "step": f"{layers} layers x (prefill {w.prefill_tokens}) + {w.decode_steps} x {layers} layers x "
                f"fused decode step (append + decode attention, one launch)",
        "l2": f"inputs larger than L2: {layers} layer caches of "
              f"{decode_bytes(w, w.prefill_tokens + 1) / 1e6:.0f} MB visited in turn",
        "launch": "one CUDA graph per step" if graph else "direct C-ABI calls",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


# ------------------------------------------------------------------ clocks

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, enabled=True):
        self.proc = None
        self.path = None
        if not enabled:
            return
        try:
            # samples go to a file of their own; KVQ_CLOCKS_DIR keeps it (default: a temporary file)
            keep = os.environ.get("KVQ_CLOCKS_DIR")
            if keep:
                os.makedirs(keep, exist_ok=True)
                self.path = os.path.join(keep, f"clocks_bench_{os.getpid()}.csv")
            else:
                fd, self.path = tempfile.mkstemp(prefix="clocks_bench_", suffix=".csv")
                os.close(fd)
            self.keep = bool(keep)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not self.keep:
            os.remove(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle baseline

def cpu_baseline(w, seconds):
    """The oracle as it stands, one (sequence, kv head) unit at a time: prefill, then every decode step
    (append + fp64 attention), until `seconds` of oracle time.  One unit is 1/Hkv of a sequence's work,
    so it is credited with sum_i T_i / Hkv tokens, in the GPU's unit.  Input generation is not timed."""
    import oracle
    T0, steps = w.prefill_tokens, w.decode_steps
    Q = [synth.queries(w, i) for i in range(steps)]
    busy = 0.0
    tokens = 0.0
    units = 0
    for unit in range(w.batch * w.kv_heads):
        b, kvh = divmod(unit, w.kv_heads)
        K = synth.keys(w, b, 1, kvh, 1)[0, 0]
        V = synth.values(w, b, 1, kvh, 1)[0, 0]
        hs = slice(kvh * w.group_q, (kvh + 1) * w.group_q)
        t0 = time.perf_counter()
        u = oracle.OracleUnit.for_workload(w)
        u.prefill(K[:T0], V[:T0])
        for i in range(steps):
            u.append(K[T0 + i], V[T0 + i])
            u.attention(Q[i][b, hs], w.softmax_scale)
            tokens += (T0 + i + 1) / w.kv_heads
        busy += time.perf_counter() - t0
        units += 1
        if busy >= seconds:
            break
    return {"value": tokens / busy, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{units} (sequence, kv head) units x (prefill {T0} + {steps} x (append + attention)), "
                      f"single-threaded C oracle, {busy:.1f} s"}


# ------------------------------------------------------------------ our implementation

def run_ours(args, dist):
    import torch

    import bit_asymmetric_kv_kvq_gb300 as kvq
    from bit_asymmetric_kv_kvq_gb300 import _build

    if _build.stale():
        _build.build()
    w = workload_of(args)
    L = args.layers
    dev = torch.device(f"cuda:{dist.local_rank}")
    torch.cuda.set_device(dev)
    T0, S = w.prefill_tokens, w.decode_steps
    B, Hkv, Hq, D = w.batch, w.kv_heads, w.q_heads, w.head_dim

    # inputs (same synthetic sequence for every layer; each layer has its own cache)
    K = synth.keys(w)
    V = synth.values(w)
    Q = np.stack([synth.queries(w, i) for i in range(S)])  # [S][B][Hq][D]
    k_pre = torch.from_numpy(np.ascontiguousarray(K[:, :, :T0])).to(dev)
    v_pre = torch.from_numpy(np.ascontiguousarray(V[:, :, :T0])).to(dev)
    k_new = torch.from_numpy(np.ascontiguousarray(K[:, :, T0:T0 + S].transpose(2, 0, 1, 3))).to(dev)  # [S][B][Hkv][D]
    v_new = torch.from_numpy(np.ascontiguousarray(V[:, :, T0:T0 + S].transpose(2, 0, 1, 3))).to(dev)
    q_dev = torch.from_numpy(Q).to(dev)
    out = torch.empty((L, S, B, Hq, D), dtype=torch.float16, device=dev)
    caches = [kvq.KVCache.for_workload(w, device=dist.local_rank) for _ in range(L)]
    handles = [c.handle for c in caches]
    Lb = kvq.lib()
    stream = torch.cuda.Stream(dev)
    sh = stream.cuda_stream
    kp, vp = k_pre.data_ptr(), v_pre.data_ptr()
    tok_bytes = B * Hkv * D * 2
    q_bytes = B * Hq * D * 2
    knp = [k_new.data_ptr() + i * tok_bytes for i in range(S)]
    vnp = [v_new.data_ptr() + i * tok_bytes for i in range(S)]
    qp = [q_dev.data_ptr() + i * q_bytes for i in range(S)]
    op = [[out[l, i].data_ptr() for i in range(S)] for l in range(L)]

    def check(st, what):
        if st != 0:
            raise kvq.KVQError(st, what)

    def step(events=None):
        for h in handles:
            check(Lb.kvq_reset(h), "reset")
            check(Lb.kvq_prefill_quantize(h, kp, vp, T0, sh), "prefill")
        n = 0
        for i in range(S):
            for l, h in enumerate(handles):
                if events is not None:
                    events[n][0].record(stream)
                check(Lb.kvq_decode_step(h, knp[i], vnp[i], qp[i], op[l][i], sh), "decode step")
                if events is not None:
                    events[n][1].record(stream)
                n += 1

    def launches():
        return sum(Lb.kvq_launch_count(h) for h in handles)

    graph = None
    with torch.cuda.stream(stream):
        step()  # first call: kernel attributes, module load
    torch.cuda.synchronize(dev)
    if args.graph:
        l0 = launches()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        graph_launches = launches() - l0

        def run():
            graph.replay()
    else:
        graph_launches = None

        def run():
            step()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            run()
    torch.cuda.synchronize(dev)
    for h in handles:
        if Lb.kvq_sync_status(h, sh) != 0:
            raise RuntimeError("device-side error after warm-up")

    # ---------------- timed region
    clocks = Clocks(dist.local_rank, enabled=not args.no_clocks)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l_before = launches()
    dist.barrier()
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            run()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    dist.barrier()
    ms_total = ev0.elapsed_time(ev1)
    clock_info = clocks.stop()
    n_launch = (launches() - l_before) if graph is None else graph_launches * args.steps
    for h in handles:
        if Lb.kvq_sync_status(h, sh) != 0:
            raise RuntimeError("device-side error in the timed region")
    ms_step = dist.max(ms_total / args.steps)

    # ---------------- per-launch timing of decode attention (direct calls, CUDA events on the launch stream);
    # decode steps 1..S-1 are one launch each (step 0 also flushes the window and is left out)
    n_dec = S * L
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_dec)]
    durs = []
    with torch.cuda.stream(stream):
        for _ in range(args.timing_steps):
            step(evs)
            torch.cuda.synchronize(dev)
            durs.extend(a.elapsed_time(b) for a, b in evs[L:])
    dec_ms = statistics.mean(durs) if durs else float("nan")
    dec_bytes = statistics.mean(decode_step_bytes(w, T0 + 1 + i) for i in range(1, S))
    import json as _json
    peaks = _json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = peaks.get("hbm_gbs", 6800.0)
    achieved = dec_bytes / (dec_ms * 1e-3) / 1e9
    traffic = decode_traffic(w)

    # ---------------- end to end through the C ABI from pinned host memory
    e2e = run_e2e(args, w, dist, caches, stream) if args.e2e_steps > 0 else None

    tokens = step_tokens(w, L)
    total_tokens = dist.sum(tokens)
    value = total_tokens / (ms_step * 1e-3)
    for c in caches:
        c.close()
    return {
        "value": value, "ms_per_step": ms_step, "gpu_launches": int(n_launch),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "kernel": "decode attention call: decode_mma_kernel (tensor cores) + merge_kernel",
                     "bytes_per_launch": dec_bytes, "ms_per_launch": dec_ms,
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if peaks else "fallback 6.8 TB/s"},
        "decode_only": {"value": B * statistics.mean(T0 + 1 + i for i in range(1, S)) / (dec_ms * 1e-3),
                        "unit": UNIT, "ms_per_launch": dec_ms},
        "clocks": clock_info, "e2e": e2e,
        "config": workload_config(w, L, graph is not None, dist.world),
    }


DECODE_SOURCES = ("kvq_decode_mma.cu", "kvq_merge.cuh", "kvq_ptx.cuh", "kvq_internal.h")
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "decode_mma_kernel_traffic.txt")


def kernel_revision():
    """Hash of the decode kernel's sources: DRAM counters are valid only for the kernel they were taken on."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_asymmetric_kv_kvq_gb300", "csrc")
    for f in DECODE_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def decode_traffic(w):
    """DRAM read+write bytes per decode launch from the committed ncu summary, or None.

    The summary holds `key: value` lines; its figure counts only when it was taken
    on this workload and on the current decode kernel sources."""
    if not os.path.exists(TRAFFIC_SUMMARY):
        return None
    kv = {}
    for line in open(TRAFFIC_SUMMARY):
        if ":" in line and not line.startswith((" ", "#")):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("workload") != w.name or kv.get("kernel_rev") != kernel_revision():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


COPY_STREAMS = 4  # host->device copy streams for the prefill inputs (several copy engines)


def run_e2e(args, w, dist, caches, stream):
    import torch

    dev = torch.device(f"cuda:{dist.local_rank}")
    T0, S, L = w.prefill_tokens, w.decode_steps, len(caches)
    K = synth.keys(w)
    V = synth.values(w)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    hk, hv = pin(K[:, :, :T0]), pin(V[:, :, :T0])
    hkn = pin(K[:, :, T0:T0 + S].transpose(2, 0, 1, 3))
    hvn = pin(V[:, :, T0:T0 + S].transpose(2, 0, 1, 3))
    hq = pin(np.stack([synth.queries(w, i) for i in range(S)]))
    hout = torch.empty((L, S) + tuple(hq.shape[1:]), dtype=torch.float16).pin_memory()
    # Copies run on streams of their own and overlap the compute; every byte is still copied inside
    # the timed region, and the compute stream waits for each copy it uses.  Every layer has its own
    # device buffer for its prompt, so all of the next step's prompts can stream in while this step
    # decodes.  A step's decode inputs (new keys, new values, queries of all its decode steps) arrive
    # in one transfer each on a stream of their own, before the decodes that read them: small copies
    # issued on the compute stream between decode launches would sit in the copy queue ahead of the
    # next step's prompts.
    nbuf = L
    copy_streams = [torch.cuda.Stream(dev) for _ in range(COPY_STREAMS)]
    dec_stream = torch.cuda.Stream(dev)
    dk = [torch.empty_like(hk, device=dev) for _ in range(nbuf)]
    dv = [torch.empty_like(hv, device=dev) for _ in range(nbuf)]
    copied = [[torch.cuda.Event() for _ in copy_streams] for _ in range(nbuf)]
    used = [torch.cuda.Event() for _ in range(nbuf)]
    dec_copied, dec_used = torch.cuda.Event(), torch.cuda.Event()
    # the batch dimension is split across the copy streams: each takes whole sequences
    parts = np.array_split(np.arange(hk.shape[0]), len(copy_streams))
    dkn = torch.empty_like(hkn, device=dev)
    dvn = torch.empty_like(hvn, device=dev)
    dq = torch.empty_like(hq, device=dev)
    dout = torch.empty(hout.shape, dtype=torch.float16, device=dev)
    h2d = 0
    d2h = 0

    def step():
        nonlocal h2d, d2h
        for l, c in enumerate(caches):
            b = l % nbuf
            for cs, part, ev in zip(copy_streams, parts, copied[b]):
                if len(part) == 0:
                    continue
                lo, hi = int(part[0]), int(part[-1]) + 1
                cs.wait_event(used[b])  # the prefill that read this buffer last has finished
                with torch.cuda.stream(cs):
                    dk[b][lo:hi].copy_(hk[lo:hi], non_blocking=True)
                    dv[b][lo:hi].copy_(hv[lo:hi], non_blocking=True)
                ev.record(cs)
                stream.wait_event(ev)
            h2d += hk.nbytes + hv.nbytes
            c.reset()
            c.prefill_quantize(dk[b], dv[b], stream=stream)
            used[b].record(stream)
        dec_stream.wait_event(dec_used)  # the previous step's decodes have read the decode inputs
        with torch.cuda.stream(dec_stream):
            dkn.copy_(hkn, non_blocking=True)
            dvn.copy_(hvn, non_blocking=True)
            dq.copy_(hq, non_blocking=True)
        dec_copied.record(dec_stream)
        h2d += hkn.nbytes + hvn.nbytes + hq.nbytes
        stream.wait_event(dec_copied)
        for i in range(S):
            for l, c in enumerate(caches):
                c.decode_step(dkn[i], dvn[i], dq[i], dout[l, i], stream=stream)
        dec_used.record(stream)
        hout.copy_(dout, non_blocking=True)
        d2h += hout.nbytes

    with torch.cuda.stream(stream):
        step()
        torch.cuda.synchronize(dev)
        h2d = d2h = 0
        dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for cs in copy_streams + [dec_stream]:
            cs.wait_event(e0)  # no copy of the timed steps starts before the clock does
        for _ in range(args.e2e_steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    dist.barrier()
    ms = dist.max(e0.elapsed_time(e1) / args.e2e_steps)
    total = dist.sum(step_tokens(w, L))
    return {"value": total / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d // args.e2e_steps, "d2h_bytes_per_step": d2h // args.e2e_steps}


# ------------------------------------------------------------------ reference arm: the CPU oracle

def run_reference(args, dist):
    w = workload_of(args)
    L = args.layers
    # each step: a bounded sample of the workload through the oracle
    per = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(w, per)
    t0 = time.perf_counter()
    vals = []
    for _ in range(args.steps):
        vals.append(cpu_baseline(w, per))
    el = time.perf_counter() - t0
    value = statistics.mean(v["value"] for v in vals)
    return {
        "impl": "reference", "value": value, "ms_per_step": el / args.steps * 1e3,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": vals[-1]["sample"] + f"; {args.steps} steps of ~{per:.1f} s"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0, "config": workload_config(w, L, False, 1),
    }


def main(argv=None):
    args = parse_args(argv)
    dist = Dist()
    if args.impl == "reference" and dist.world > 1 and dist.rank != 0:
        dist.close()
        return 0
    if args.impl == "reference":
        res = run_reference(args, dist)
        line = {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)", **res}
        print(json.dumps(line))
        dist.close()
        return 0
    res = run_ours(args, dist)
    line = {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u2 codes, f16 tensor-core mma (f32 accumulate), f16 out",
            "data": "synthetic (seeded): keys N(0,1) with 4 outlier channels per head ~ sign*N(40,5), values N(0,1)",
            "config": res["config"], "e2e": res["e2e"], "roofline": res["roofline"],
            "decode_only": res["decode_only"], "gpu_launches": res["gpu_launches"], "clocks": res["clocks"]}
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(workload_of(args), args.cpu_seconds)
    if dist.rank == 0:
        print(json.dumps(line))
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
