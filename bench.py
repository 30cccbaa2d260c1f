#!/usr/bin/env python
"""Benchmark: decode-attention KV tokens/s of the 2-bit quantized KV cache (one JSON line).

Default workload: the Llama-3-8B-shaped GQA layer (B=32, 8 KV / 32 query heads,
D=128, context 32768, K2V2, G=32, R=128), the largest 2-bit workload.  One step,
for each of L layer caches (default 4): a full prefill quantize-and-pack of the
32768-token prompt, then the workload's fused decode steps (kvq_decode_step:
append one token, flushing the full fp16 window into a page first, then decode
attention over the whole cache).  Every layer reads a 4.3 GB prompt and its own
805 MB cache, so nothing a kernel reads is L2-resident (L2 is 129 MB).  The other
workloads run with --workload N (N = 0..4).

value   = KV tokens attended per second over the whole step (sum over decodes of
          B*T), inputs resident in HBM, one CUDA graph per step.
decode  = the decode-attention call alone (decode kernel + the kernel merging its
          partials), timed per call with CUDA events on the launching stream over
          at least 50 calls that rotate over the L caches: median and p90, KV
          tokens/s = B*T / median, and HBM GB/s of its algorithmic bytes (packed
          codes + scales and zero points + sparse entries + fp16 window + q + out).
prefill = the prefill call alone, timed the same way.
roofline: the kernel that takes the larger share of the step (by the medians
          above), against the measured HBM copy bandwidth.
e2e     = the same metric through the public C-ABI calls with the inputs in
          pinned host memory: every step copies its prompts, appended tokens and
          queries host->device and reads every output back.
cpu_baseline: the CPU oracle (the plain C reference the tests check against) on
          a bounded sample of the same workload, on one thread and on every host
          core (one process per core, each over its own (sequence, kv head) units).

After the timed region one sampled (sequence, kv head) unit of the last step is
checked against the oracle: its packed stores bit for bit and its attention
output within 2e-3.

`--impl reference` times the CPU oracle on every host core, step by step.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode-attention KV tokens/s and HBM GB/s (% of GB300 roofline) at 2-bit"
UNIT = "KV tokens/s"
DEFAULT_WORKLOAD = 3


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description="Decode-attention throughput of the quantized KV cache (one JSON line).")
    ap.add_argument("--gpus", type=int, default=1, help="GPUs (one process each under torchrun; replicas)")
    ap.add_argument("--steps", type=int, default=300, help="timed steps")
    ap.add_argument("--warmup", type=int, default=3, help="untimed warm-up steps (at least 3)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours",
                    help="the CUDA library, or the CPU oracle on a bounded sample")
    ap.add_argument("--layers", type=int, default=4, help="layer caches visited in turn per step")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, help="index into synth.WORKLOADS")
    ap.add_argument("--graph", type=int, default=1, help="replay each step as one CUDA graph (1) or call directly (0)")
    ap.add_argument("--e2e-steps", type=int, default=5, help="steps timed end to end from pinned host buffers")
    ap.add_argument("--decode-calls", type=int, default=64, help="decode-attention calls timed one by one (>= 50)")
    ap.add_argument("--prefill-calls", type=int, default=12, help="prefill calls timed one by one")
    ap.add_argument("--cpu-seconds", type=float, default=8.0, help="oracle time of each CPU-baseline leg")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--no-self-check", action="store_true", help="skip the post-timing check against the oracle")
    ap.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi clocks")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (small profiling cases)")
    ap.add_argument("--tokens", type=int, default=0, help="override the workload's prompt length")
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
    if args.batch:
        w = w.scaled(batch=args.batch, name=w.name + f" (batch {args.batch})")
    if args.tokens:
        w = w.scaled(prefill_tokens=args.tokens, name=w.name + f" (prompt {args.tokens})")
    if args.sink:
        w = w.scaled(sink=args.sink)
    if args.codebook:
        w = dataclasses.replace(w, k_levels=tuple(codebook_levels(w.k_bits).tolist()),
                                v_levels=tuple(codebook_levels(w.v_bits).tolist()))
    return w


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


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


def prefill_bytes(w, T0):
    """Algorithmic bytes of one prefill call: the fp16 prompt read once, the packed pages and the fp16
    sink and window rows written (packed codes + scales and zero points + sparse entries)."""
    D, G = w.head_dim, w.group
    n_s = min(T0, w.sink)
    Tq = quantized_tokens(T0 - n_s, w.residual)
    n_r = T0 - n_s - Tq
    written = (Tq * D * (w.k_bits + w.v_bits) // 8 + (Tq // G) * D * 4 + Tq * (D // G) * 4 + Tq * w.k_sparse * 3
               + (n_r + n_s) * D * 4)
    return w.batch * w.kv_heads * (T0 * D * 4 + written)


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
        **({"k_sparse": w.k_sparse} if w.k_sparse else {}),
        **({"rope": f"keys stored pre-RoPE, rotated at decode (base {w.rope_base:g})"} if w.rope else {}),
        **({"sink_tokens": w.sink} if w.sink else {}),
        **({"codebook": "cosine-spaced levels (non-uniform)"} if w.k_levels else {}),
        "step": f"{layers} layers x (prefill {w.prefill_tokens}) + {w.decode_steps} x {layers} layers x "
                f"fused decode step (append, flushing a full window first, + decode attention)",
        "l2": f"inputs larger than L2: a {prefill_bytes(w, w.prefill_tokens) / 1e9:.2f} GB prefill per layer and "
              f"{layers} layer caches of {decode_bytes(w, w.prefill_tokens + 1) / 1e6:.0f} MB visited in turn",
        "launch": "one CUDA graph per step" if graph else "direct C-ABI calls",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
    }


def timing_stats(ms_list):
    """Median, p90 and mean (ms) of per-call times."""
    a = np.asarray(ms_list, np.float64)
    return {"median_us": float(np.median(a)) * 1e3, "p90_us": float(np.percentile(a, 90)) * 1e3,
            "mean_us": float(a.mean()) * 1e3, "calls": int(a.size)}


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
                                          "--format=csv,noheader,nounits", "-lms", "50"],
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
        sm, mx, power, reasons = [], [], [], set()
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
            try:
                power.append(float(parts[3]))
            except ValueError:
                pass
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not self.keep:
            os.remove(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "sm_mhz_min": min(sm), "sm_mhz_p10": float(np.percentile(sm, 10)),
                **({"power_w_median": statistics.median(power)} if power else {})}


# ------------------------------------------------------------------ CPU oracle baseline

def _oracle_units(w, units, Q, seconds):
    """The oracle as it stands over (sequence, kv head) units in turn -- prefill, then every decode step
    (append + fp64 attention of the unit's query heads) -- until `seconds` of oracle time.  A unit is
    1/Hkv of its sequence's work and is credited with sum_i T_i / Hkv tokens, in the GPU's unit.
    Input generation is not timed."""
    import oracle
    T0, steps = w.prefill_tokens, w.decode_steps
    busy = 0.0
    tokens = 0.0
    done = 0
    for unit in units:
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
        done += 1
        if busy >= seconds:
            break
    return {"tokens": tokens, "busy": busy, "units": done}


def _oracle_worker(job):
    """One process of the all-core leg: its own units, its own generator threads set to one."""
    wl, units, Q, seconds = job
    return _oracle_units(wl, units, Q, seconds)


class OraclePool:
    """One single-threaded oracle process per host core (spawned: no CUDA state is inherited)."""

    def __init__(self, cores=None):
        import multiprocessing as mp
        self.cores = cores or host_cores()
        ctx = mp.get_context("spawn")
        env_before = os.environ.get("KVQ_SYNTH_THREADS")
        os.environ["KVQ_SYNTH_THREADS"] = "1"  # the workers' input generation stays on their own core
        try:
            self.pool = ctx.Pool(self.cores)
        finally:
            if env_before is None:
                os.environ.pop("KVQ_SYNTH_THREADS", None)
            else:
                os.environ["KVQ_SYNTH_THREADS"] = env_before

    def run(self, w, Q, seconds, offset=0):
        """Every process runs the oracle over units offset+k, offset+k+C, ... for `seconds` of oracle time;
        the throughput is the units' tokens over the longest process's oracle time."""
        n_units = w.batch * w.kv_heads
        jobs = []
        for k in range(self.cores):
            units = [(offset + k + j * self.cores) % n_units for j in range(n_units)]
            jobs.append((w, units, Q, seconds))
        res = self.pool.map(_oracle_worker, jobs)
        tokens = sum(r["tokens"] for r in res)
        wall = max(r["busy"] for r in res)
        return {"value": tokens / wall, "tokens": tokens, "busy_max": wall, "units": sum(r["units"] for r in res)}

    def close(self):
        self.pool.close()
        self.pool.join()


def all_queries(w):
    return [synth.queries(w, i) for i in range(w.decode_steps)]


def cpu_baseline(w, seconds, pool=None):
    """The oracle timed on one thread and on every host core of this machine."""
    T0, steps = w.prefill_tokens, w.decode_steps
    Q = all_queries(w)
    one = _oracle_units(w, range(w.batch * w.kv_heads), Q, seconds)
    own = pool is None
    pool = pool or OraclePool()
    try:
        allc = pool.run(w, Q, seconds)
    finally:
        if own:
            pool.close()
    work = f"(sequence, kv head) units x (prefill {T0} + {steps} x (append + fp64 attention))"
    return {"value": allc["value"], "unit": UNIT, "cores": pool.cores, "kind": "oracle",
            "host_cores": host_cores(),
            "sample": f"{allc['units']} {work} on {pool.cores} single-threaded oracle processes (one per core), "
                      f"{allc['busy_max']:.1f} s of oracle time each",
            "single_thread": {"value": one["tokens"] / one["busy"], "unit": UNIT, "cores": 1,
                              "sample": f"{one['units']} {work}, {one['busy']:.1f} s"}}


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
    Q = np.stack(all_queries(w))  # [S][B][Hq][D]
    k_pre = torch.from_numpy(np.ascontiguousarray(K[:, :, :T0])).to(dev)
    v_pre = torch.from_numpy(np.ascontiguousarray(V[:, :, :T0])).to(dev)
    k_new = torch.from_numpy(np.ascontiguousarray(K[:, :, T0:T0 + S].transpose(2, 0, 1, 3))).to(dev)  # [S][B][Hkv][D]
    v_new = torch.from_numpy(np.ascontiguousarray(V[:, :, T0:T0 + S].transpose(2, 0, 1, 3))).to(dev)
    q_dev = torch.from_numpy(Q).to(dev)
    out = torch.empty((L, S, B, Hq, D), dtype=torch.float16, device=dev)
    out_dec = torch.empty((L, B, Hq, D), dtype=torch.float16, device=dev)
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

    def prefill(h):
        check(Lb.kvq_reset(h), "reset")
        check(Lb.kvq_prefill_quantize(h, kp, vp, T0, sh), "prefill")

    def step():
        for h in handles:
            prefill(h)
        for i in range(S):
            for l, h in enumerate(handles):
                check(Lb.kvq_decode_step(h, knp[i], vnp[i], qp[i], op[l][i], sh), "decode step")

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

    # ---------------- the timed path checked against the oracle: one sampled unit of the last step
    self_check = None
    if not args.no_self_check:
        self_check = check_against_oracle(w, caches[0], out[0, S - 1], K, V, Q[S - 1])

    # ---------------- per-call timing (CUDA events on the launching stream), rotating over the layers:
    # decode attention over each cache's state after the step, then the prefill
    def per_call(n, call):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        with torch.cuda.stream(stream):
            # the GPU spins first (about 60 us per call to come) so that the host has enqueued every
            # call before the first runs: the events then bracket device time, not the host's launches
            torch.cuda._sleep(int(120_000 * n))
            for j in range(n):
                evs[j][0].record(stream)
                call(j)
                evs[j][1].record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in evs]

    T_dec = T0 + S
    n_dec = max(args.decode_calls, 1)
    dec_ms = per_call(n_dec, lambda j: check(Lb.kvq_decode_attention(handles[j % L], qp[S - 1],
                                                                     out_dec[j % L].data_ptr(), sh), "decode"))
    pre_ms = per_call(max(args.prefill_calls, 1), lambda j: prefill(handles[j % L]))
    for h in handles:
        if Lb.kvq_sync_status(h, sh) != 0:
            raise RuntimeError("device-side error in the per-call timing")
    dec = timing_stats(dec_ms)
    pre = timing_stats(pre_ms)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = json.load(open(peaks_path)) if os.path.exists(peaks_path) else {}
    peak = peaks.get("hbm_gbs", 6800.0)
    peak_source = "MEASURED_PEAKS.json hbm_gbs (of measured)" if peaks else "fallback 6.8 TB/s"
    dec_b = decode_bytes(w, T_dec)
    pre_b = prefill_bytes(w, T0)
    dec_gbs = dec_b / (dec["median_us"] * 1e-6) / 1e9
    pre_gbs = pre_b / (pre["median_us"] * 1e-6) / 1e9
    kernels = {
        "decode_attention": {
            "bound": "hbm", "achieved": dec_gbs, "peak": peak, "unit": "GB/s", "frac": dec_gbs / peak,
            "traffic": kernel_traffic("decode", w), "bytes_per_call": dec_b, **dec, "tokens_attended": T_dec,
            "kernel": f"decode attention call: {decode_kernel_name(w)} + merge_kernel (programmatic dependent launch)"},
        "prefill": {
            "bound": "hbm", "achieved": pre_gbs, "peak": peak, "unit": "GB/s", "frac": pre_gbs / peak,
            "traffic": kernel_traffic("prefill", w), "bytes_per_call": pre_b, **pre,
            "kernel": f"prefill call: {prefill_kernel_name(w)} + copy_tokens_kernel (window tail)"},
    }
    # the dominant kernel: the larger share of the step
    share_pre = L * pre["median_us"]
    share_dec = L * S * dec["median_us"]
    dom = "prefill" if share_pre >= share_dec else "decode_attention"
    roof = dict(kernels[dom])
    roof["name"] = dom
    roof["peak_source"] = peak_source
    # its share of the step's device time, from the per-call medians (calls timed one by one carry
    # their own launch gaps, so the two shares are taken relative to each other, not to ms_per_step)
    roof["step_share"] = (share_pre if dom == "prefill" else share_dec) / (share_pre + share_dec)

    # ---------------- end to end through the C ABI from pinned host memory
    e2e = run_e2e(args, w, dist, caches, stream) if args.e2e_steps > 0 else None
    if e2e and e2e["link_peak_gbs"]:
        # the step cannot end before its inputs have crossed the link nor before its compute has run
        link_ms = e2e["h2d_bytes_per_step"] / (e2e["link_peak_gbs"] * 1e9) * 1e3
        e2e["floor_ms_per_step"] = max(link_ms, ms_step)
        e2e["floor_bound"] = "link" if link_ms > ms_step else "compute"
        e2e["frac_of_floor"] = e2e["floor_ms_per_step"] / e2e["ms_per_step"]

    tokens = step_tokens(w, L)
    total_tokens = dist.sum(tokens)
    value = total_tokens / (ms_step * 1e-3)
    for c in caches:
        c.close()
    return {
        "value": value, "ms_per_step": ms_step, "gpu_launches": int(n_launch),
        "roofline": roof,
        "decode_only": {"value": B * T_dec / (dec["median_us"] * 1e-6), "unit": UNIT,
                        "hbm_gbs": dec_gbs, "frac": dec_gbs / peak, **dec},
        "kernels": kernels,
        "clocks": clock_info, "e2e": e2e, "self_check": self_check,
        "config": workload_config(w, L, graph is not None, dist.world),
    }


def check_against_oracle(w, cache, out_last, K, V, q_last):
    """One sampled unit of the timed path against the oracle: stores bit for bit, attention within 2e-3."""
    import oracle
    T0, S = w.prefill_tokens, w.decode_steps
    rng = np.random.default_rng(1234)
    b = int(rng.integers(w.batch))
    kvh = int(rng.integers(w.kv_heads))
    u = oracle.OracleUnit.for_workload(w)
    u.prefill(K[b, kvh, :T0], V[b, kvh, :T0])
    for i in range(S):
        u.append(K[b, kvh, T0 + i], V[b, kvh, T0 + i])
    got = cache.export_unit(b, kvh)
    ref = u.stores()
    stores_equal = all(np.array_equal(got[k], ref[k]) for k in ref)
    hs = slice(kvh * w.group_q, (kvh + 1) * w.group_q)
    o_ref = u.attention(q_last[b, hs], w.softmax_scale)
    o = out_last.float().cpu().numpy()[b, hs].astype(np.float64)
    err = oracle.max_rel_err(o, o_ref)
    ok = bool(stores_equal and err <= 2e-3)
    if not ok:
        raise RuntimeError(f"self-check failed on unit (b={b}, kvh={kvh}): stores equal {stores_equal}, "
                           f"attention error {err:.3e}")
    return {"unit": [b, kvh], "stores_bit_exact": stores_equal, "attention_max_rel_err": err, "ok": ok}


# sources of each kernel family: a change to any of them invalidates that family's DRAM counters
KERNEL_SOURCES = {
    "decode_mma": ("kvq_decode_mma.cu", "kvq_decode.cu", "kvq_merge.cuh", "kvq_ptx.cuh", "kvq_internal.h"),
    "decode_cuda_core": ("kvq_decode_kernel.cuh", "kvq_decode.cu", "kvq_merge.cuh", "kvq_ptx.cuh", "kvq_internal.h"),
    "prefill": ("kvq_quant.cu", "kvq_quantizer.cuh", "kvq_ptx.cuh", "kvq_internal.h"),
}


def decode_kernel_name(w):
    return "decode_mma_kernel" if kernel_family("decode", w) == "decode_mma" else "decode_kernel"


def prefill_kernel_name(w):
    """The page kernel the library picks for this layout (fragment order: 2/4-bit codes, keys after RoPE)."""
    frag = not w.rope and w.k_bits in (2, 4) and w.v_bits in (2, 4)
    if frag and w.residual == 128 and w.head_dim == 128 and w.group == 32 and not w.k_sparse and not w.k_levels:
        return "quantize_std_kernel"
    if not frag and not w.k_levels and w.residual == 128 and w.head_dim == 128 and w.group in (32, 64) and w.k_sparse <= 4:
        return "quantize_bits_kernel"
    return "quantize_pages_kernel"


def kernel_family(kind, w):
    """The kernel that serves a call of this workload (the launch-time choice of the library)."""
    if kind == "prefill":
        return "prefill"
    mma = not w.rope and not w.k_levels and w.k_bits in (2, 4) and w.v_bits in (2, 4)
    return "decode_mma" if mma else "decode_cuda_core"


TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def kernel_revision(family):
    """Hash of a kernel family's sources: DRAM counters are valid only for the kernel they were taken on."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_asymmetric_kv_kvq_gb300", "csrc")
    for f in KERNEL_SOURCES[family]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def kernel_traffic(kind, w):
    """DRAM read+write bytes per call from the committed ncu summary, or None.

    The summary holds blocks of `key: value` lines separated by blank lines; a block counts only when
    it was taken on this kernel kind, this workload and the current sources of that kernel."""
    if not os.path.exists(TRAFFIC_SUMMARY):
        return None
    blocks, cur = [], {}
    for line in open(TRAFFIC_SUMMARY):
        if not line.strip():
            if cur:
                blocks.append(cur)
            cur = {}
            continue
        if ":" in line and not line.startswith((" ", "#")):
            k, v = line.split(":", 1)
            cur[k.strip()] = v.strip()
    if cur:
        blocks.append(cur)
    rev = kernel_revision(kernel_family(kind, w))
    for kv in blocks:
        if kv.get("kind") == kind and kv.get("workload") == w.name and kv.get("kernel_rev") == rev:
            try:
                return float(kv["dram_bytes_per_call"])
            except (KeyError, ValueError):
                return None
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
    hq = pin(np.stack(all_queries(w)))
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

    # the link's own rate: one plain pinned host->device copy of a prompt buffer, best of three
    link_peak = 0.0
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        with torch.cuda.stream(stream):
            dk[0].copy_(hk, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize(dev)
        link_peak = max(link_peak, hk.nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
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
    link = (h2d // args.e2e_steps) / (ms * 1e-3) / 1e9
    return {"value": total / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d // args.e2e_steps, "d2h_bytes_per_step": d2h // args.e2e_steps,
            "h2d_gbs": link, "link_peak_gbs": link_peak, "link_frac": link / link_peak if link_peak else None}


# ------------------------------------------------------------------ reference arm: the CPU oracle

def run_reference(args, dist):
    w = workload_of(args)
    L = args.layers
    Q = all_queries(w)
    # each step: every host core runs the oracle over its own units for a bounded time
    per = max(0.2, args.cpu_seconds / max(1, args.steps + args.warmup))
    pool = OraclePool()
    try:
        for i in range(args.warmup):
            pool.run(w, Q, per, offset=i)
        t0 = time.perf_counter()
        vals = [pool.run(w, Q, per, offset=args.warmup + i) for i in range(args.steps)]
        el = time.perf_counter() - t0
    finally:
        pool.close()
    value = statistics.mean(v["value"] for v in vals)
    units = sum(v["units"] for v in vals)
    return {
        "impl": "reference", "value": value, "ms_per_step": el / args.steps * 1e3,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.cores, "kind": "oracle",
                         "host_cores": host_cores(),
                         "sample": f"{units} (sequence, kv head) units over {args.steps} steps, each step "
                                   f"~{per:.1f} s of oracle time on {pool.cores} single-threaded oracle processes"},
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
    # the oracle processes start before the first GPU call (spawned, so nothing of CUDA is inherited)
    pool = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        pool = OraclePool()
    try:
        res = run_ours(args, dist)
        w = workload_of(args)
        line = {"metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": f"u{w.k_bits}/u{w.v_bits} codes, f16 tensor-core mma (f32 accumulate), f16 out",
                "data": "synthetic (seeded): keys N(0,1) with outlier channels, values N(0,1), queries N(0,1)",
                "config": res["config"], "e2e": res["e2e"], "roofline": res["roofline"],
                "decode_only": res["decode_only"], "kernels": res["kernels"], "self_check": res["self_check"],
                "gpu_launches": res["gpu_launches"], "clocks": res["clocks"]}
        if pool is not None:
            line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, pool)
    finally:
        if pool is not None:
            pool.close()
    if dist.rank == 0:
        print(json.dumps(line))
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
