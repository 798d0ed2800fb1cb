"""Benchmark: one GQA decode step (paged KV append + split-KV decode + combine).

Default workload: the Llama-2/3-70B-shaped paged decode (bf16, H=64, K=8,
d=128, batch 32, context lengths seeded uniform in [128, 32768], block_size 16,
shuffled block table), the largest single-GPU configuration.
Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--kernel auto|mma|fma]

N > 1 runs under torchrun as independent replicas (the step has no exchange):
every rank decodes its own copy of the workload; value = bytes of all ranks /
the slowest rank's time.

Metric: achieved decode-attention bandwidth = algorithmic bytes of the step
(K/V (+int8 scales) of every cached token read once, Q read, O written, block
table and lengths read, the appended token's K/V written) / step time; also
tokens/s = batch / step time for one attention layer.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attention HBM GB/s (% of GB300 peak) and tokens/s per decode step, 1 GPU"
DEFAULT_WORKLOAD = "llama70b_bf16_b32_ragged"
L2_BYTES = 129 * 2 ** 20
KERNEL_NAME = "split_kv_kernel"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "split_kv_kernel_traffic.txt")
PREFILL_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "prefill_tc2_kernel_traffic.txt")
# gqa_prefill's kernel choice (include/gqa_decode.h GQA_PREFILL_*) and the kernel it runs
PREFILL_KERNEL = {"auto": 0, "tc1": 1, "mma_sync": 2, "tc2": 3, "tc2_paired": 4}


def attended_range(wl, L: int) -> tuple:
    """First position any query of a length-L sequence attends, and L: with T
    new tokens and a window W the union of the queries' ranges is
    [max(0, L - T + 1 - W), L)."""
    lo = max(0, L - wl.queries + 1 - wl.window) if wl.window > 0 else 0
    return lo, L


def algorithmic_bytes(wl, lens) -> dict:
    """Bytes a decode step must move: KV (+scales) of every attended cached
    token once, q in, out (fp32) out, block-table entries and lengths, plus the
    append of the T new tokens."""
    es = {"f32": 4, "f16": 2, "bf16": 2, "i8": 1, "fp8": 1, "i4": 0.5, "i4kc": 0.5}[wl.cache_dtype]
    qes = {"f32": 4, "f16": 2, "bf16": 2}[wl.q_dtype]
    coded = wl.cache_dtype in ("i8", "fp8", "i4", "i4kc")
    kc = wl.cache_dtype == "i4kc"                  # K scales per (block, kv-head, channel)
    K, d, T = wl.num_kv_heads, wl.head_dim, wl.queries
    ranges = [attended_range(wl, int(x)) for x in lens]
    tokens = int(sum(hi - lo for lo, hi in ranges))
    per_token = int(2 * K * d * es)
    if coded:
        per_token += (1 if kc else 2) * K * 2     # fp16 scales per (token, kv-head)
    blocks = int(sum(-(-hi // 16) - lo // 16 for lo, hi in ranges))
    B = len(lens)
    kv = tokens * per_token + (blocks * K * 2 * d if kc else 0)
    q = B * T * wl.num_heads * d * qes
    o = B * T * wl.num_heads * d * 4
    meta = blocks * 4 + B * 4
    new_es = qes if coded else es
    append = int(B * T * 2 * K * d * (new_es + es)) + B * 4
    if kc:
        # K: every block the new tokens reach is rewritten whole (codes of its
        # present slots, d scales), its older slots read from the fp32
        # residual, and new rows of an unfinished block written back to it;
        # V: per-token scales
        append = int(B * T * K * (2 * d * new_es + d * es + 2)) + B * 4
        for L in lens:
            p0 = max(0, int(L) - T)
            for jb in range(p0 // 16, (p0 + T - 1) // 16 + 1):
                first = 16 * jb
                tend = min(16, p0 + T - first)
                old = max(0, p0 - first)
                append += K * (old * d * 4 + int(tend * d * es) + 2 * d)
                if tend < 16:
                    append += K * (tend - old) * d * 4
    decode = kv + q + o + meta
    return {"kv": kv, "decode": decode, "append": append, "step": decode + append,
            "tokens": tokens, "blocks": blocks}


# The sources the split-KV kernel is compiled from: a traffic figure taken on
# other sources no longer describes it.
SPLIT_KV_SOURCES = ("gqa_decode_kernels.cuh", "gqa_device.cuh", "gqa_internal.h", "gqa_decode.cu",
                    "gqa_decode_general.cu")
PREFILL_SOURCES = ("gqa_prefill.cu", "gqa_device.cuh", "gqa_internal.h")


def kernel_source_hash(files=SPLIT_KV_SOURCES) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gqa_decode_attention_kv_gb300", "csrc")
    for name in sorted(files):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic(workload: str, kernel: str, path: str = TRAFFIC_FILE, sources=SPLIT_KV_SOURCES):
    """DRAM bytes per launch from a committed ncu summary (blocks of
    'key: value' lines separated by blank lines, one per workload), if one was
    taken on the current source of that kernel for this workload; else None."""
    try:
        text = open(path).read()
    except OSError:
        return None
    src = kernel_source_hash(sources)
    for block in text.split("\n\n"):
        vals = {}
        for ln in block.splitlines():
            if ":" in ln and not ln.startswith("#"):
                k, _, v = ln.partition(":")
                vals[k.strip()] = v.strip()
        if vals.get("source_hash") != src or vals.get("workload") != workload:
            continue
        if vals.get("kernel_variant", "auto") != kernel:
            continue
        try:
            return float(vals["traffic_bytes_per_launch"])
        except (KeyError, ValueError):
            return None
    return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling; keeps the samples taken inside the
    timed window (host wall clock, the GPU being busy for all of it)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self, t_begin: float, t_end: float):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        import datetime
        rows = []
        for ln in open(self.path).read().splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            rows.append((ts, parts))
        os.unlink(self.path)
        inside = [p for ts, p in rows if t_begin <= ts <= t_end]
        window = "timed region"
        if not inside and rows:             # timed region shorter than the sampling period
            mid = 0.5 * (t_begin + t_end)
            inside = [min(rows, key=lambda r: abs(r[0] - mid))[1]]
            window = "nearest sample (timed region shorter than sampling period)"
        if not inside:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[2]) for r in inside) if v is not None]
        mx = [v for v in (num(r[3]) for r in inside) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside), "window": window}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def resolve_workload(name: str, batch: int = 0):
    """A named workload, or the 70B-shaped KV-head sweep point '<70B name>_k<K>';
    batch > 0 keeps only the first `batch` sequences (a smaller case of the same
    workload, for profiling; named '<name>_first<batch>')."""
    import dataclasses
    import gqa_inputs as gi
    if name in gi.WORKLOADS:
        wl = gi.WORKLOADS[name]
    else:
        base, _, k = name.rpartition("_k")
        if base == "llama70b_bf16_b32_ragged" and k.isdigit():
            wl = gi.kv_sweep_workload(int(k))
        else:
            raise SystemExit(f"unknown workload {name!r}")
    if 0 < batch < wl.batch:
        wl = dataclasses.replace(wl, name=f"{wl.name}_first{batch}", batch=batch)
    return wl


ROW_LAYOUT = {"auto": 0, "split": 1, "shared": 2}


def kernel_code(name: str) -> int:
    return {"auto": 0, "mma": 1, "fma": 2}[name]


def max_over_ranks(vals, device):
    """Element-wise max of per-rank timings (the slowest replica decides)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(vals), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_gbs(bytes_per_rank: float, world: int, ms: float) -> float:
    """Aggregate bandwidth of N replicas that each moved bytes_per_rank in ms."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


# ----------------------------------------------------------------------------- read ceiling

READ_PROBE_FORMS = ((0, 2, "bulk copies, 8 KB chunks, 2 stages per warp, 2 CTAs/SM"),
                    (0, 3, "bulk copies, 8 KB chunks, 2 stages per warp, 3 CTAs/SM"),
                    (1, 2, "bulk copies, 8 KB chunks, 3 stages per warp, 2 CTAs/SM"),
                    (2, 3, "bulk copies, 4 KB chunks, 4 stages per warp, 3 CTAs/SM"),
                    (3, 4, "16-byte loads, 4 x 256 threads per SM"),
                    (3, 8, "16-byte loads, 8 x 256 threads per SM"))


def read_probe(dev, gib: float = 4.0, reps: int = 10) -> dict:
    """Measured HBM read ceiling: the probe library's pure read streams over a
    buffer larger than L2 (each form warmed up, then `reps` launches timed with
    CUDA events on the launching stream); the best form is reported."""
    import ctypes
    import torch
    from gqa_decode_attention_kv_gb300 import build as gbuild
    lib = ctypes.CDLL(gbuild.PROBE_LIB_PATH)
    lib.hbm_read_probe.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_void_p]
    lib.hbm_read_probe.restype = ctypes.c_int
    nbytes = int(gib * 2 ** 30) // 8192 * 8192
    buf = torch.full((nbytes // 4,), 0x01020304, dtype=torch.int32, device=dev)
    sink = torch.zeros(1, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream()
    results = {}
    for form, cps, how in READ_PROBE_FORMS:
        def launch():
            rc = lib.hbm_read_probe(buf.data_ptr(), nbytes, sink.data_ptr(), form, cps, stream.cuda_stream)
            if rc != 0:
                raise RuntimeError(f"hbm_read_probe failed with {rc}")
        for _ in range(3):
            launch()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            launch()
        e1.record(stream)
        torch.cuda.synchronize()
        results[how] = round(nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
    if int(sink.item()) >= 1 << 40:
        raise RuntimeError("hbm_read_probe: a bounded wait expired")
    best = max(results, key=results.get)
    del buf
    return {"gbs": results[best], "form": best, "bytes_per_launch": nbytes, "forms": results,
            "how": f"pure read of a {nbytes / 2 ** 30:.0f} GiB buffer (> L2), {reps} launches per form "
                   "after 3 warm-ups, CUDA events; best form"}


# ----------------------------------------------------------------------------- our arm

def prefill_flops(wl, lens) -> float:
    """Algorithmic flops of causal prefill: query i of a length-L sequence with T
    new tokens attends min(L - T + i + 1, W) positions; 4*d flops per head and
    attended position (q.k and p.v, multiply-add each)."""
    T = wl.queries
    total = 0
    for L in lens:
        L = int(L)
        for i in range(T):
            n = L - T + i + 1
            if n <= 0:
                continue
            total += min(n, wl.window) if wl.window > 0 else n
    return 4.0 * wl.head_dim * wl.num_heads * total


def pipelined_e2e(stream, host_inputs, out_like, run, steps, warmup, nbuf=2):
    """End-to-end timing through the public API: every step copies its inputs
    from pinned host memory, runs, and reads its output back into pinned host
    memory. As a serving loop would, the copies go on two copy streams under
    the neighbouring steps' kernels, inputs and outputs double-buffered.
    Returns (ms per step, the last step's host output, H2D bytes, D2H bytes)."""
    import torch
    dev = out_like.device
    dev_in = [[torch.empty_like(h, device=dev) for h in host_inputs] for _ in range(nbuf)]
    out_d = [torch.empty_like(out_like) for _ in range(nbuf)]
    out_h = [torch.empty(out_like.shape, dtype=out_like.dtype).pin_memory() for _ in range(nbuf)]
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]      # inputs of buffer b landed
    ev_run = [torch.cuda.Event() for _ in range(nbuf)]     # kernels reading buffer b done
    ev_back = [torch.cuda.Event() for _ in range(nbuf)]    # output of buffer b read back
    for e in ev_in + ev_run + ev_back:
        e.record(stream)

    def one(i):
        b = i % nbuf
        h2d_s.wait_event(ev_run[b])                # the step two back is done with buffer b
        with torch.cuda.stream(h2d_s):
            for dst, src in zip(dev_in[b], host_inputs):
                dst.copy_(src, non_blocking=True)
        ev_in[b].record(h2d_s)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_back[b])
        run(*dev_in[b], out_d[b])
        ev_run[b].record(stream)
        d2h_s.wait_event(ev_run[b])
        with torch.cuda.stream(d2h_s):
            out_h[b].copy_(out_d[b], non_blocking=True)
        ev_back[b].record(d2h_s)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_s.wait_event(e0)
    for i in range(steps):
        one(i)
    for e in ev_back:
        stream.wait_event(e)                       # every read-back inside the timed region
    e1.record(stream)
    torch.cuda.synchronize()
    h2d = sum(t.numel() * t.element_size() for t in host_inputs)
    d2h = out_h[0].numel() * out_h[0].element_size()
    return e0.elapsed_time(e1) / steps, out_h[(steps - 1) % nbuf], h2d, d2h


def run_prefill(args, wl):
    """One prefill step: the varlen append of every prompt's K/V, then causal
    attention of all prompt tokens over the paged cache."""
    import torch
    import torch.distributed as dist

    import gqa_inputs as gi
    import gqa_decode_attention_kv_gb300 as gq
    from gqa_decode_attention_kv_gb300 import build as gbuild

    world, rank, local = dist_info()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gbuild.build()
    gq.load()
    case = gi.case_for(wl, seed=args.seed + rank, device=str(dev), extra_tokens=0)
    cache = gq.cache_from_case(case)
    B, T, H, K, d = wl.batch, wl.queries, wl.num_heads, wl.num_kv_heads, wl.head_dim
    q = case.q.reshape(B * T, H, d)
    kn = case.k_new.reshape(B * T, K, d)
    vn = case.v_new.reshape(B * T, K, d)
    starts = torch.arange(0, B * T + 1, T, dtype=torch.int32, device=dev)
    lens = case.context_lens
    pos = (lens - T).clamp(min=0)
    out = torch.empty((B * T, H, d), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flops = prefill_flops(wl, lens.cpu().tolist())
    stream = torch.cuda.current_stream()

    pk = PREFILL_KERNEL[args.prefill_kernel]
    kname = {0: "prefill_tc2_kernel" if d == 128 else "prefill_tc_kernel", 1: "prefill_tc_kernel",
             2: "prefill_kernel", 3: "prefill_tc2_kernel" if d == 128 else "prefill_tc_kernel",
             4: "prefill_tc2_kernel" if d == 128 else "prefill_tc_kernel"}[pk]

    def step(qq=q, kk=kn, vv=vn):
        gq.kv_append_varlen(cache, kk, vv, starts, T, case.block_table, pos, err=err)
        gq.gqa_prefill(cache, qq, starts, T, case.block_table, lens, case.scale, out=out,
                       window=wl.window, err=err, kernel=pk)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if err.item() != 0:
        raise RuntimeError(f"device error flags {err.item()}")
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.5)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    w0 = time.time()
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    clk = clocks.stop(w0, w1)
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    # the attention kernel alone (events around each launch, own loop)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        gq.kv_append_varlen(cache, kn, vn, starts, T, case.block_table, pos, err=err)
        kev[i][0].record(stream)
        gq.gqa_prefill(cache, q, starts, T, case.block_table, lens, case.scale, out=out,
                       window=wl.window, err=err, kernel=pk)
        kev[i][1].record(stream)
    torch.cuda.synchronize()
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    # end to end with host buffers (copies overlapped with neighbouring steps)
    host_in = [t.detach().cpu().pin_memory() for t in (q, kn, vn)]
    e2e_ms, last_out, h2d, d2h = pipelined_e2e(
        stream, host_in, out, lambda qd, knd, vnd, od: (
            gq.kv_append_varlen(cache, knd, vnd, starts, T, case.block_table, pos, err=err),
            gq.gqa_prefill(cache, qd, starts, T, case.block_table, lens, case.scale, out=od,
                           window=wl.window, err=err, kernel=pk)),
        args.steps, max(3, args.warmup))
    if err.item() != 0:
        raise RuntimeError(f"device error flags {err.item()}")
    if not torch.equal(last_out, out.cpu()):
        raise RuntimeError("end-to-end output differs from the device-timed step's")
    ms, e2e_ms, kern_ms = max_over_ranks([ms, e2e_ms, kern_ms], dev)
    if rank == 0:
        peaks, peak_kind = measured_peaks()
        peak = float(peaks["bf16_tflops"])
        tf = flops * world / (ms * 1e-3) / 1e12
        kern_tf = flops / (kern_ms * 1e-3) / 1e12
        line = {
            "metric": "prefill attention TFLOP/s (causal, algorithmic flops), 1 GPU",
            "value": round(tf, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.cache_dtype, "data": "synthetic",
            "config": {"workload": wl.name, "batch": B, "prompt_tokens": T, "num_heads": H,
                       "prefill_kernel": args.prefill_kernel,
                       "num_kv_heads": K, "head_dim": d, "context_lens": wl.lens,
                       "sliding_window": wl.window, "cache_dtype": wl.cache_dtype,
                       "block_size": 16, "block_table": "seeded shuffle",
                       "l2": "K/V re-read by every query tile of a sequence (mostly from L2)",
                       "step": "kv_append_varlen + gqa_prefill, one attention layer"},
            "tokens_per_s": round(B * T * world / (ms * 1e-3), 1),
            "roofline": {"bound": "tensor", "achieved": round(kern_tf, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(kern_tf / peak, 4),
                         "traffic": read_traffic(wl.name, args.prefill_kernel, PREFILL_TRAFFIC_FILE,
                                                 PREFILL_SOURCES),
                         "kernel": kname, "algorithmic_flops_per_launch": flops,
                         "avg_launch_ms": round(kern_ms, 5),
                         "kernel_timing": "CUDA events around every prefill launch, own timed loop",
                         "peak_source": f"{peak_kind} bf16_tflops (burst, cuBLAS; MEASURED_PEAKS.json)"},
            "e2e": {"value": round(flops * world / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5),
                    "how": "kv_append_varlen + gqa_prefill per step with its pinned-host inputs copied in "
                           "and output read back; copies on two streams overlap neighbouring steps"},
            "gpu_launches": 2 * args.steps,
            "clocks": clk,
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = prefill_cpu_baseline(wl, case, flops, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def prefill_cpu_baseline(wl, case, flops_all, seconds: float) -> dict:
    """The oracle on the last queries of sequence 0 (as many as fit in about
    `seconds`), scaled to TFLOP/s by their own algorithmic flops."""
    import numpy as np
    import oracle
    oracle.build()
    threads = oracle.num_cpus()
    q, kd, vd, sl = _oracle_inputs(wl, case, [0])
    T = wl.queries
    n = 1
    while True:
        sub = q[:, T - n:]
        t = time.perf_counter()
        oracle.decode(sub, kd, vd, sl, case.scale, nthreads=threads, window=wl.window)
        dt = time.perf_counter() - t
        if dt * 2 > seconds or n == T:
            break
        n = min(T, n * 2)
    L = int(sl[0])
    att = sum(min(L - T + i + 1, wl.window) if wl.window > 0 else L - T + i + 1 for i in range(T - n, T))
    f = 4.0 * wl.head_dim * wl.num_heads * att
    return {"value": round(f / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "seconds": round(dt, 3),
            "sample": f"last {n} of {T} prompt tokens of sequence 0 (all {wl.num_heads} heads), fp64 C oracle"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import gqa_inputs as gi
    import gqa_decode_attention_kv_gb300 as gq
    from gqa_decode_attention_kv_gb300 import build as gbuild

    if resolve_workload(args.workload).kind == "prefill":
        return run_prefill(args, resolve_workload(args.workload, args.batch))
    world, rank, local = dist_info()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gbuild.build()
    gq.load()

    wl = resolve_workload(args.workload, args.batch)
    case = gi.case_for(wl, seed=args.seed + rank, device=str(dev), extra_tokens=0)
    cache = gq.cache_from_case(case)
    lens = case.context_lens
    if case.k_src is not None:
        # code cache drawn as N(0, 1) rows: the library's append quantises them in
        gq.kv_append_varlen(cache, case.k_src, case.v_src, case.src_start, int(lens.max().item()),
                            case.block_table, torch.zeros_like(lens))
        torch.cuda.synchronize()
    pos = (lens - wl.queries).clamp(min=0)    # the step re-appends the last T tokens
    ab = algorithmic_bytes(wl, lens.cpu().tolist())
    out = torch.empty(case.q.shape, dtype=torch.float32, device=dev)
    ws = gq.workspace_for(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim, dev, wl.queries)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kern = kernel_code(args.kernel)
    layout = ROW_LAYOUT[args.row_layout]
    stream = torch.cuda.current_stream()
    launches_per_step = 3

    def step(events=None):
        gq.kv_append(cache, case.k_new, case.v_new, case.block_table, pos, err=err)
        gq.gqa_decode(cache, case.q, case.block_table, lens, case.scale, out=out, workspace=ws,
                      kernel=kern, events=events, err=err, window=wl.window, row_layout=layout)

    # warm-up
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if err.item() != 0:
        raise RuntimeError(f"device error flags {err.item()}")

    # The K timed steps as one CUDA graph (the way a serving loop replays its
    # decode step): the kernels keep their programmatic-launch edges and the
    # host's enqueue cost stays out of the measurement at any K.
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(args.steps):
                step()
    stream.wait_stream(cap)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.5)                            # sampler start-up
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for _ in range(max(3, args.warmup)):       # busy right up to the timed region (clocks up)
        step()
    w0 = time.time()
    t0.record(stream)
    graph.replay()                             # exactly K steps
    t1.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    clk = clocks.stop(w0, w1)
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    if err.item() != 0:
        raise RuntimeError(f"device error flags {err.item()}")
    del graph

    # the split-KV kernel alone: events recorded by the library around each launch
    # (a separate timed loop, since an event between kernels ends the overlap)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in kev:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    for i in range(args.steps):
        step(events=kev[i])
    torch.cuda.synchronize()
    kern_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)

    # end to end through the public API with host buffers (copies overlapped with
    # neighbouring steps)
    host_in = [t.detach().cpu().pin_memory() for t in (case.q, case.k_new, case.v_new)]
    e2e_ms, last_out, h2d, d2h = pipelined_e2e(
        stream, host_in, out, lambda qd, knd, vnd, od: (
            gq.kv_append(cache, knd, vnd, case.block_table, pos, err=err),
            gq.gqa_decode(cache, qd, case.block_table, lens, case.scale, out=od, workspace=ws,
                          kernel=kern, err=err, window=wl.window, row_layout=layout)),
        args.steps, max(3, args.warmup))
    if not torch.equal(last_out, out.cpu()):
        raise RuntimeError("end-to-end output differs from the device-timed step's")
    if err.item() != 0:
        raise RuntimeError(f"device error flags {err.item()}")

    probe = read_probe(dev) if not args.no_read_probe else None

    # slowest rank decides
    ms, e2e_ms, kern_ms = max_over_ranks([ms, e2e_ms, kern_ms], dev)

    if rank == 0:
        peaks, peak_kind = measured_peaks()
        hbm = float(peaks["hbm_gbs"])
        gbs = whole_job_gbs(ab["step"], world, ms)
        kern_gbs = ab["decode"] / (kern_ms * 1e-3) / 1e9
        traffic = read_traffic(wl.name, args.kernel)
        line = {
            "metric": METRIC,
            "value": round(gbs, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": max(3, args.warmup),
            "ms_per_step": round(ms, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": wl.cache_dtype,
            "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.batch, "num_heads": wl.num_heads,
                       "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                       "context_lens": wl.lens, "cache_dtype": wl.cache_dtype,
                       "q_dtype": wl.q_dtype, "block_size": 16, "block_table": "seeded shuffle",
                       "tokens_per_seq": wl.queries, "sliding_window": wl.window,
                       "kernel": args.kernel, "row_layout": args.row_layout,
                       "l2": f"inputs larger than L2: {ab['kv'] / 1e9:.2f} GB of K/V per step > 129 MB",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "step": "kv_append + gqa_decode (split-KV + combine), one attention layer",
                       "timed_as": "the K steps captured in one CUDA graph, replayed once"},
            "tokens_per_s": round(wl.batch * wl.queries * world / (ms * 1e-3), 1),
            "pct_of_peak": {"measured_hbm": round(100 * gbs / world / hbm, 2),
                            "nominal_8tbs": round(100 * gbs / world / 8000.0, 2)},
            "roofline": {"bound": "hbm", "achieved": round(kern_gbs, 2), "peak": hbm,
                         "unit": "GB/s", "frac": round(kern_gbs / hbm, 4),
                         "traffic": traffic, "kernel": KERNEL_NAME,
                         "algorithmic_bytes_per_launch": ab["decode"],
                         "avg_launch_ms": round(kern_ms, 5),
                         "kernel_timing": "CUDA events around every split-KV launch, own timed loop",
                         "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)"},
            "e2e": {"value": round(whole_job_gbs(ab["step"], world, e2e_ms), 2), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms, 5),
                    "how": "kv_append + gqa_decode per step with its pinned-host inputs copied in and "
                           "output read back; copies on two streams overlap neighbouring steps"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
        }
        if probe is not None:
            line["read_probe"] = probe
            line["roofline"]["frac_of_read_probe"] = round(kern_gbs / probe["gbs"], 4)
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl, case, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- oracle arm

def _oracle_inputs(wl, case, rows):
    import numpy as np
    import oracle
    lens = case.context_lens.cpu().numpy()
    if case.k_src is not None:
        # code cache drawn as N(0, 1) rows: the oracle quantises the sampled
        # rows with its own rule (it never reads the device cache)
        S = max(int(lens[b]) for b in rows)
        K, d = wl.num_kv_heads, wl.head_dim
        kd = np.zeros((len(rows), S, K, d))
        vd = np.zeros((len(rows), S, K, d))
        st = case.src_start.cpu().numpy()
        for n, b in enumerate(rows):
            ks = case.k_src[int(st[b]):int(st[b + 1])].cpu().numpy()
            vs = case.v_src[int(st[b]):int(st[b + 1])].cpu().numpy()
            kd[n, :len(ks)] = oracle.quantised_sequence(ks, wl.cache_dtype, wl.cache_dtype == "i4kc")[0]
            vd[n, :len(vs)] = oracle.quantised_sequence(vs, wl.cache_dtype)[0]
        q = case.q.float().cpu().numpy().astype(np.float64)[rows]
        return q, kd, vd, lens[rows]
    table = case.block_table.cpu().numpy()
    sel = []
    for b in rows:
        nb = -(-int(lens[b]) // 16)
        sel.append(table[b, :nb])
    # copy only the blocks the sampled sequences use. Any cache layout is one
    # row of stride_block elements per physical block (the paged pool and the
    # un-paged [B, S_pad, K, d] buffer alike); the ids are checked here, on the
    # host, before they index device memory.
    import torch
    ids_np = np.concatenate(sel).astype(np.int64)
    if ids_np.size and (ids_np.min() < 0 or ids_np.max() >= case.num_blocks):
        raise ValueError("block table entry outside the cache")
    ids = torch.from_numpy(ids_np).to(case.k_cache.device)
    def host(t):
        t = t.reshape(case.num_blocks, -1).index_select(0, ids)
        if t.dtype in (torch.int8, torch.uint8):
            return t.cpu().numpy()
        if t.dtype == torch.float8_e4m3fn:
            return t.cpu().view(torch.uint8).numpy()
        return t.float().cpu().numpy()
    kp, vp = host(case.k_cache), host(case.v_cache)
    new_table = np.zeros((len(rows), table.shape[1]), dtype=np.int64)
    off = 0
    for i, s in enumerate(sel):
        new_table[i, :len(s)] = np.arange(off, off + len(s))
        off += len(s)
    sub_lens = lens[rows]
    K, d = wl.num_kv_heads, wl.head_dim
    packed4 = wl.cache_dtype in ("i4", "i4kc")
    rd = d // 2 if packed4 else d                        # stored row (4-bit: bytes)
    div = 2 if packed4 else 1                            # strides count 4-bit elements
    sb, sh, st = kp.shape[1], case.stride_head // div, case.stride_token // div
    kd = oracle.gather_dense(kp, new_table, sub_lens, sb, sh, st, K, rd)
    vd = oracle.gather_dense(vp, new_table, sub_lens, sb, sh, st, K, rd)
    if not packed4:
        kd, vd = kd.astype(np.float64), vd.astype(np.float64)
    if wl.cache_dtype in ("i8", "fp8", "i4", "i4kc"):
        ksp = case.k_scale.index_select(0, ids).float().cpu().numpy()
        vsp = case.v_scale.index_select(0, ids).float().cpu().numpy()
        vss = oracle.gather_scales(vsp, new_table, sub_lens, K)
        if wl.cache_dtype == "i4kc":                     # K scales per (block, kv-head, channel)
            kcs = oracle.gather_channel_scales(ksp.astype(np.float64), new_table, sub_lens)
            kd = oracle.unpack_int4(kd).astype(np.float64) * kcs
            vd = oracle.dequantize_int4(vd, vss)
        elif wl.cache_dtype == "i8":
            kss = oracle.gather_scales(ksp, new_table, sub_lens, K)
            kd = oracle.dequantize_int8(kd, kss)
            vd = oracle.dequantize_int8(vd, vss)
        elif wl.cache_dtype == "i4":
            kss = oracle.gather_scales(ksp, new_table, sub_lens, K)
            kd = oracle.dequantize_int4(kd, kss)
            vd = oracle.dequantize_int4(vd, vss)
        else:
            kss = oracle.gather_scales(ksp, new_table, sub_lens, K)
            kd = oracle.dequantize_fp8(kd.astype(np.uint8), kss)
            vd = oracle.dequantize_fp8(vd.astype(np.uint8), vss)
    q = case.q.float().cpu().numpy().astype(np.float64)[rows]
    return q, kd, vd, sub_lens


def _oracle_decode(wl, q, kd, vd, sl, scale, threads):
    import oracle
    return oracle.decode(q, kd, vd, sl, scale, nthreads=threads, window=wl.window)


def cpu_baseline(wl, case, seconds: float) -> dict:
    """Time the oracle, as it stands, on a bounded sample of the workload: as
    many sequences as fit in about `seconds` of host time, repeating the whole
    batch if one pass is shorter than that."""
    import oracle
    oracle.build()
    threads = oracle.num_cpus()
    q, kd, vd, sl = _oracle_inputs(wl, case, [0])
    t = time.perf_counter()
    _oracle_decode(wl, q, kd, vd, sl, case.scale, threads)
    one = max(time.perf_counter() - t, 1e-4)
    n = max(1, min(wl.batch, int(seconds / one)))
    rows = list(range(n))
    q, kd, vd, sl = _oracle_inputs(wl, case, rows)
    t = time.perf_counter()
    _oracle_decode(wl, q, kd, vd, sl, case.scale, threads)
    dt = time.perf_counter() - t
    reps = max(1, int(seconds / max(dt, 1e-3))) if n == wl.batch else 1
    if reps > 1:
        t = time.perf_counter()
        for _ in range(reps):
            _oracle_decode(wl, q, kd, vd, sl, case.scale, threads)
        dt = (time.perf_counter() - t) / reps
    lens = case.context_lens.cpu().tolist()
    sub = algorithmic_bytes(wl, [lens[b] for b in rows])
    # the same oracle on one thread, on sequence 0 alone
    q1, kd1, vd1, sl1 = _oracle_inputs(wl, case, [0])
    t = time.perf_counter()
    _oracle_decode(wl, q1, kd1, vd1, sl1, case.scale, 1)
    dt1 = time.perf_counter() - t
    one = algorithmic_bytes(wl, [lens[0]])
    return {"value": round(sub["decode"] / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt * reps, 3),
            "sample": f"{n} of {wl.batch} sequences (all {wl.num_heads} heads) x {reps} passes, "
                      f"fp64 C oracle, decode only",
            "one_thread": {"value": round(one["decode"] / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                           "seconds": round(dt1, 3),
                           "sample": f"sequence 0 ({lens[0]} tokens, all {wl.num_heads} heads), "
                                     "fp64 C oracle on one thread"}}


def run_reference(args):
    """The oracle as the reference arm: each step decodes a bounded sample of the
    workload on the host cores (rank 0 only)."""
    import torch
    world, rank, local = dist_info()
    if rank != 0:
        return
    import gqa_inputs as gi
    import oracle
    oracle.build()
    wl = resolve_workload(args.workload, args.batch)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = gi.case_for(wl, seed=args.seed, device=dev, extra_tokens=0)
    threads = oracle.num_cpus()
    if wl.kind == "prefill":
        return run_reference_prefill(args, wl, case, threads, world)
    rows = [0]
    q, kd, vd, sl = _oracle_inputs(wl, case, rows)
    lens = case.context_lens.cpu().tolist()
    sample_bytes = algorithmic_bytes(wl, [lens[b] for b in rows])["decode"]
    for _ in range(max(3, args.warmup)):
        _oracle_decode(wl, q, kd, vd, sl, case.scale, threads)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        _oracle_decode(wl, q, kd, vd, sl, case.scale, threads)
        times.append(time.perf_counter() - t)
    dt = statistics.mean(times)
    v = round(sample_bytes / dt / 1e9, 4)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "num_heads": wl.num_heads,
                   "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim,
                   "context_lens": wl.lens, "cache_dtype": wl.cache_dtype},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"1 of {wl.batch} sequences (all {wl.num_heads} heads) per step, "
                                   "fp64 C oracle"},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_prefill(args, wl, case, threads, world):
    """Reference arm of a prefill workload: each step runs the oracle on the last
    queries of sequence 0 (about a second of host time), in TFLOP/s."""
    import oracle
    q, kd, vd, sl = _oracle_inputs(wl, case, [0])
    T, L = wl.queries, int(sl[0])
    n = 1
    while n < T:
        t = time.perf_counter()
        oracle.decode(q[:, T - n:], kd, vd, sl, case.scale, nthreads=threads, window=wl.window)
        if time.perf_counter() - t > 0.5:
            break
        n = min(T, n * 2)
    sub = q[:, T - n:]
    att = sum(min(L - T + i + 1, wl.window) if wl.window > 0 else L - T + i + 1 for i in range(T - n, T))
    f = 4.0 * wl.head_dim * wl.num_heads * att
    for _ in range(max(3, args.warmup)):
        oracle.decode(sub, kd, vd, sl, case.scale, nthreads=threads, window=wl.window)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.decode(sub, kd, vd, sl, case.scale, nthreads=threads, window=wl.window)
        times.append(time.perf_counter() - t)
    dt = statistics.mean(times)
    v = round(f / dt / 1e12, 6)
    sample = f"last {n} of {T} prompt tokens of sequence 0 (all {wl.num_heads} heads) per step, fp64 C oracle"
    print(json.dumps({
        "impl": "reference", "metric": "prefill attention TFLOP/s (causal, algorithmic flops), 1 GPU",
        "value": v, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "prompt_tokens": T,
                   "num_heads": wl.num_heads, "num_kv_heads": wl.num_kv_heads,
                   "head_dim": wl.head_dim, "context_lens": wl.lens},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--kernel", choices=["auto", "mma", "fma"], default="auto")
    ap.add_argument("--prefill-kernel", choices=list(PREFILL_KERNEL), default="auto",
                    help="prefill workloads: two-tile tcgen05 (tc2), one-tile tcgen05 (tc1) or mma.sync")
    ap.add_argument("--row-layout", choices=list(ROW_LAYOUT), default="auto",
                    help="more than 8 query rows per kv-head: 8-row unit streams or a shared ring")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0,
                    help="keep only the first N sequences of the workload (smaller case for profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-read-probe", action="store_true",
                    help="skip the HBM read-ceiling probe (decode workloads)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
