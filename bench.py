#!/usr/bin/env python
"""Benchmark of the exact-attention hot path on GB300.

One step is one pass of the whole hot path over one batch of synthetic
input, on one GPU:
  * forward: b4 s512 h32 d128 bf16 (the problem timed in "Why
    FlashAttention is fast"), O and LSE, one kernel;
  * split-KV decode: b1 h16 sk32768 d128 bf16 (the small-batch decode of
    the flash-decoding issue), heuristic split count, one split kernel whose
    last-finishing split of each head does the LSE combine.
Headline: forward TFLOP/s (4*b*h*sq*sk*d per call); decode is reported as
HBM GB/s beside it. Inputs are resident in HBM when the timed region starts;
L2 is flushed before every timed kernel: a 512 MiB write, then a read of a
second 512 MiB buffer, so that the write's own dirty lines are back in HBM
before the timed kernel starts (the clean state ncu's cache control leaves)
instead of being written back inside it; the same kernels after the write
alone are in ``extras.write_only_flush``. Each kernel is timed with CUDA
events on the stream it runs on.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (launched by torchrun, one process per GPU) every rank runs the
same problem on its own GPU: the path has no exchange step, so the ranks are
independent replicas; ``value`` is the work of all ranks over the slowest
rank's time. ``--impl reference`` times the fp64 CPU oracle instead, on a
bounded sample of the same forward problem, on rank 0's host cores.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "fwd attention TFLOP/s (b4 s512 h32 d128 bf16); split-KV decode HBM GB/s"
FWD = workloads.WORKLOADS["mid_fwd"]
DEC = workloads.WORKLOADS["decode_b1_h16_sk32768"]
# The pages' own figure for this forward problem: ~9.7 ms per flash_attn_func
# call, 17.18 GFLOP, i.e. about 1.77 TFLOP/s (wall clock, unspecified GPU).
PAGE_FWD_TFLOPS = 1.77
FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CONFIG = {
    "workload": "fwd b4 s512 h32 d128 bf16 + split-KV decode b1 h16 sk32768 d128 bf16",
    "fwd": {"b": FWD.b, "sq": FWD.sq, "sk": FWD.sk, "h": FWD.h, "d": FWD.d, "dtype": "bf16",
            "causal": False},
    "decode": {"b": DEC.b, "sq": DEC.sq, "sk": DEC.sk, "h": DEC.h, "d": DEC.d, "dtype": "bf16",
               "num_splits": "heuristic"},
    "l2": "flushed before every timed kernel: a 512 MiB write, then a read of a second 512 MiB "
          "buffer (the write's dirty lines go back to HBM before the timed kernel; "
          "extras.write_only_flush has the same kernels after the write alone)",
    "inputs": "seeded N(0,1), torch.Generator seed 42, fp32 draw rounded to bf16",
    "parallelism": "replicas (no exchange step)",
}


# ------------------------------------------------------------------ ranks
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, ws, local


def dist_init(backend: str):
    rank, ws, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, ws


def aggregate(local_ms: dict, local_units: dict) -> tuple[dict, dict]:
    """Max of each timing and sum of each work count over all ranks (identity
    on one rank)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return dict(local_ms), dict(local_units)
    dev = torch.device("cuda", torch.cuda.current_device()) if (
        dist.get_backend() == "nccl") else torch.device("cpu")
    keys_t, keys_u = sorted(local_ms), sorted(local_units)
    t = torch.tensor([local_ms[k] for k in keys_t], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units[k] for k in keys_u], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return ({k: float(x) for k, x in zip(keys_t, t.tolist())},
            {k: float(x) for k, x in zip(keys_u, u.tolist())})


def barrier():
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------------ peaks / profiles
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# the sources each captured kernel is compiled from
KERNEL_SOURCES = {
    "fwd_mid": ("exact_attention_65_gb300/csrc/fwd.cu", "exact_attention_65_gb300/csrc/ptx.cuh",
                "exact_attention_65_gb300/csrc/internal.h"),
    "decode_b1": ("exact_attention_65_gb300/csrc/decode.cu", "exact_attention_65_gb300/csrc/ptx.cuh",
                  "exact_attention_65_gb300/csrc/internal.h"),
}


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def ncu_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel's current sources; otherwise None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get("kernels", {}).get(kernel)
    if e is None or e.get("source_sha256") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100", "-f", self.path]
            if self.uuid:
                cmd[1:1] = ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.4)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        power = [float(r[4]) for r in rows if r[4].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ our arm
def place(w, dev, pin=False):
    q, k, v = workloads.make_workload(w, pin=pin)
    return (q, k, v), tuple(t.to(dev, non_blocking=False) for t in (q, k, v))


def time_loop(fns, steps, warmup, flush, stream):
    """Run `fns` (list of callables) per step, each preceded by an L2 flush
    and bracketed by events; return mean ms per callable and the wall s."""
    for _ in range(warmup):
        for fn in fns:
            flush()
            fn()
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in fns] for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        for j, fn in enumerate(fns):
            flush()
            ev[i][j][0].record(stream)
            fn()
            ev[i][j][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - t0
    ms = [sum(ev[i][j][0].elapsed_time(ev[i][j][1]) for i in range(steps)) / steps
          for j in range(len(fns))]
    return ms, wall


def cpu_baseline(host_qkv, seconds: float = 8.0):
    """Time the fp64 oracle, as it stands, on a bounded sample of the forward
    problem: R query rows of every (b, h), R chosen for about `seconds`."""
    import oracle

    oracle.build()
    q, k, v = host_qkv
    per_row_flops = 4 * FWD.sk * FWD.d * FWD.b * FWD.h
    t0 = time.perf_counter()
    oracle.attention(q, k, v, FWD.scale, rows=list(range(4)))
    t_probe = max(time.perf_counter() - t0, 1e-4)
    rows_n = int(min(FWD.sq, max(4, 4 * seconds / t_probe)))
    rows = list(range(0, FWD.sq, max(1, FWD.sq // rows_n)))[:rows_n]
    t0 = time.perf_counter()
    oracle.attention(q, k, v, FWD.scale, rows=rows)
    dt = time.perf_counter() - t0
    return {"value": per_row_flops * len(rows) / dt / 1e12, "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"fp64 oracle on {len(rows)} of {FWD.sq} query rows of every (b, h) of "
                      f"b4 s512 h32 d128 ({dt:.1f} s)"}


def run_ours(args):
    import exact_attention_65_gb300 as ea

    rank, ws, local = dist_env()
    torch.cuda.set_device(local)
    dist_init("nccl")
    dev = torch.device("cuda", local)
    ea.load_library()
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()

    (hq, hk, hv), (q, k, v) = place(FWD, dev, pin=True)
    _, (dq, dk, dv) = place(DEC, dev)
    o = torch.empty_like(q)
    lse = torch.empty(FWD.b, FWD.h, FWD.sq, dtype=torch.float32, device=dev)
    do = torch.empty_like(dq)
    dlse = torch.empty(DEC.b, DEC.h, DEC.sq, dtype=torch.float32, device=dev)
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean_buf = torch.zeros(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.zero_()
        # one reduction kernel reading the whole buffer (int32 max: no
        # conversion pass, so nothing else is written)
        clean_buf.view(torch.int32).max()

    def flush_write_only():
        flush_buf.zero_()

    splits = ea.attn_decode_num_splits(DEC.b, DEC.sq, DEC.sk, DEC.h, DEC.d)

    def fwd():
        ea.attn_fwd(q, k, v, scale=FWD.scale, out=o, lse=lse)

    def dec():
        ea.attn_decode_splitkv(dq, dk, dv, scale=DEC.scale, num_splits=0, out=do, lse=dlse)

    if ea.attn_get_device_status() != ea.ATTN_OK:
        raise RuntimeError("device status not clean before the benchmark")

    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    sampler = ClockSampler(f"GPU-{uuid}" if uuid is not None else None)
    sampler.start()
    (fwd_ms, dec_ms), wall = time_loop([fwd, dec], args.steps, args.warmup, flush, stream)
    clocks = sampler.stop()
    if ea.attn_get_device_status() != ea.ATTN_OK:
        raise RuntimeError("a kernel reported a timeout during the timed region")

    # end to end through the public API: one attn_fwd_host call per step on
    # pinned host buffers (its device workspace, uploads, forward and
    # downloads all inside the timed region, on this stream and the
    # library's two copy streams joined back to it)
    e2e_steps = min(args.steps, 200)
    ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)

    def e2e_step():
        ea.attn_fwd_host(hq, hk, hv, scale=FWD.scale, out=ho, lse=hl, sync=False)

    (e2e_ms,), _ = time_loop([e2e_step], e2e_steps, 3, lambda: None, stream)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()

    times, units = aggregate(
        {"fwd_ms": fwd_ms, "dec_ms": dec_ms, "e2e_ms": e2e_ms, "wall_s": wall},
        {"fwd_flops": FWD.flops, "dec_bytes": DEC.io_bytes})
    n = ws
    fwd_tflops = units["fwd_flops"] / (times["fwd_ms"] * 1e-3) / 1e12
    dec_gbs = units["dec_bytes"] / (times["dec_ms"] * 1e-3) / 1e9
    per_rank_fwd_tflops = FWD.flops / (fwd_ms * 1e-3) / 1e12
    per_rank_dec_gbs = DEC.io_bytes / (dec_ms * 1e-3) / 1e9
    e2e_tflops = units["fwd_flops"] / (times["e2e_ms"] * 1e-3) / 1e12

    extras = {}
    if rank == 0 and not args.no_extras:
        extras = measure_extras(ea, dev, flush, stream, peaks)
        # the headline kernels after the write alone: its dirty lines are then
        # written back to HBM inside the timed kernel
        (w_fwd, w_dec), _ = time_loop([fwd, dec], min(args.steps, 200), 3, flush_write_only, stream)
        extras["write_only_flush"] = {
            "fwd_ms": round(w_fwd, 5), "fwd_TFLOP/s": round(FWD.flops / (w_fwd * 1e-3) / 1e12, 2),
            "decode_ms": round(w_dec, 5),
            "decode_GB/s": round(DEC.io_bytes / (w_dec * 1e-3) / 1e9, 1)}
    cpu = cpu_baseline((hq, hk, hv)) if (rank == 0 and ws == 1 and not args.no_cpu) else None

    line = {
        "metric": METRIC,
        "value": round(fwd_tflops, 3),
        "unit": "TFLOP/s",
        "n_gpus": n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(times["fwd_ms"] + times["dec_ms"], 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(fwd_tflops / PAGE_FWD_TFLOPS, 2),
        "dtype": "bf16",
        "data": "synthetic",
        "config": CONFIG,
        "decode": {"value": round(dec_gbs, 1), "unit": "GB/s", "splits": splits,
                   "ms": round(times["dec_ms"], 5)},
        "fwd_ms": round(times["fwd_ms"], 5),
        "wall_ms_per_step_incl_flush": round(times["wall_s"] * 1e3 / args.steps, 4),
        "roofline": {"bound": "tensor", "achieved": round(per_rank_fwd_tflops, 2),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(per_rank_fwd_tflops / peaks["bf16_tflops"], 4),
                     "traffic": ncu_traffic("fwd_mid"), "peak_source": peak_src,
                     "kernel": "fwd_kernel<128, bf16>", "algorithmic_per_launch": FWD.flops},
        "roofline_decode": {"bound": "hbm", "achieved": round(per_rank_dec_gbs, 1),
                            "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": round(per_rank_dec_gbs / peaks["hbm_gbs"], 4),
                            "traffic": ncu_traffic("decode_b1"), "peak_source": peak_src,
                            "kernel": "decode_split_kernel<128, 1, bf16> (combine in-kernel)",
                            "algorithmic_per_launch": DEC.io_bytes},
        "e2e": {"value": round(e2e_tflops, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(times["e2e_ms"], 4)},
        "gpu_launches": args.steps * 2,  # the forward kernel and the split decode kernel
        "clocks": clocks,
        "cpu_baseline": cpu,
        "extras": extras,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier()
    if dist.is_initialized():
        dist.destroy_process_group()


def host_call_us(ea, q, k, v, w, stream, calls=200):
    """Host time to issue one forward (small problems are dominated by it):
    the Python binding and the bare C-ABI call, each averaged over `calls`
    calls issued while the GPU is held busy, so the host never waits."""
    lib = ea.load_library()
    o = torch.empty_like(q)
    lse = torch.empty((w.b, w.h, w.sq), dtype=torch.float32, device=q.device)
    st = ctypes.c_void_p(stream.cuda_stream)
    dt = ea.ATTN_BF16 if w.dtype == torch.bfloat16 else ea.ATTN_FP16
    res = {}
    for label, fn in (
            ("python", lambda: ea.attn_fwd(q, k, v, scale=w.scale, out=o, lse=lse)),
            ("c_abi", lambda: lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                           lse.data_ptr(), w.b, w.sq, w.sk, w.h, w.d, w.scale, dt,
                                           st))):
        fn()
        torch.cuda.synchronize()
        torch.cuda._sleep(int(2e8))  # about 0.1 s of GPU time at ~2 GHz
        t0 = time.perf_counter()
        for _ in range(calls):
            fn()
        res[label] = round((time.perf_counter() - t0) / calls * 1e6, 2)
        torch.cuda.synchronize()
    return res


def measure_extras(ea, dev, flush, stream, peaks):
    """Per-problem kernel times for the other workloads (20 timed calls each)."""
    out = {}
    gen = torch.Generator(device=dev)
    gen.manual_seed(workloads.SEED)

    def rand(w):
        q = torch.randn((w.b, w.sq, w.h, w.d), generator=gen, device=dev).to(w.dtype)
        k = torch.randn((w.b, w.sk, w.h, w.d), generator=gen, device=dev).to(w.dtype)
        v = torch.randn((w.b, w.sk, w.h, w.d), generator=gen, device=dev).to(w.dtype)
        return q, k, v

    for name in ("tiny_fwd", "small_head_b2_s50", "small_head_b2_s300", "small_head_b512_s150",
                 "long_fwd"):
        w = workloads.WORKLOADS[name]
        q, k, v = rand(w)
        fn = lambda: ea.attn_fwd(q, k, v, scale=w.scale)  # noqa: E731
        (ms,), _ = time_loop([fn], 20, 3, flush, stream)
        tf = w.flops / (ms * 1e-3) / 1e12
        gbs = w.io_bytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": round(ms, 5), "TFLOP/s": round(tf, 2),
                     "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                     "GB/s": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)}
        if name != "long_fwd":
            out[name]["host_call_us"] = host_call_us(ea, q, k, v, w, stream)
        if name == "small_head_b512_s150":
            # the same problem on the general key-tile-loop kernel, which the
            # short forward (all keys of a head in one tile) replaces here
            ea.attn_debug_set_flags(ea.ATTN_DEBUG_GENERAL_FWD)
            try:
                (ms,), _ = time_loop([fn], 20, 3, flush, stream)
            finally:
                ea.attn_debug_set_flags(0)
            out[name + "/general_kernel"] = {"ms": round(ms, 5),
                                             "GB/s": round(w.io_bytes / (ms * 1e-3) / 1e9, 1)}
        del q, k, v
    # causal forward (bottom-right aligned; sq == sk here): FLOP counts only
    # the unmasked scores, 4*b*h*d * sum over rows of the keys a row sees
    for name in ("mid_fwd", "long_fwd"):
        w = workloads.WORKLOADS[name]
        q, k, v = rand(w)
        fn = lambda: ea.attn_fwd(q, k, v, scale=w.scale, causal=True)  # noqa: E731
        (ms,), _ = time_loop([fn], 20, 3, flush, stream)
        flops = 4 * w.b * w.h * w.d * (w.sq * (w.sq + 1) // 2)
        tf = flops / (ms * 1e-3) / 1e12
        out[f"{name}/causal"] = {"ms": round(ms, 5), "TFLOP/s": round(tf, 2),
                                 "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4)}
        del q, k, v
    # backward pass (dQ, dK, dV); FLOP = the five products of the chain
    # rule, 10*b*h*sq*sk*d (the dQ pass recomputes two of them, not counted);
    # the small-head shapes are the ones the flash-attn timing issue times
    # forward and backward
    for name in ("small_head_b2_s300", "small_head_b512_s150"):
        w = workloads.WORKLOADS[name]
        q, k, v = rand(w)
        do = torch.randn((w.b, w.sq, w.h, w.d), generator=gen, device=dev).to(w.dtype)
        o, lse = ea.attn_fwd(q, k, v, scale=w.scale)
        fn = lambda: ea.attn_bwd(q, k, v, o, lse, do, scale=w.scale)  # noqa: E731
        (ms,), _ = time_loop([fn], 10, 3, flush, stream)
        tf = 10 * w.b * w.h * w.sq * w.sk * w.d / (ms * 1e-3) / 1e12
        io = 8 * w.b * w.sq * w.h * w.d * w.elem_bytes  # q, k, v, o, dO read; dq, dk, dv written
        out[f"{name}/backward"] = {"ms": round(ms, 5), "TFLOP/s": round(tf, 2),
                                   "GB/s": round(io / (ms * 1e-3) / 1e9, 1)}
        del q, k, v, do, o, lse
    for name in ("mid_fwd", "long_fwd"):
        w = workloads.WORKLOADS[name]
        q, k, v = rand(w)
        do = torch.randn((w.b, w.sq, w.h, w.d), generator=gen, device=dev).to(w.dtype)
        o, lse = ea.attn_fwd(q, k, v, scale=w.scale)
        fn = lambda: ea.attn_bwd(q, k, v, o, lse, do, scale=w.scale)  # noqa: E731
        (ms,), _ = time_loop([fn], 10, 3, flush, stream)
        tf = 10 * w.b * w.h * w.sq * w.sk * w.d / (ms * 1e-3) / 1e12
        out[f"{name}/backward"] = {"ms": round(ms, 5), "TFLOP/s": round(tf, 2),
                                   "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4)}
        # causal backward: the five products over the unmasked scores only
        o, lse = ea.attn_fwd(q, k, v, scale=w.scale, causal=True)
        fn = lambda: ea.attn_bwd(q, k, v, o, lse, do, scale=w.scale,  # noqa: E731
                                 causal=True)
        (ms,), _ = time_loop([fn], 10, 3, flush, stream)
        tf = 10 * w.b * w.h * w.d * (w.sq * (w.sq + 1) // 2) / (ms * 1e-3) / 1e12
        out[f"{name}/backward_causal"] = {"ms": round(ms, 5), "TFLOP/s": round(tf, 2),
                                          "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4)}
        del q, k, v, do, o, lse
    # several new query rows share each K/V read (tensor-core decode path)
    for name, sq in (("decode_b8_h48_sk8192", 10), ("decode_b1_h16_sk32768", 10)):
        w = workloads.WORKLOADS[name]
        gen_q = torch.randn((w.b, sq, w.h, w.d), generator=gen, device=dev).to(w.dtype)
        _, k, v = rand(w)
        for causal in (False, True):
            fn = lambda: ea.attn_decode_splitkv(gen_q, k, v, scale=w.scale,  # noqa: E731
                                                causal=causal)
            (ms,), _ = time_loop([fn], 20, 3, flush, stream)
            kv = 2 * k.numel() * k.element_size()
            gbs = kv / (ms * 1e-3) / 1e9
            tag = "/causal" if causal else ""
            out[f"{name}/sq={sq}{tag}"] = {"ms": round(ms, 5), "GB/s (K+V)": round(gbs, 1),
                                           "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)}
        del k, v, gen_q
    # paged KV cache: the same decode problems with K/V in shuffled pages of
    # 256 keys behind a block table
    for name in ("decode_b8_h48_sk8192", "decode_b1_h16_sk32768"):
        w = workloads.WORKLOADS[name]
        q, k, v = rand(w)
        ps = 256
        npg = w.sk // ps
        perm = torch.randperm(w.b * npg, generator=gen, device=dev)
        kp = torch.empty((w.b * npg, ps, w.h, w.d), dtype=w.dtype, device=dev)
        vp = torch.empty_like(kp)
        kp[perm] = k.reshape(w.b * npg, ps, w.h, w.d)
        vp[perm] = v.reshape(w.b * npg, ps, w.h, w.d)
        table = perm.to(torch.int32).reshape(w.b, npg).contiguous()
        lens = torch.full((w.b,), w.sk, dtype=torch.int32, device=dev)
        del k, v
        fn = lambda: ea.attn_decode_paged(q, kp, vp, table, lens, scale=w.scale)  # noqa: E731
        (ms,), _ = time_loop([fn], 20, 3, flush, stream)
        gbs = w.io_bytes / (ms * 1e-3) / 1e9
        out[f"{name}/paged256"] = {"ms": round(ms, 5), "GB/s": round(gbs, 1),
                                   "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)}
        del q, kp, vp
    # paged KV cache with small pages: one new row per sequence, and 10 new
    # rows (the tensor-core path, 128-key tiles gathered from 64-key pages)
    for name in ("decode_b8_h48_sk8192", "decode_b1_h16_sk32768"):
        w = workloads.WORKLOADS[name]
        _, k, v = rand(w)
        for ps in (16, 64):
            npg = w.sk // ps
            perm = torch.randperm(w.b * npg, generator=gen, device=dev)
            kp = torch.empty((w.b * npg, ps, w.h, w.d), dtype=w.dtype, device=dev)
            vp = torch.empty_like(kp)
            kp[perm] = k.reshape(w.b * npg, ps, w.h, w.d)
            vp[perm] = v.reshape(w.b * npg, ps, w.h, w.d)
            table = perm.to(torch.int32).reshape(w.b, npg).contiguous()
            lens = torch.full((w.b,), w.sk, dtype=torch.int32, device=dev)
            kv = 2 * kp.numel() * kp.element_size()
            for sq in (1, 10):
                q = torch.randn((w.b, sq, w.h, w.d), generator=gen, device=dev).to(w.dtype)
                fn = lambda: ea.attn_decode_paged(q, kp, vp, table, lens,  # noqa: E731
                                                  scale=w.scale)
                (ms,), _ = time_loop([fn], 20, 3, flush, stream)
                gbs = kv / (ms * 1e-3) / 1e9
                out[f"{name}/paged{ps}/sq={sq}"] = {"ms": round(ms, 5), "GB/s (K+V)": round(gbs, 1),
                                                    "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)}
                del q
            del kp, vp, table
        del k, v
    for name, split_list in (("decode_b8_h48_sk8192", [0]),
                             ("decode_b1_h16_sk32768", [0, 1, 2, 4, 8, 16])):
        w = workloads.WORKLOADS[name]
        q, k, v = rand(w)
        for s in split_list:
            fn = lambda: ea.attn_decode_splitkv(q, k, v, scale=w.scale, num_splits=s)  # noqa: E731
            (ms,), _ = time_loop([fn], 20, 3, flush, stream)
            gbs = w.io_bytes / (ms * 1e-3) / 1e9
            out[f"{name}/splits={s}"] = {"ms": round(ms, 5), "GB/s": round(gbs, 1),
                                         "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)}
        del q, k, v
    if ea.attn_get_device_status() != ea.ATTN_OK:
        raise RuntimeError("a kernel reported a timeout during the extra measurements")
    return out


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    """The fp64 CPU oracle timed on rank 0's host cores, each step a bounded
    sample of the forward problem."""
    rank, ws = dist_init("gloo")
    if rank != 0:
        return
    import oracle

    oracle.build()
    q, k, v = workloads.make_workload(FWD)
    per_row_flops = 4 * FWD.sk * FWD.d * FWD.b * FWD.h
    t0 = time.perf_counter()
    oracle.attention(q, k, v, FWD.scale, rows=[0])
    t_row = max(time.perf_counter() - t0, 1e-5)
    budget_s = 150.0 / max(1, args.steps + args.warmup)  # whole run within a few minutes
    rows_n = int(max(1, min(FWD.sq, budget_s / t_row)))
    rows = list(range(rows_n))
    for _ in range(args.warmup):
        oracle.attention(q, k, v, FWD.scale, rows=rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention(q, k, v, FWD.scale, rows=rows)
    dt = time.perf_counter() - t0
    value = per_row_flops * rows_n * args.steps / dt / 1e12
    sample = (f"fp64 oracle on {rows_n} of {FWD.sq} query rows of every (b, h) of "
              "b4 s512 h32 d128 per step")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": CONFIG,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip the per-problem extra timings")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--backward", action="store_true",
                    help="with --profile-only on a forward workload: run its backward pass instead")
    ap.add_argument("--profile-only", choices=sorted(workloads.WORKLOADS), default=None,
                    help="profiling aid: only run warmup + steps calls of one workload's kernels "
                         "(no timing, no JSON line), e.g. under ncu")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    _, ws, _ = dist_env()
    if args.gpus != ws and not (args.gpus == 1 and ws == 1):
        if ws == 1 and args.gpus > 1:
            ap.error("--gpus N > 1 runs under torchrun, one process per GPU")
    if args.profile_only:
        run_profile_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


def run_profile_only(args):
    """Runs one workload's kernels (forward, or split-KV decode with the
    heuristic split count) warmup + steps times on seeded device inputs."""
    import exact_attention_65_gb300 as ea

    w = workloads.WORKLOADS[args.profile_only]
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(workloads.SEED)
    q = torch.randn((w.b, w.sq, w.h, w.d), generator=gen, device=dev).to(w.dtype)
    k = torch.randn((w.b, w.sk, w.h, w.d), generator=gen, device=dev).to(w.dtype)
    v = torch.randn((w.b, w.sk, w.h, w.d), generator=gen, device=dev).to(w.dtype)
    fn = (lambda: ea.attn_fwd(q, k, v)) if w.kind == "fwd" else (
        lambda: ea.attn_decode_splitkv(q, k, v, num_splits=0))
    if args.backward:
        if w.kind != "fwd":
            raise SystemExit("--backward needs a forward workload")
        do = torch.randn((w.b, w.sq, w.h, w.d), generator=gen, device=dev).to(w.dtype)
        o, lse = ea.attn_fwd(q, k, v)
        fn = lambda: ea.attn_bwd(q, k, v, o, lse, do)  # noqa: E731
    for _ in range(args.warmup + args.steps):
        fn()
    if ea.attn_get_device_status() != ea.ATTN_OK:
        raise RuntimeError("a kernel reported a timeout")


if __name__ == "__main__":
    main()
