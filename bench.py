#!/usr/bin/env python3
"""Benchmark of the paged-attention hot path on GB300.

One step = one call of the C-ABI entry point over one batch of the workload
(for the decode workload: the split page-walk kernel and the combine kernel).
Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload decode|prefill|tails|long_decode|tiny] [--op attention|append]
                  [--schedule auto|decode|prefill] [--no-causal] [--mask]
  python bench.py --workload mixed   (a ragged continuous-batching step)

Default workload: batched decode, B=64, L=1, H_q=32, H_kv=8, D=128,
page_size=128, context lengths U{128..4096}, scattered pages (seeded).
Metric: achieved HBM GB/s = algorithmic bytes / device time (bf16), or TFLOP/s
= 4 * H_q * D * visible (row, key) pairs / device time where the FLOP time at
the measured bf16 rate exceeds the byte time at the measured copy bandwidth
(the causal prefill).

The default line (the decode workload) carries a `prefill` record: the causal
prefill workload (B=4, L=S=2048) measured the same way in the same run, in
TFLOP/s, with its own roofline, e2e, clocks and cpu_baseline (--no-prefill
leaves it out).

The timed region holds two passes of K steps: the call as a user makes it
(value, ms_per_step) and the same calls with CUDA events around the dominant
kernel (roofline.achieved); L2 is flushed between steps.

--impl reference times the fp64 CPU oracle on the host cores over a bounded
sample of the same workload (the method has no other reference program).

--no-causal runs the workload with mask=None (every key of the context visible)
instead of the causal rule.

--mask adds a seeded fp32 additive mask [B * H_q, L, S_mask] (N(0,1) biases,
a third of the positions at -inf) to every call; the mask read makes every
workload HBM-bound, so the line is in GB/s with the visible mask bytes
counted.

--op append measures the K/V append instead (pa_append_kv: the workload's L
new tokens per sequence written into their pages), in HBM GB/s.
Under torchrun each rank runs its own replica (the path has no exchange
step); rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_cache_03_gb300 import synth  # noqa: E402

METRIC = "paged-attn decode HBM GB/s & prefill TFLOP/s vs GB300 roofline (bf16, d128)"
METRIC_MASKED = "paged-attn with an fp32 additive mask, HBM GB/s (bf16, d128)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300's nominal figures: HBM3e copy bandwidth and dense bf16 tensor rate.
NOMINAL_PEAKS = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}
L2_FLUSH_BYTES = 256 << 20

METRIC_MIXED = "paged-attn ragged batch (decode steps + prefill chunks), HBM GB/s (bf16, d128)"


# ---------------------------------------------------------------------------
# algorithmic work (per call)
# ---------------------------------------------------------------------------
def algorithmic_bytes(inp) -> int:
    """Minimum bytes one call moves: every visible K and V row of each
    (sequence, kv head) once (2 * H_kv * D * elt per context token), query in
    and output out once, the block-table entries of the used pages and the
    context lengths."""
    es = 2 if inp.dtype == "bf16" else 4
    tokens = int(inp.context_lens.astype(np.int64).sum())
    kv = 2 * inp.H_kv * inp.D * es * tokens
    qo = 2 * inp.query.size * es
    pages = sum((int(s) + inp.page_size - 1) // inp.page_size for s in inp.context_lens)
    return kv + qo + 4 * pages + 4 * inp.B


def visible_pairs(inp) -> int:
    """(query row, key) pairs with the key visible, per query head."""
    L = inp.L
    tot = 0
    for s in inp.context_lens.astype(np.int64):
        s = int(s)
        tot += (L * (s - L) + L * (L + 1) // 2) if inp.causal else L * s
    return tot


def algorithmic_flops(inp) -> int:
    """4 * H_q * D * visible pairs: a multiply-add per element of Q.K^T and
    of P.V."""
    return 4 * inp.H_q * inp.D * visible_pairs(inp)


def ragged_bytes(r) -> int:
    """Minimum bytes of one ragged-batch call: every visible K and V row of
    each sequence with queries once, queries in and outputs out once, the
    used block-table entries, context lengths and offsets."""
    es = 2 if r.dtype == "bf16" else 4
    lens = r.q_lens
    ctx = r.context_lens.astype(np.int64)
    live = lens > 0
    kv = 2 * r.H_kv * r.D * es * int(ctx[live].sum())
    qo = 2 * r.query.size * es
    pages = int(sum((int(s) + r.page_size - 1) // r.page_size for s in ctx[live]))
    return kv + qo + 4 * pages + 4 * r.B + 4 * (r.B + 1)


def ragged_flops(r) -> int:
    """4 * H_q * D per visible (query row, key) pair."""
    tot = 0
    for Lb, S in zip(r.q_lens, r.context_lens):
        Lb, S = int(Lb), int(S)
        tot += (Lb * (S - Lb) + Lb * (Lb + 1) // 2) if r.causal else Lb * S
    return 4 * r.H_q * r.D * tot


def mask_bytes(inp) -> int:
    """Bytes of an fp32 additive mask a call must read: one element per
    visible (query row, key) pair of every query head."""
    return 4 * inp.H_q * visible_pairs(inp)


def mask_width(inp) -> int:
    """S_mask of the benchmarked masks: the block table's capacity rounded up
    to a multiple of 4."""
    cap = inp.block_table.shape[1] * inp.page_size
    return (cap + 3) // 4 * 4


def append_bytes(inp) -> int:
    """Minimum bytes one K/V append moves: the new K and V rows read once and
    written once into the pool (2 tensors x 2 x B*H_kv*L*D*elt), the
    block-table entries of the pages that receive them and the context
    lengths."""
    es = 2 if inp.dtype == "bf16" else 4
    rows = 2 * inp.B * inp.H_kv * inp.L * inp.D * es
    pages = 0
    for s in inp.context_lens.astype(np.int64):
        s = int(s)
        pages += (s - 1) // inp.page_size - (s - inp.L) // inp.page_size + 1
    return 2 * rows + 4 * pages + 4 * inp.B


def workload_desc(name, inp) -> str:
    kw = synth.WORKLOADS[name]
    ctx = (f"ctx~U[{kw['ctx_range'][0]},{kw['ctx_range'][1]}]" if "ctx_range" in kw
           else f"ctx={sorted(set(int(x) for x in inp.context_lens))}")
    ks = f" K*{kw['k_scale']}" if kw.get("k_scale", 1.0) != 1.0 else ""
    return (f"{name}: B={inp.B} L={inp.L} H_q={inp.H_q} H_kv={inp.H_kv} D={inp.D} "
            f"page_size={inp.page_size} pool={inp.num_pages} pages {ctx} "
            f"{'causal' if inp.causal else 'full'}{ks} seed={kw['seed']}")


def bench_inputs(args):
    """The named workload, with every key before the frontier visible
    (mask=None) under --no-causal."""
    return synth.workload(args.workload, **({"causal": False} if args.no_causal else {}))


def variant(args) -> str:
    """Workload key of the recorded traffic: the workload name, +full for
    --no-causal, +mask for --mask."""
    return args.workload + ("+full" if args.no_causal else "") + ("+mask" if args.mask else "")


def roofline_bound(bytes_step, flops_step, peaks) -> str:
    """The roofline that binds a call: the larger of its byte time at the
    measured copy bandwidth and its FLOP time at the measured bf16 rate."""
    t_bytes = bytes_step / (peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]) * 1e9)
    t_flops = flops_step / (peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]) * 1e12)
    return "hbm" if t_bytes >= t_flops else "tensor"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# The sources each kernel is built from: its recorded DRAM traffic stays valid
# while these are unchanged.
KERNEL_SOURCES = {
    "decode_split_kernel": ("decode.cu", "ptx.cuh", "tc.cuh", "internal.h"),
    "prefill_tile_kernel": ("prefill.cu", "tc.cuh", "ptx.cuh", "internal.h"),
    "append_kv_kernel": ("append.cu", "internal.h"),
}


def _code_only(text: str) -> str:
    """The source without comments and blank lines (so that a comment edit
    does not retire the recorded counters)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln.strip())


def kernel_source_digest(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_03_gb300", "csrc")
    for fn in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, fn), encoding="utf-8") as f:
            h.update(fn.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel sources changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[f"{kernel}@{workload}"]
        if e.get("source_digest") != kernel_source_digest(kernel):
            return None
        return int(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        try:
            fd, self.path = tempfile.mkstemp(prefix="pa_clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons, pw = [], [], set(), []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 5:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                    pw.append(float(parts[3]))
                    bits = int(parts[4], 16)
                except ValueError:
                    continue
                for b, name in REASON_BITS.items():
                    if bits & b and name != "gpu_idle":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: no data-path collective)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(backend: str):
    import torch.distributed as dist
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, device) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def aggregate(bytes_per_step: float, steps: int, local_ms_total: float, world: int, device):
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    t = reduce_max(local_ms_total, device)
    return bytes_per_step * steps * world / (t * 1e-3), t


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------
def host_us_per_call(call, n=200):
    """Median CPU time, in microseconds, of enqueueing one call (host-side
    argument checks, tensor-map encoding, kernel launches), measured call by
    call without synchronising; the caller synchronises afterwards."""
    ts = []
    for _ in range(n):
        t0 = time.perf_counter()
        call()
        ts.append(time.perf_counter() - t0)
    return round(float(np.median(ts)) * 1e6, 2)


def sub_batch(inp, n):
    """The first n sequences of a workload (same pool)."""
    return synth.PagedInputs(np.ascontiguousarray(inp.query[:n]), inp.key_pages,
                             inp.value_pages, np.ascontiguousarray(inp.block_table[:n]),
                             np.ascontiguousarray(inp.context_lens[:n]), inp.page_size,
                             inp.scale, inp.causal, inp.dtype, inp.name)


def time_oracle(inp, target_s: float, unit_fn, mask_fn=None):
    """Runs the oracle on growing leading sub-batches until one run takes
    about target_s; returns (units/s, seconds, description, threads).
    mask_fn(n), if given, returns the additive mask of the first n sequences."""
    import oracle
    lib = oracle.load()
    cores = oracle.host_cores()
    n = 1
    while True:
        sub = sub_batch(inp, n)
        m = mask_fn(n) if mask_fn else None
        t0 = time.perf_counter()
        lib.paged_attention(sub.query, sub.key_pages, sub.value_pages, sub.block_table,
                            sub.context_lens, sub.scale, sub.causal, num_threads=cores, mask=m)
        dt = time.perf_counter() - t0
        if dt >= target_s or n >= inp.B:
            break
        grow = max(2, int(math.ceil(target_s / max(dt, 1e-3) * 0.9)))
        n = min(inp.B, n * grow)
    if dt >= target_s:
        return unit_fn(sub) / dt, dt, f"first {n} of {inp.B} sequences, one full oracle call", cores
    # the whole batch takes less than target_s: repeat it
    reps = max(1, int(math.ceil(target_s / max(dt, 1e-3))))
    t0 = time.perf_counter()
    for _ in range(reps):
        lib.paged_attention(sub.query, sub.key_pages, sub.value_pages, sub.block_table,
                            sub.context_lens, sub.scale, sub.causal, num_threads=cores, mask=m)
    dt = time.perf_counter() - t0
    return (unit_fn(sub) * reps / dt, dt,
            f"all {inp.B} sequences, {reps} full oracle calls", cores)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    """Our arm: the requested workload's line; on the default decode line, a
    `prefill` record of the causal prefill workload measured the same way in
    the same run (the metric's second half)."""
    import copy

    import torch
    from paged_kv_cache_03_gb300 import binding as B
    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist_init("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    B.load()
    line = measure(args, device, world, rank)
    if headline(args) and not args.no_prefill:
        pargs = copy.copy(args)
        pargs.workload = "prefill"
        sub = measure(pargs, device, world, rank)
        line["prefill"] = prefill_record(sub)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return line


def headline(args) -> bool:
    """The default line (the decode workload as the library runs it), which
    carries the causal prefill record beside it."""
    return (args.workload == "decode" and args.op == "attention" and args.schedule == "auto"
            and not args.mask and not args.no_causal)


PREFILL_KEYS = ("metric", "value", "unit", "ms_per_step", "steps", "warmup", "dtype",
                "clocks", "e2e", "gpu_launches", "roofline", "cpu_baseline", "step_ms_median",
                "wall_s_timed_region", "host_us_per_call")


def prefill_record(sub) -> dict:
    rec = {k: sub[k] for k in PREFILL_KEYS if k in sub}
    rec["metric"] = "causal prefill TFLOP/s (4 * H_q * D * visible pairs / device time)"
    rec["config"] = sub["config"]
    return rec


def measure(args, device, world, rank):
    """One workload: warm-up, K timed steps (two passes), e2e, cpu baseline;
    returns the JSON line (rank 0's cpu baseline only)."""
    import torch
    from paged_kv_cache_03_gb300 import binding as B

    inp = bench_inputs(args)
    bytes_step = algorithmic_bytes(inp) + (mask_bytes(inp) if args.mask else 0)
    flops_step = algorithmic_flops(inp)
    bound = roofline_bound(bytes_step, flops_step, load_peaks()[0])
    es = 2 if inp.dtype == "bf16" else 4
    tdt = torch.bfloat16 if inp.dtype == "bf16" else torch.float32

    def dev_tensor(a, dt=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if dt is not None:
            t = t.view(dt)
        return t.to(device)

    q = dev_tensor(inp.query, tdt)
    kp = dev_tensor(inp.key_pages, tdt)
    vp = dev_tensor(inp.value_pages, tdt)
    bt = dev_tensor(inp.block_table)
    ctx = dev_tensor(inp.context_lens)
    out = torch.empty_like(q)
    shape = B.shape_of(q, kp, bt)
    sched = {"auto": B.pa_choose_schedule(shape), "decode": B.PA_SCHED_DECODE,
             "prefill": B.PA_SCHED_PREFILL}[args.schedule]
    launches = B.pa_launch_count(shape, sched)
    ws = B.new_workspace(shape, device)
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    dominant = {B.PA_SCHED_DECODE: "decode_split_kernel",
                B.PA_SCHED_PREFILL: "prefill_tile_kernel"}[sched]
    mask = None
    if args.mask:
        mask = synth.additive_mask_device(inp.B * inp.H_q, inp.L, mask_width(inp), 4343, device)
        torch.cuda.empty_cache()  # the draw's temporaries

    def call(ev0=None, ev1=None):
        if mask is None:
            st = B.pa_paged_attention_profiled(
                shape, q, kp, vp, bt, ctx, inp.scale, inp.causal, out, ws, ws.numel(), stream,
                sched, ev0.cuda_event if ev0 is not None else None,
                ev1.cuda_event if ev1 is not None else None)
        else:  # the masked entry has no kernel events: the whole call is timed
            if ev0 is not None:
                ev0.record(stream)
            st = B.pa_paged_attention_masked(shape, q, kp, vp, bt, ctx, inp.scale, inp.causal,
                                             mask, mask.shape[2], out, ws, ws.numel(), stream,
                                             sched)
            if ev1 is not None:
                ev1.record(stream)
        if st != B.PA_OK:
            raise RuntimeError(f"pa_paged_attention: {B.status_str(st)}")

    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize(device)
    st, flag = B.pa_check_device_flag(ws, stream=stream)
    if flag:
        raise RuntimeError(f"device flag {flag:#x} after warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for e in ev:  # create the CUDA events up front (torch makes them on first record)
        for x in e:
            x.record(stream)
    torch.cuda.synchronize(device)

    sampler = ClockSampler(device.index)
    if rank == 0:
        sampler.start()
    barrier(device)
    torch.cuda.synchronize(device)
    wall0 = time.perf_counter()
    # Pass 1, the step: the call exactly as a user makes it.  (Events recorded
    # inside the call would sit between its kernels and stop the combine from
    # starting early: 7 us of a 125 us decode step.)
    for k in range(K):
        flush.zero_()  # L2 flush between timed steps (outside the step's events)
        e = ev[k]
        e[0].record(stream)
        call()
        e[3].record(stream)
    # Pass 2, the dominant kernel: the same K calls with events around it.
    for k in range(K):
        flush.zero_()
        call(ev[k][1], ev[k][2])
    torch.cuda.synchronize(device)
    barrier(device)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if rank == 0 else None
    step_ms = np.array([e[0].elapsed_time(e[3]) for e in ev])
    kern_ms = np.array([e[1].elapsed_time(e[2]) for e in ev])
    st, flag = B.pa_check_device_flag(ws, stream=stream)
    if flag:
        raise RuntimeError(f"device flag {flag:#x} after timed steps")
    host_us = host_us_per_call(call)
    torch.cuda.synchronize(device)

    value, t_max = aggregate(bytes_step, K, float(step_ms.sum()), world, device)
    ms_per_step = t_max / K
    if bound == "tensor":
        value_unit, value = "TFLOP/s", flops_step * K * world / (t_max * 1e-3) / 1e12
    else:
        value_unit, value = "GB/s", value / 1e9

    peaks, peaks_src = load_peaks()
    kern_avg_s = float(kern_ms.mean()) * 1e-3
    if bound == "tensor":
        achieved = flops_step / kern_avg_s / 1e12
        peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        runit = "TFLOP/s"
    else:
        achieved = bytes_step / kern_avg_s / 1e9
        peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        runit = "GB/s"
    nominal = NOMINAL_PEAKS["bf16_tflops" if bound == "tensor" else "hbm_gbs"]
    roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": runit,
                "frac": round(achieved / peak, 4), "nominal_peak": nominal,
                "frac_nominal": round(achieved / nominal, 4),
                "call_ms_avg": round(float(step_ms.mean()), 5),
                "traffic": recorded_traffic(dominant, variant(args)),
                "kernel": dominant + (" (whole call)" if mask is not None and launches > 1
                                      else ""),
                "kernel_ms_avg": round(float(kern_ms.mean()), 5),
                "kernel_ms_median": round(float(np.median(kern_ms)), 5),
                "peak_source": f"{peaks_src} (MEASURED_PEAKS.json)" if peaks_src == "measured"
                else "fallback", "algorithmic_bytes": bytes_step,
                "algorithmic_flops": flops_step}

    # ---- end to end through the public call with host buffers ----------------
    e2e = None
    if not args.no_e2e:
        host = {n: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
                for n, a in (("query", inp.query), ("key_pages", inp.key_pages),
                             ("value_pages", inp.value_pages), ("block_table", inp.block_table),
                             ("context_lens", inp.context_lens))}
        out_host = torch.empty(out.shape, dtype=tdt).pin_memory()
        dst = {"query": q, "key_pages": kp, "value_pages": vp, "block_table": bt,
               "context_lens": ctx}
        if mask is not None:
            host["mask"] = mask.cpu().pin_memory()
            dst["mask"] = mask
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out.numel() * out.element_size()
        Ke = max(3, min(args.e2e_steps, K))

        def e2e_step():
            for n, t in host.items():
                d = dst[n]
                d.view(torch.uint8).view(-1).copy_(t.view(torch.uint8).view(-1),
                                                   non_blocking=True)
            if mask is None:
                st = B.pa_paged_attention(shape, q, kp, vp, bt, ctx, inp.scale, inp.causal, out,
                                          ws, ws.numel(), stream)
            else:
                st = B.pa_paged_attention_masked(shape, q, kp, vp, bt, ctx, inp.scale,
                                                 inp.causal, mask, mask.shape[2], out, ws,
                                                 ws.numel(), stream)
            if st != B.PA_OK:
                raise RuntimeError(B.status_str(st))
            out_host.copy_(out, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(device)
        barrier(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(Ke):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(device)
        e2e_ms = a.elapsed_time(b)
        e2e_ms = reduce_max(e2e_ms, device)
        if bound == "tensor":
            ev_ = flops_step * Ke * world / (e2e_ms * 1e-3) / 1e12
        else:
            ev_ = bytes_step * Ke * world / (e2e_ms * 1e-3) / 1e9
        e2e = {"value": round(ev_, 3), "unit": value_unit, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": Ke,
               "ms_per_step": round(e2e_ms / Ke, 4),
               "note": "pinned host inputs (query, both page pools, block table, context "
                       "lengths" + (", mask" if mask is not None else "") + ") copied to HBM, "
                       "one call, output copied back, every step"}

    line = {
        "metric": METRIC_MASKED if mask is not None else METRIC, "value": round(value, 3),
        "unit": value_unit, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": inp.dtype,
        "data": "synthetic (seeded N(0,1) bf16, scattered pages)",
        "config": {"workload": workload_desc(args.workload, inp), "schedule":
                   {1: "decode", 2: "prefill"}[sched],
                   "l2": "flushed: 256 MiB write between timed steps (outside step events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "algorithmic_bytes_per_step": bytes_step,
                   "algorithmic_flops_per_step": flops_step,
                   **({"mask": f"fp32 [B*H_q, L, {mask.shape[2]}], N(0,1) biases, 1/3 -inf, "
                               f"seed 4343 (device draw); {mask_bytes(inp)} visible bytes"}
                      if mask is not None else {})},
        "clocks": clocks, "e2e": e2e, "gpu_launches": 2 * K * launches, "roofline": roofline,
        "timing": "steps: K calls as a user makes them; kernel: a second pass of K calls "
                  "with events around the dominant kernel, same timed region",
        "step_ms_median": round(float(np.median(step_ms)), 5),
        "wall_s_timed_region": round(wall, 3),
        "host_us_per_call": host_us,
    }
    if rank == 0 and not args.no_cpu_baseline:
        unit_fn = (lambda s: algorithmic_flops(s) / 1e12) if bound == "tensor" else (
            lambda s: algorithmic_bytes(s) / 1e9)
        mask_fn = None
        if mask is not None:
            unit_fn = lambda s: (algorithmic_bytes(s) + mask_bytes(s)) / 1e9  # noqa: E731
            mask_fn = lambda n: mask[:n * inp.H_q].cpu().numpy()  # noqa: E731
        v, secs, desc, cores = time_oracle(inp, args.cpu_seconds, unit_fn, mask_fn)
        line["cpu_baseline"] = {"value": round(v, 6), "unit": value_unit, "cores": cores,
                                "kind": "oracle", "sample": desc, "seconds": round(secs, 3)}
    return line


def ragged_sub_batch(r, n):
    """The first n sequences of a ragged batch (same pool)."""
    cu = r.cu_q[:n + 1]
    return synth.RaggedInputs(np.ascontiguousarray(r.query[:int(cu[-1])]), r.key_pages,
                              r.value_pages, np.ascontiguousarray(r.block_table[:n]),
                              np.ascontiguousarray(r.context_lens[:n]), np.ascontiguousarray(cu),
                              r.page_size, r.scale, r.causal, r.dtype, r.name)


def ragged_desc(r) -> str:
    lens = r.q_lens
    n_dec = int((lens == 1).sum())
    chunks = sorted(set(int(x) for x in lens if x > 1))
    return (f"mixed: B={r.B} ({n_dec} decodes L=1 ctx~U[128,4096], {r.B - n_dec} prefill chunks "
            f"L={chunks} ctx~U[128,2048]) total_q={int(r.cu_q[-1])} H_q={r.H_q} H_kv={r.H_kv} "
            f"D={r.D} page_size={r.page_size} pool={r.num_pages} pages, causal, seed=6")


def run_mixed(args):
    """One step = one pa_paged_attention_varlen call over the continuous-
    batching step (the device routes decodes to the page walk and chunks to
    the tensor-core tiles)."""
    import torch
    from paged_kv_cache_03_gb300 import binding as B
    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist_init("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    B.load()
    r = synth.mixed_workload()
    bytes_step, flops_step = ragged_bytes(r), ragged_flops(r)

    def dev_tensor(a, dt=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(dt) if dt is not None else t).to(device)

    q = dev_tensor(r.query, torch.bfloat16)
    kp, vp = dev_tensor(r.key_pages, torch.bfloat16), dev_tensor(r.value_pages, torch.bfloat16)
    bt, ctx, cu = dev_tensor(r.block_table), dev_tensor(r.context_lens), dev_tensor(r.cu_q)
    out = torch.empty_like(q)
    shape = B.shape_of_varlen(q, kp, bt, r.max_L)
    ws = B.new_workspace(shape, device)
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    T = int(r.cu_q[-1])
    sched = {"auto": B.PA_SCHED_AUTO, "decode": B.PA_SCHED_DECODE,
             "prefill": B.PA_SCHED_PREFILL}[args.schedule]

    def call():
        st = B.pa_paged_attention_varlen(shape, q, kp, vp, bt, ctx, cu, T, r.scale, r.causal, out,
                                         ws, ws.numel(), stream, sched)
        if st != B.PA_OK:
            raise RuntimeError(f"pa_paged_attention_varlen: {B.status_str(st)}")

    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize(device)
    _, flag = B.pa_check_device_flag(ws, stream=stream)
    if flag:
        raise RuntimeError(f"device flag {flag:#x} after warm-up")
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for e in ev:
        for x in e:
            x.record(stream)
    torch.cuda.synchronize(device)
    sampler = ClockSampler(device.index)
    if rank == 0:
        sampler.start()
    barrier(device)
    torch.cuda.synchronize(device)
    for k in range(K):
        flush.zero_()
        ev[k][0].record(stream)
        call()
        ev[k][1].record(stream)
    torch.cuda.synchronize(device)
    barrier(device)
    clocks = sampler.stop() if rank == 0 else None
    step_ms = np.array([e[0].elapsed_time(e[1]) for e in ev])
    _, flag = B.pa_check_device_flag(ws, stream=stream)
    if flag:
        raise RuntimeError(f"device flag {flag:#x} after timed steps")
    host_us = host_us_per_call(call)
    torch.cuda.synchronize(device)
    value, t_max = aggregate(bytes_step, K, float(step_ms.sum()), world, device)
    peaks, peaks_src = load_peaks()
    achieved = bytes_step / (float(step_ms.mean()) * 1e-3) / 1e9
    peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    # pair plan + tile kernel, page walk + combine, or both pairs
    launches = {"auto": 4, "decode": 2, "prefill": 2}[args.schedule]
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "nominal_peak": NOMINAL_PEAKS["hbm_gbs"],
                "frac_nominal": round(achieved / NOMINAL_PEAKS["hbm_gbs"], 4), "traffic": None,
                "kernel": {"auto": "whole call (pair_plan + prefill_tile + decode_split + "
                                   "decode_combine)",
                           "decode": "whole call (decode_split + decode_combine)",
                           "prefill": "whole call (pair_plan + prefill_tile)"}[args.schedule],
                "kernel_ms_avg": round(float(step_ms.mean()), 5),
                "kernel_ms_median": round(float(np.median(step_ms)), 5),
                "peak_source": f"{peaks_src} (MEASURED_PEAKS.json)" if peaks_src == "measured"
                else "fallback", "algorithmic_bytes": bytes_step,
                "algorithmic_flops": flops_step,
                "tensor_floor_ms": round(flops_step / (peaks.get(
                    "bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]) * 1e12) * 1e3, 5)}
    e2e = None
    if not args.no_e2e:
        host = {n: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
                for n, a in (("q", r.query), ("kp", r.key_pages), ("vp", r.value_pages),
                             ("bt", r.block_table), ("ctx", r.context_lens), ("cu", r.cu_q))}
        dst = {"q": q, "kp": kp, "vp": vp, "bt": bt, "ctx": ctx, "cu": cu}
        out_host = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out.numel() * out.element_size()
        Ke = max(3, min(args.e2e_steps, K))

        def e2e_step():
            for n, t in host.items():
                dst[n].view(torch.uint8).view(-1).copy_(t.view(torch.uint8).view(-1),
                                                        non_blocking=True)
            call()
            out_host.copy_(out, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(device)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(Ke):
            e2e_step()
        b_.record(stream)
        torch.cuda.synchronize(device)
        e2e_ms = reduce_max(a.elapsed_time(b_), device)
        e2e = {"value": round(bytes_step * Ke * world / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": Ke,
               "ms_per_step": round(e2e_ms / Ke, 4),
               "note": "pinned host query, pools, block table, context lengths and offsets "
                       "copied to HBM, one call, output copied back, every step"}
    line = {
        "metric": METRIC_MIXED, "value": round(value / 1e9, 3), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(t_max / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": r.dtype,
        "data": "synthetic (seeded N(0,1) bf16, scattered pages)",
        "config": {"workload": ragged_desc(r), "schedule": args.schedule,
                   "l2": "flushed: 256 MiB write between timed steps (outside step events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "algorithmic_bytes_per_step": bytes_step,
                   "algorithmic_flops_per_step": flops_step},
        "clocks": clocks, "e2e": e2e, "gpu_launches": K * launches, "roofline": roofline,
        "host_us_per_call": host_us,
    }
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        lib = oracle.load()
        cores = oracle.host_cores()
        n, dt = 1, 0.0
        while True:
            sub = ragged_sub_batch(r, n)
            t0 = time.perf_counter()
            lib.paged_attention_varlen(sub.query, sub.key_pages, sub.value_pages, sub.block_table,
                                       sub.context_lens, sub.cu_q, sub.scale, sub.causal,
                                       num_threads=cores)
            dt = time.perf_counter() - t0
            if dt >= args.cpu_seconds or n >= r.B:
                break
            n = min(r.B, max(n + 1, int(n * args.cpu_seconds / max(dt, 1e-3) * 0.9)))
        reps, desc = 1, f"first {n} of {r.B} sequences, one oracle call"
        if dt < args.cpu_seconds:  # the whole batch is quicker: repeat it
            reps = max(1, int(math.ceil(args.cpu_seconds / max(dt, 1e-3))))
            t0 = time.perf_counter()
            for _ in range(reps):
                lib.paged_attention_varlen(sub.query, sub.key_pages, sub.value_pages,
                                           sub.block_table, sub.context_lens, sub.cu_q, sub.scale,
                                           sub.causal, num_threads=cores)
            dt = time.perf_counter() - t0
            desc = f"all {r.B} sequences, {reps} oracle calls"
        line["cpu_baseline"] = {"value": round(ragged_bytes(sub) * reps / dt / 1e9, 6),
                                "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": round(dt, 3)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return line


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------
def run_append(args):
    """One step = one pa_append_kv call storing the workload's L new tokens
    per sequence (seeded N(0,1) rows) in their pages."""
    import torch
    from paged_kv_cache_03_gb300 import binding as B
    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist_init("nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    B.load()
    inp = synth.workload(args.workload)
    kn_np, vn_np = synth.new_kv(inp.B, inp.H_kv, inp.L, inp.D, 4242, inp.dtype)
    tdt = torch.bfloat16 if inp.dtype == "bf16" else torch.float32

    def dev_tensor(a, dt=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(dt) if dt is not None else t).to(device)

    kn, vn = dev_tensor(kn_np, tdt), dev_tensor(vn_np, tdt)
    kp, vp = dev_tensor(inp.key_pages, tdt), dev_tensor(inp.value_pages, tdt)
    bt, ctx = dev_tensor(inp.block_table), dev_tensor(inp.context_lens)
    shape = B.make_shape(inp.B, inp.H_kv, inp.H_kv, inp.L, inp.D, inp.num_pages, inp.page_size,
                         inp.block_table.shape[1], B.PA_BF16 if inp.dtype == "bf16" else B.PA_F32)
    ws = torch.zeros(256, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    bytes_step = append_bytes(inp)

    def call():
        st = B.pa_append_kv(shape, kn, vn, kp, vp, bt, ctx, ws, ws.numel(), stream)
        if st != B.PA_OK:
            raise RuntimeError(f"pa_append_kv: {B.status_str(st)}")

    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize(device)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for e in ev:
        for x in e:
            x.record(stream)
    torch.cuda.synchronize(device)
    sampler = ClockSampler(device.index)
    if rank == 0:
        sampler.start()
    barrier(device)
    torch.cuda.synchronize(device)
    for k in range(K):
        flush.zero_()
        ev[k][0].record(stream)
        call()
        ev[k][1].record(stream)
    torch.cuda.synchronize(device)
    barrier(device)
    clocks = sampler.stop() if rank == 0 else None
    step_ms = np.array([e[0].elapsed_time(e[1]) for e in ev])
    _, flag = B.pa_check_device_flag(ws, stream=stream)
    if flag:
        raise RuntimeError(f"device flag {flag:#x} after timed steps")
    host_us = host_us_per_call(call)
    torch.cuda.synchronize(device)
    value, t_max = aggregate(bytes_step, K, float(step_ms.sum()), world, device)
    peaks, peaks_src = load_peaks()
    achieved = bytes_step / (float(step_ms.mean()) * 1e-3) / 1e9
    peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "nominal_peak": NOMINAL_PEAKS["hbm_gbs"],
                "frac_nominal": round(achieved / NOMINAL_PEAKS["hbm_gbs"], 4),
                "traffic": recorded_traffic("append_kv_kernel", args.workload),
                "kernel": "append_kv_kernel", "kernel_ms_avg": round(float(step_ms.mean()), 5),
                "peak_source": f"{peaks_src} (MEASURED_PEAKS.json)" if peaks_src == "measured"
                else "fallback", "algorithmic_bytes": bytes_step}
    e2e = None
    if not args.no_e2e:
        host = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
                for a in (kn_np, vn_np, inp.block_table, inp.context_lens)]
        dsts = [kn, vn, bt, ctx]
        flag_host = torch.empty(1, dtype=torch.int32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host)
        Ke = max(3, min(args.e2e_steps, K))

        def e2e_step():
            for h, d in zip(host, dsts):
                d.view(torch.uint8).view(-1).copy_(h.view(torch.uint8).view(-1), non_blocking=True)
            call()
            flag_host.copy_(ws[:4].view(torch.int32), non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(Ke):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(device)
        e2e_ms = reduce_max(a.elapsed_time(b), device)
        e2e = {"value": round(bytes_step * Ke * world / (e2e_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 4, "steps": Ke,
               "ms_per_step": round(e2e_ms / Ke, 4),
               "note": "pinned host new rows, block table and context lengths copied to HBM, "
                       "one call, flag word copied back, every step (the pools stay in HBM)"}
    line = {
        "metric": "paged K/V append HBM GB/s (bf16, d128)", "value": round(value / 1e9, 3),
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(t_max / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": inp.dtype,
        "data": "synthetic (seeded N(0,1) new rows, scattered pages)",
        "config": {"workload": "append of the new tokens of " + workload_desc(args.workload, inp),
                   "l2": "flushed: 256 MiB write between timed steps (outside step events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "algorithmic_bytes_per_step": bytes_step},
        "clocks": clocks, "e2e": e2e, "gpu_launches": K, "roofline": roofline,
    }
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        lib = oracle.load()
        reps, t0 = 0, time.perf_counter()
        while True:
            lib.append_kv(kn_np, vn_np, inp.key_pages, inp.value_pages, inp.block_table,
                          inp.context_lens)
            reps += 1
            if time.perf_counter() - t0 > min(args.cpu_seconds, 10.0):
                break
        secs = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": round(bytes_step * reps / secs / 1e9, 6), "unit": "GB/s",
                                "cores": 1, "kind": "oracle",
                                "sample": f"{reps} whole appends (includes the oracle's copy "
                                          "of both pools)", "seconds": round(secs, 3)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return line


def run_reference(args):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return None
    import oracle
    lib = oracle.load()
    cores = oracle.host_cores()
    inp = bench_inputs(args)
    bound = roofline_bound(algorithmic_bytes(inp), algorithmic_flops(inp), load_peaks()[0])
    unit_fn = (lambda s: algorithmic_flops(s) / 1e12) if bound == "tensor" else (
        lambda s: algorithmic_bytes(s) / 1e9)
    unit = "TFLOP/s" if bound == "tensor" else "GB/s"
    # size each step so the whole run takes about args.ref_budget seconds
    per_step = max(0.05, min(3.0, args.ref_budget / max(1, args.steps + args.warmup)))
    _, _, _, _ = time_oracle(inp, min(per_step, 0.5), unit_fn)  # warm the library
    n = 1
    while n < inp.B:
        sub = sub_batch(inp, n)
        t0 = time.perf_counter()
        lib.paged_attention(sub.query, sub.key_pages, sub.value_pages, sub.block_table,
                            sub.context_lens, sub.scale, sub.causal, num_threads=cores)
        dt = time.perf_counter() - t0
        if dt >= per_step:
            break
        n = min(inp.B, max(n + 1, int(n * per_step / max(dt, 1e-4) * 0.9)))
    sub = sub_batch(inp, n)

    def step():
        lib.paged_attention(sub.query, sub.key_pages, sub.value_pages, sub.block_table,
                            sub.context_lens, sub.scale, sub.causal, num_threads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    v = unit_fn(sub) * args.steps / dt
    desc = f"first {n} of {inp.B} sequences per step, one full oracle call"
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16, scattered pages)",
            "config": {"workload": workload_desc(args.workload, inp), "sample": desc},
            "cpu_baseline": {"value": round(v, 6), "unit": unit, "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(v, 6), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    if headline(args) and not args.no_prefill:
        # the causal prefill beside it, on a bounded leading sample
        pinp = synth.workload("prefill")
        pv, secs, pdesc, _ = time_oracle(pinp, args.cpu_seconds,
                                         lambda s: algorithmic_flops(s) / 1e12)
        line["prefill"] = {
            "metric": "causal prefill TFLOP/s (4 * H_q * D * visible pairs / device time)",
            "value": round(pv, 6), "unit": "TFLOP/s", "seconds": round(secs, 3),
            "config": {"workload": workload_desc("prefill", pinp), "sample": pdesc},
            "cpu_baseline": {"value": round(pv, 6), "unit": "TFLOP/s", "cores": cores,
                             "kind": "oracle", "sample": pdesc},
            "e2e": {"value": round(pv, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return line


def run_mixed_reference(args):
    """--impl reference for the ragged step: the oracle on the host cores, a
    bounded leading sub-batch per step."""
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return None
    import oracle
    lib = oracle.load()
    cores = oracle.host_cores()
    r = synth.mixed_workload()
    per_step = max(0.05, min(3.0, args.ref_budget / max(1, args.steps + args.warmup)))
    n = 1
    while n < r.B:
        sub = ragged_sub_batch(r, n)
        t0 = time.perf_counter()
        lib.paged_attention_varlen(sub.query, sub.key_pages, sub.value_pages, sub.block_table,
                                   sub.context_lens, sub.cu_q, sub.scale, sub.causal,
                                   num_threads=cores)
        dt = time.perf_counter() - t0
        if dt >= per_step:
            break
        n = min(r.B, max(n + 1, int(n * per_step / max(dt, 1e-4) * 0.9)))
    sub = ragged_sub_batch(r, n)

    def step():
        lib.paged_attention_varlen(sub.query, sub.key_pages, sub.value_pages, sub.block_table,
                                   sub.context_lens, sub.cu_q, sub.scale, sub.causal,
                                   num_threads=cores)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    v = ragged_bytes(sub) / 1e9 * args.steps / dt
    desc = f"first {n} of {r.B} sequences per step, one full oracle call"
    line = {"impl": "reference", "metric": METRIC_MIXED, "value": round(v, 6), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16, scattered pages)",
            "config": {"workload": ragged_desc(r), "sample": desc},
            "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return line


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(synth.WORKLOADS) + ["mixed"], default="decode",
                    help="mixed: a ragged continuous-batching step (decodes + prefill chunks)")
    ap.add_argument("--op", choices=["attention", "append"], default="attention",
                    help="the path (paged attention) or the K/V append before it")
    ap.add_argument("--schedule", choices=["auto", "decode", "prefill"], default="auto",
                    help="force a schedule (auto: the library's choice)")
    ap.add_argument("--no-causal", action="store_true",
                    help="every key of the context visible (mask=None) instead of causal")
    ap.add_argument("--mask", action="store_true",
                    help="add a seeded fp32 additive mask to every call (attention only)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-prefill", action="store_true",
                    help="leave the causal prefill record out of the default decode line")
    ap.add_argument("--ref-budget", type=float, default=90.0,
                    help="seconds the reference arm's timed steps should take in total")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.op == "append":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the append's reference arm is its oracle: see cpu_baseline"}))
            return None
        return run_append(args)
    if args.workload == "mixed":
        if args.op != "attention" or args.mask or args.no_causal:
            ap.error("--workload mixed takes neither --op append, --mask nor --no-causal")
        return run_mixed_reference(args) if args.impl == "reference" else run_mixed(args)
    if args.impl == "reference":
        if args.mask:
            print(json.dumps({"impl": "reference", "unavailable":
                              "the masked arm's reference is its oracle: see cpu_baseline"}))
            return None
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    main()
