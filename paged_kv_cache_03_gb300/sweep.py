#!/usr/bin/env python3
"""Operator sweep: times both schedules over a grid of shapes.

For every (GQA group G, query positions L, context length S) of the grid it
runs the decode schedule (split-S page walk on CUDA cores + combine) and the
prefill schedule (tcgen05 tensor-core tiles), each forced through the C ABI
on the same seeded inputs, and reports the device time of one call (median
of CUDA-event timings, L2 flushed before each call).  The crossover between
the two is what the library's dispatch rule (pa_choose_schedule) encodes.

The grid restates the Week 2 operator grid of "Week 2 Day 5" (contexts up to
256, L in {1, 2, 4, 8}, GQA groups 1 and 4) on paged inputs and extends it to
longer contexts and more query positions, where the schedules trade places.

  python -m paged_kv_cache_03_gb300.sweep [--reps 15] [--json out.jsonl]
  python -m paged_kv_cache_03_gb300.sweep --prefill-scan

Needs a GPU; prints a markdown table.
"""
from __future__ import annotations

import argparse
import json
import statistics
import sys

H_KV = 8
D = 128
PAGE = 128
B = 8
GROUPS = (1, 4)
LS = (1, 2, 4, 8, 16, 32, 64, 128)
SS = (64, 256, 1024, 4096, 16384)


def _inputs(G, L, S, seed, B=B):
    """Seeded device inputs: N(0,1) bf16 query and pool, every sequence of
    length S on a random permutation of the pool's pages."""
    import torch
    g = torch.Generator(device="cuda").manual_seed(seed)
    npg = (S + PAGE - 1) // PAGE
    pool = B * npg
    q = torch.randn(B, G * H_KV, L, D, generator=g, device="cuda").to(torch.bfloat16)
    kp = torch.randn(pool, H_KV, PAGE, D, generator=g, device="cuda").to(torch.bfloat16)
    vp = torch.randn(pool, H_KV, PAGE, D, generator=g, device="cuda").to(torch.bfloat16)
    perm = torch.randperm(pool, generator=g, device="cuda").to(torch.int32)
    bt = perm.view(B, npg).contiguous()
    ctx = torch.full((B,), S, dtype=torch.int32, device="cuda")
    return q, kp, vp, bt, ctx


def _time(call, reps, flush):
    import torch
    for _ in range(3):
        call()
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(ts)


def run(reps=15, json_path=None, groups=GROUPS, ls=LS, ss=SS, batches=(B,)):
    import torch
    from paged_kv_cache_03_gb300 import binding as Bd
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    rows_out = []
    print("| B | G | L | rows G*L | S | decode (us) | prefill (us) | faster | rule picks |")
    print("|---|---|---|---|---|---|---|---|---|")
    seed = 1000
    for nb in batches:
        for G in groups:
            for L in ls:
                for S in ss:
                    if L > S:
                        continue
                    seed += 1
                    q, kp, vp, bt, ctx = _inputs(G, L, S, seed, nb)
                    sh = Bd.shape_of(q, kp, bt)
                    ws = Bd.new_workspace(sh)
                    out = torch.empty_like(q)
                    scale = D ** -0.5
                    t = {}
                    for name, sched in (("decode", Bd.PA_SCHED_DECODE), ("prefill", Bd.PA_SCHED_PREFILL)):
                        def call(sched=sched):
                            st = Bd.pa_paged_attention_sched(sh, q, kp, vp, bt, ctx, scale, True, out,
                                                             ws, ws.numel(), None, sched)
                            if st != Bd.PA_OK:
                                raise Bd.PagedAttentionError(st, "pa_paged_attention_sched")
                        try:
                            t[name] = _time(call, reps, flush)
                        except Bd.PagedAttentionError:
                            t[name] = float("nan")
                    auto = Bd.pa_choose_schedule(sh)
                    picks = {Bd.PA_SCHED_DECODE: "decode", Bd.PA_SCHED_PREFILL: "prefill"}.get(auto, "?")
                    faster = min(t, key=lambda k: t[k] if t[k] == t[k] else float("inf"))
                    rec = {"G": G, "L": L, "rows": G * L, "S": S, "B": nb, "H_kv": H_KV,
                           "decode_us": round(t["decode"], 2), "prefill_us": round(t["prefill"], 2),
                           "faster": faster, "rule": picks}
                    rows_out.append(rec)
                    print(f"| {nb} | {G} | {L} | {G * L} | {S} | {t['decode']:.1f} | {t['prefill']:.1f} "
                          f"| {faster} | {picks} |", flush=True)
                    del q, kp, vp, bt, ctx, ws, out
    if json_path:
        with open(json_path, "w") as f:
            for r in rows_out:
                f.write(json.dumps(r) + "\n")
    return rows_out


# Causal prefills of equal total tokens, from many short sequences to one long
# one (L = context length, GQA group 4): how the tile schedule's fixed cost per
# CTA is amortised by more key tiles per CTA.
SCAN = ((16, 512), (8, 1024), (4, 2048), (2, 4096), (1, 8192), (1, 16384))


def _measured_bf16_tflops():
    import os
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return None


def prefill_scan(reps=15, scan=SCAN):
    """Times the tile schedule on causal prefills with L = context length;
    algorithmic FLOP = 4 * H_q * D per visible (row, key) pair, L (L + 1) / 2
    pairs per sequence and head."""
    import torch
    from paged_kv_cache_03_gb300 import binding as Bd
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    peak = _measured_bf16_tflops()
    print("| B x L | tile schedule (us) | TFLOP/s | of measured bf16 peak |")
    print("|---|---|---|---|")
    G, seed = 4, 2000
    for nb, L in scan:
        seed += 1
        q, kp, vp, bt, ctx = _inputs(G, L, L, seed, nb)
        sh = Bd.shape_of(q, kp, bt)
        ws = Bd.new_workspace(sh)
        out = torch.empty_like(q)

        def call():
            st = Bd.pa_paged_attention_sched(sh, q, kp, vp, bt, ctx, D ** -0.5, True, out, ws,
                                             ws.numel(), None, Bd.PA_SCHED_PREFILL)
            if st != Bd.PA_OK:
                raise Bd.PagedAttentionError(st, "pa_paged_attention_sched")
        us = _time(call, reps, flush)
        flops = 4.0 * nb * G * H_KV * D * L * (L + 1) / 2
        tf = flops / (us * 1e-6) / 1e12
        frac = f"{tf / peak:.3f}" if peak else "n/a"
        print(f"| {nb} x {L} | {us:.1f} | {tf:.0f} | {frac} |", flush=True)
        del q, kp, vp, bt, ctx, ws, out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--reps", type=int, default=15)
    ap.add_argument("--json", default=None)
    ints = lambda x: tuple(int(v) for v in x.split(","))  # noqa: E731
    ap.add_argument("--groups", type=ints, default=GROUPS, help="GQA groups, e.g. 1,4")
    ap.add_argument("--ls", type=ints, default=LS, help="query positions, e.g. 1,2,4")
    ap.add_argument("--ss", type=ints, default=SS, help="context lengths")
    ap.add_argument("--batches", type=ints, default=(B,), help="batch sizes")
    ap.add_argument("--prefill-scan", action="store_true",
                    help="time the tile schedule on causal prefills of equal total tokens")
    a = ap.parse_args(argv)
    if a.prefill_scan:
        prefill_scan(a.reps)
    else:
        run(a.reps, a.json, a.groups, a.ls, a.ss, a.batches)


if __name__ == "__main__":
    sys.exit(main())
