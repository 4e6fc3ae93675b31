"""bench.py's host logic on CPU: the algorithmic byte and FLOP counts its
roofline divides by, and the reference arm (the oracle on the host cores)
for the uniform and the ragged workloads."""
import json
import os
import subprocess
import sys

import numpy as np

import bench
from paged_kv_cache_03_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def brute_visible_pairs(L, S, causal):
    """(row, key) pairs with the key visible, counted one by one."""
    return sum(1 for l in range(L) for s in range(S) if (not causal or s <= l + S - L))


def test_visible_pairs_matches_counting():
    for L, ctx, causal in ((5, [13, 40], True), (1, [7, 300], True), (4, [4, 9], False),
                           (65, [65, 100, 1000], True)):
        inp = synth.generate(len(ctx), 4, 2, L, 128, 16, context_lens=ctx, causal=causal, seed=1)
        want = sum(brute_visible_pairs(L, int(S), causal) for S in ctx)
        assert bench.visible_pairs(inp) == want


def test_flops_and_mask_bytes_follow_visible_pairs():
    inp = synth.workload("tiny")
    vp = bench.visible_pairs(inp)
    assert bench.algorithmic_flops(inp) == 4 * inp.H_q * inp.D * vp
    assert bench.mask_bytes(inp) == 4 * inp.H_q * vp


def test_algorithmic_bytes_counts_each_visible_kv_row_once():
    inp = synth.workload("tiny")  # contexts 13 and 40, page 16, bf16
    kv = 2 * inp.H_kv * inp.D * 2 * (13 + 40)
    qo = 2 * inp.query.size * 2
    pages = 1 + 3
    assert bench.algorithmic_bytes(inp) == kv + qo + 4 * pages + 4 * inp.B


def test_ragged_counts_reduce_to_the_uniform_counts():
    """A ragged batch of equal query counts moves the same bytes as the
    uniform batch (plus its offsets) and does the same FLOPs."""
    u = synth.generate(3, 8, 2, 6, 128, 16, context_lens=[6, 50, 300], seed=3)
    r = synth.RaggedInputs(np.ascontiguousarray(u.query.transpose(0, 2, 1, 3).reshape(-1, 8, 128)),
                           u.key_pages, u.value_pages, u.block_table, u.context_lens,
                           np.arange(0, 19, 6, dtype=np.int32), u.page_size, u.scale, u.causal,
                           u.dtype, "uniform-as-ragged")
    assert bench.ragged_flops(r) == bench.algorithmic_flops(u)
    assert bench.ragged_bytes(r) == bench.algorithmic_bytes(u) + 4 * (u.B + 1)


def test_ragged_counts_skip_sequences_without_queries():
    r = synth.generate_ragged(8, 2, 128, 16, [2, 0, 3], [10, 500, 20], seed=4)
    kv = 2 * r.H_kv * r.D * 2 * (10 + 20)
    qo = 2 * r.query.size * 2
    pages = 1 + 2
    assert bench.ragged_bytes(r) == kv + qo + 4 * pages + 4 * r.B + 4 * (r.B + 1)
    want = sum(brute_visible_pairs(L, S, True) for L, S in ((2, 10), (3, 20)))
    assert bench.ragged_flops(r) == 4 * r.H_q * r.D * want


def test_append_bytes():
    inp = synth.workload("tails")
    rows = inp.B * inp.H_kv * inp.L * inp.D * 2
    assert bench.append_bytes(inp) >= 4 * rows
    assert bench.append_bytes(inp) < 4 * rows + 4 * inp.B * (inp.L // inp.page_size + 3)


def _run_bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_reference_arm_runs_the_oracle():
    line = _run_bench("--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup",
                      "3", "--ref-budget", "2")
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["gpu_launches"] == 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_of_the_ragged_step():
    line = _run_bench("--impl", "reference", "--workload", "mixed", "--steps", "3", "--warmup",
                      "3", "--ref-budget", "2")
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["config"]["workload"].startswith("mixed")


def test_reference_arm_default_line_carries_the_prefill_record():
    """The default (decode) line of the reference arm carries the causal
    prefill workload's oracle rate beside it, in TFLOP/s."""
    line = _run_bench("--impl", "reference", "--steps", "3", "--warmup", "3", "--ref-budget",
                      "2", "--cpu-seconds", "0.5")
    assert line["unit"] == "GB/s" and line["config"]["workload"].startswith("decode")
    pre = line["prefill"]
    assert pre["unit"] == "TFLOP/s" and pre["value"] > 0
    assert pre["config"]["workload"].startswith("prefill")
    assert pre["cpu_baseline"]["kind"] == "oracle"


def test_headline_rule():
    import argparse
    base = dict(workload="decode", op="attention", schedule="auto", mask=False,
                no_causal=False)
    assert bench.headline(argparse.Namespace(**base))
    for k, v in (("workload", "prefill"), ("mask", True), ("schedule", "decode"),
                 ("no_causal", True), ("op", "append")):
        assert not bench.headline(argparse.Namespace(**{**base, k: v}))


def test_recorded_traffic_follows_the_code_not_the_comments():
    """The digest that keeps profiles/traffic.json tied to the kernels it was
    measured on ignores comments and blank lines, and nothing else."""
    src = "int f(int x) {\n    return x + 1;  // one more\n}\n"
    assert bench._code_only(src) == bench._code_only(
        "/* a new header\n   comment */\nint f(int x) {\n\n    return x + 1;\n}  // end\n")
    assert bench._code_only(src) != bench._code_only(src.replace("x + 1", "x + 2"))
    # a recorded entry whose digest no longer matches is not reported
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        recorded = json.load(f)
    key = next(iter(recorded))
    kernel, workload = key.split("@")
    stale = recorded[key]["source_digest"] != bench.kernel_source_digest(kernel)
    assert (bench.recorded_traffic(kernel, workload) is None) == stale
