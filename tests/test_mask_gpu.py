"""Explicit additive masks (pa_paged_attention_masked) vs the oracle.

The pages normalise explicit masks to [B * H_q, L, S] and keep the causal
flag next to them ("Week 2 Day 5: Fused Decode Attention", Task 1).  Both
schedules take the mask; each is forced on shapes it supports and compared
element by element with the oracle's masked attention, with biases and a
third of the positions removed (-inf), together with the causal rule and
without it.  Also: a fully masked row outputs 0, a zero mask leaves the page
walk's output bitwise unchanged, the fp32 control, and argument checks.
"""
import dataclasses

import numpy as np
import pytest

import gpu_util as gu
from paged_kv_cache_03_gb300 import binding as B
from paged_kv_cache_03_gb300 import synth

pytestmark = pytest.mark.gpu


def _capacity(inp):
    return inp.block_table.shape[1] * inp.page_size


def _s_mask(inp, extra=0):
    cap = _capacity(inp)
    return (cap + 3) // 4 * 4 + extra


def run_masked(inp, mask, schedule, dev=None):
    import torch
    dev = dev or gu.to_device(inp)
    sh = B.shape_of(dev["query"], dev["key_pages"], dev["block_table"])
    ws = B.new_workspace(sh)
    out = torch.full_like(dev["query"], float("nan"))
    m = torch.from_numpy(np.ascontiguousarray(mask)).cuda()
    st = B.pa_paged_attention_masked(sh, dev["query"], dev["key_pages"], dev["value_pages"],
                                     dev["block_table"], dev["context_lens"], inp.scale,
                                     inp.causal, m, mask.shape[2], out, ws, ws.numel(), None,
                                     schedule)
    assert st == B.PA_OK, B.status_str(st)
    torch.cuda.synchronize()
    st, flag = B.pa_check_device_flag(ws)
    assert flag == 0, hex(flag)
    return out


def _small_cases():
    return [
        synth.workload("tiny"),
        synth.generate(B=3, H_q=8, H_kv=2, L=65, D=128, page_size=128,
                       context_lens=[300, 1000, 65], seed=61, name="tails-small"),
        synth.generate(B=2, H_q=32, H_kv=8, L=1, D=128, page_size=16,
                       context_lens=[700, 129], seed=62, name="decode-small"),
        synth.generate(B=2, H_q=4, H_kv=1, L=200, D=128, page_size=16,
                       context_lens=[200, 513], seed=63, name="ps16-crossing"),
    ]


CASES = [(i, c) for i in range(4) for c in (True, False)]


@pytest.mark.parametrize("sched", ["decode", "prefill"])
@pytest.mark.parametrize("case,causal", CASES, ids=[f"case{i}-{'causal' if c else 'full'}"
                                                    for i, c in CASES])
def test_masked_matches_oracle(oracle_lib, sched, case, causal):
    inp = dataclasses.replace(_small_cases()[case], causal=causal)
    mask = synth.additive_mask(inp.B * inp.H_q, inp.L, _s_mask(inp, 4), 70 + case)
    schedule = B.PA_SCHED_DECODE if sched == "decode" else B.PA_SCHED_PREFILL
    out = run_masked(inp, mask, schedule)
    got = gu.out_to_f64(out)
    ref = oracle_lib.paged_attention(inp.query, inp.key_pages, inp.value_pages,
                                     inp.block_table, inp.context_lens, inp.scale, inp.causal,
                                     mask=mask)
    gu.assert_parity(got, ref, "bf16", f"{inp.name} {sched} masked")


@pytest.mark.parametrize("name", ["decode", "tails"])
def test_masked_workloads_auto(oracle_lib, name):
    """The named workloads with a mask, automatic schedule, every element."""
    import torch
    inp = synth.workload(name)
    mask = synth.additive_mask(inp.B * inp.H_q, inp.L, _s_mask(inp), 80)
    dev = gu.to_device(inp)
    out = B.paged_attention(dev["query"], dev["key_pages"], dev["value_pages"],
                            dev["block_table"], dev["context_lens"], inp.page_size,
                            scale=inp.scale, causal=True,
                            mask=torch.from_numpy(mask).cuda())
    torch.cuda.synchronize()
    got = gu.out_to_f64(out)
    ref = oracle_lib.paged_attention(inp.query, inp.key_pages, inp.value_pages,
                                     inp.block_table, inp.context_lens, inp.scale, True,
                                     mask=mask)
    gu.assert_parity(got, ref, "bf16", f"{name} masked auto")


@pytest.mark.parametrize("G,L", [(1, 130), (2, 90), (8, 50), (16, 30)])
def test_masked_tiles_every_group_size(oracle_lib, G, L):
    """The tile schedule's mask stager stages one box per head of Lt = 128 / G
    rows: every GQA group size it takes, causal, every element."""
    H_kv = 2 if G <= 8 else 1
    inp = synth.generate(B=2, H_q=G * H_kv, H_kv=H_kv, L=L, D=128, page_size=32,
                         context_lens=[L, 400], seed=100 + G, name=f"mask-G{G}")
    mask = synth.additive_mask(inp.B * inp.H_q, inp.L, _s_mask(inp, 4), 110 + G)
    got = gu.out_to_f64(run_masked(inp, mask, B.PA_SCHED_PREFILL))
    ref = oracle_lib.paged_attention(inp.query, inp.key_pages, inp.value_pages,
                                     inp.block_table, inp.context_lens, inp.scale, True,
                                     mask=mask)
    gu.assert_parity(got, ref, "bf16", f"mask G={G} tiles")


@pytest.mark.parametrize("sched", ["decode", "prefill"])
def test_fully_masked_row_outputs_zero(oracle_lib, sched):
    inp = _small_cases()[1]
    mask = synth.additive_mask(inp.B * inp.H_q, inp.L, _s_mask(inp), 90, removed=0.1)
    mask[1 * inp.H_q + 3, 7, :] = -np.inf  # every key of row (b=1, h=3, l=7)
    schedule = B.PA_SCHED_DECODE if sched == "decode" else B.PA_SCHED_PREFILL
    got = gu.out_to_f64(run_masked(inp, mask, schedule))
    assert not got[1, 3, 7].any()
    ref = oracle_lib.paged_attention(inp.query, inp.key_pages, inp.value_pages,
                                     inp.block_table, inp.context_lens, inp.scale, True,
                                     mask=mask)
    gu.assert_parity(got, ref, "bf16", f"fully masked row, {sched}")


def test_zero_mask_leaves_the_page_walk_bitwise_unchanged():
    import torch
    inp = _small_cases()[2]
    ref, _ = gu.run(inp, B.PA_SCHED_DECODE)
    zero = np.zeros((inp.B * inp.H_q, inp.L, _s_mask(inp)), dtype=np.float32)
    out = run_masked(inp, zero, B.PA_SCHED_DECODE)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_masked_fp32_control(oracle_lib):
    inp = synth.generate(B=2, H_q=8, H_kv=2, L=9, D=128, page_size=16,
                         context_lens=[40, 130], seed=64, dtype="f32", name="mask-f32")
    mask = synth.additive_mask(inp.B * inp.H_q, inp.L, _s_mask(inp), 91)
    got = gu.out_to_f64(run_masked(inp, mask, B.PA_SCHED_DECODE))
    ref = oracle_lib.paged_attention(inp.query, inp.key_pages, inp.value_pages,
                                     inp.block_table, inp.context_lens, inp.scale, True,
                                     mask=mask)
    gu.assert_parity(got, ref, "f32", "fp32 masked")


def test_masked_argument_checks():
    import torch
    inp = synth.workload("tiny")
    dev = gu.to_device(inp)
    sh = B.shape_of(dev["query"], dev["key_pages"], dev["block_table"])
    ws = B.new_workspace(sh)
    out = torch.empty_like(dev["query"])
    cap = _capacity(inp)
    rows = inp.B * inp.H_q

    def call(mask, s_mask):
        return B.pa_paged_attention_masked(sh, dev["query"], dev["key_pages"],
                                           dev["value_pages"], dev["block_table"],
                                           dev["context_lens"], inp.scale, True, mask, s_mask,
                                           out, ws, ws.numel(), None, B.PA_SCHED_AUTO)

    good = torch.zeros(rows * inp.L * (cap + 4) + 4, dtype=torch.float32, device="cuda")
    assert call(good, cap) == B.PA_OK
    torch.cuda.synchronize()
    assert call(None, cap) == B.PA_ERR_INVALID_ARG
    assert call(good, cap - 4) == B.PA_ERR_INVALID_ARG      # shorter than the capacity
    assert call(good, cap + 2) == B.PA_ERR_INVALID_ARG      # not a multiple of 4
    assert call(good[1:], cap) == B.PA_ERR_INVALID_ARG      # not 16-byte aligned
