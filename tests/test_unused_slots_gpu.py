"""Unused page slots hold anything.

A page's slots past its sequence's context length, and pages that no block
table names, are not part of any sequence ("Week 3 Day 5: Paged
FlashAttention", Task 1: only positions s < context_len are translated), so
their contents must not reach the output.  Every such K/V row is filled with
NaN or +-Inf and the outputs must be bitwise those of the clean pool, for
both schedules, the explicit mask and the ragged batch.  (The tile schedule
copies whole boxes of page rows, so the last K/V tile of a sequence can carry
rows past the context: their weights are exactly 0, but 0 * NaN is not.)
"""
import numpy as np
import pytest

import gpu_util as gu
from paged_kv_cache_03_gb300 import binding as B
from paged_kv_cache_03_gb300 import synth

pytestmark = pytest.mark.gpu

BF16_BITS = {"nan": 0x7FC0, "inf": 0x7F80, "-inf": 0xFF80}


def used_slots(block_table, context_lens, num_pages, page_size):
    """[num_pages, page_size] True where a slot holds a position s < context
    length of some sequence."""
    used = np.zeros((num_pages, page_size), dtype=bool)
    for b, S in enumerate(context_lens):
        for s in range(int(S)):
            used[block_table[b, s // page_size], s % page_size] = True
    return used


def poisoned_pool(pool, used, fill, dtype):
    out = pool.copy()
    if dtype == "bf16":
        out.view(np.uint16)[~used] = BF16_BITS[fill]
    else:
        out[~used] = {"nan": np.nan, "inf": np.inf, "-inf": -np.inf}[fill]
    return out


def poisoned(inp, fill):
    used = used_slots(inp.block_table, inp.context_lens, inp.key_pages.shape[0], inp.page_size)
    # [num_pages, H_kv, ps, D]: the slot mask broadcast over heads and dims
    u = np.broadcast_to(used[:, None, :, None], inp.key_pages.shape)
    kp = poisoned_pool(inp.key_pages, u, fill, inp.dtype)
    vp = poisoned_pool(inp.value_pages, u, fill, inp.dtype)
    return kp, vp


def _uniform_cases():
    return [
        synth.workload("tiny"),  # page 16, contexts 13 and 40
        synth.generate(B=3, H_q=8, H_kv=2, L=65, D=128, page_size=128,
                       context_lens=[300, 1000, 65], seed=71, name="tails-small"),
        synth.generate(B=2, H_q=4, H_kv=1, L=200, D=128, page_size=16,
                       context_lens=[200, 513], num_pages=50, seed=72,
                       name="ps16-crossing"),  # 4 pages no table names
        synth.generate(B=2, H_q=16, H_kv=4, L=77, D=128, page_size=64,
                       context_lens=[77, 390], causal=False, seed=73, name="ps64-full"),
        synth.generate(B=2, H_q=32, H_kv=8, L=1, D=128, page_size=16,
                       context_lens=[700, 129], seed=74, name="decode-small"),
        # contexts that end on a page boundary inside a key tile: the tiles'
        # last key tile is partial with no box past the context (400: its
        # fourth tile reuses a slot; 208: its second tile is the slot's first)
        synth.generate(B=2, H_q=16, H_kv=4, L=80, D=128, page_size=16,
                       context_lens=[400, 208], seed=79, name="ps16-page-aligned-ends"),
    ]


def _bitwise_equal(a, b):
    import torch
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


@pytest.mark.parametrize("fill", ["nan", "inf"])
@pytest.mark.parametrize("sched", ["decode", "prefill"])
@pytest.mark.parametrize("case", range(6))
def test_unused_slots_never_reach_the_output(case, sched, fill):
    import torch
    inp = _uniform_cases()[case]
    schedule = {"decode": B.PA_SCHED_DECODE, "prefill": B.PA_SCHED_PREFILL}[sched]
    dev = gu.to_device(inp)
    clean, _ = gu.run(inp, schedule, dev=dev)  # every case is a shape both schedules take
    kp, vp = poisoned(inp, fill)
    conv = (lambda a: torch.from_numpy(a).view(torch.bfloat16).cuda()) if inp.dtype == "bf16" \
        else (lambda a: torch.from_numpy(a).cuda())
    dev2 = dict(dev, key_pages=conv(kp), value_pages=conv(vp))
    out, flag = gu.run(inp, schedule, dev=dev2)
    assert flag == 0
    assert torch.isfinite(out.float()).all(), f"{inp.name}/{sched}: non-finite output"
    assert _bitwise_equal(clean, out), f"{inp.name}/{sched}: unused slots changed the output"


def test_unused_slots_fp32_page_walk():
    import torch
    inp = synth.generate(B=2, H_q=8, H_kv=2, L=3, D=128, page_size=16, context_lens=[37, 5],
                         seed=75, dtype="f32", name="f32-small")
    dev = gu.to_device(inp)
    clean, _ = gu.run(inp, B.PA_SCHED_DECODE, dev=dev)
    kp, vp = poisoned(inp, "nan")
    dev2 = dict(dev, key_pages=torch.from_numpy(kp).cuda(), value_pages=torch.from_numpy(vp).cuda())
    out, _ = gu.run(inp, B.PA_SCHED_DECODE, dev=dev2)
    assert _bitwise_equal(clean, out)


@pytest.mark.parametrize("sched", ["decode", "prefill"])
def test_unused_slots_with_an_explicit_mask(sched):
    import torch
    from test_mask_gpu import _s_mask, run_masked
    inp = synth.generate(B=2, H_q=4, H_kv=1, L=40, D=128, page_size=16, context_lens=[45, 130],
                         seed=76, name="mask-ps16")
    mask = synth.additive_mask(inp.B * inp.H_q, inp.L, _s_mask(inp), seed=77)
    schedule = {"decode": B.PA_SCHED_DECODE, "prefill": B.PA_SCHED_PREFILL}[sched]
    dev = gu.to_device(inp)
    clean = run_masked(inp, mask, schedule, dev=dev)
    kp, vp = poisoned(inp, "nan")
    dev2 = dict(dev, key_pages=torch.from_numpy(kp).view(torch.bfloat16).cuda(),
                value_pages=torch.from_numpy(vp).view(torch.bfloat16).cuda())
    out = run_masked(inp, mask, schedule, dev=dev2)
    assert _bitwise_equal(clean, out)


@pytest.mark.parametrize("schedule", [B.PA_SCHED_AUTO, B.PA_SCHED_DECODE, B.PA_SCHED_PREFILL],
                         ids=["auto", "decode", "tiles"])
def test_unused_slots_in_a_ragged_batch(schedule):
    import torch
    from test_varlen_gpu import run_varlen, to_device
    inp = synth.generate_ragged(8, 2, 128, 16, [1, 0, 37, 1, 5, 130, 3], [50, 9, 300, 1, 5, 700, 33],
                                seed=78)
    dev = to_device(inp)
    r = run_varlen(inp, schedule, dev=dev)
    assert r is not None, "the forced schedule refused a shape it takes"
    clean = r[0]
    kp, vp = poisoned(inp, "-inf")
    dev2 = dict(dev, key_pages=torch.from_numpy(kp).view(torch.bfloat16).cuda(),
                value_pages=torch.from_numpy(vp).view(torch.bfloat16).cuda())
    out, _ = run_varlen(inp, schedule, dev=dev2)
    assert _bitwise_equal(clean, out)
