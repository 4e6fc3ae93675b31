"""Pages shared between sequences (a common prefix held once).

Nothing in the page translation ("Week 3 Day 5: Paged FlashAttention",
Task 1) requires a physical page to belong to one sequence, and the pool is
only read, so several block-table rows may name the same page.  The result
must not depend on it: a batch whose sequences share their prefix pages is
compared bitwise with the same batch holding private copies of those pages,
and with the oracle, for both schedules and the ragged batch.
"""
import numpy as np
import pytest

import gpu_util as gu
from paged_kv_cache_03_gb300 import binding as B
from paged_kv_cache_03_gb300 import synth

pytestmark = pytest.mark.gpu


def share_prefix(inp, n_shared):
    """(private, shared): the first n_shared logical pages of every sequence
    hold sequence 0's prefix; `private` copies it into each sequence's own
    pages, `shared` points every table row at sequence 0's pages."""
    kp, vp, bt = inp.key_pages.copy(), inp.value_pages.copy(), inp.block_table.copy()
    for b in range(1, len(bt)):
        for i in range(n_shared):
            kp[bt[b, i]] = kp[bt[0, i]]
            vp[bt[b, i]] = vp[bt[0, i]]
    shared_bt = bt.copy()
    shared_bt[1:, :n_shared] = bt[0, :n_shared]
    return (kp, vp, bt), (kp, vp, shared_bt)


def with_pool(inp, kp, vp, bt):
    return synth.PagedInputs(inp.query, kp, vp, bt, inp.context_lens, inp.page_size, inp.scale,
                             inp.causal, inp.dtype, inp.name)


CASES = [
    # (B, H_q, H_kv, L, page_size, contexts, shared pages)
    (4, 8, 2, 1, 16, [100, 130, 77, 200], 4),
    (3, 8, 2, 40, 16, [100, 130, 300], 5),
    (3, 32, 8, 65, 128, [300, 1000, 700], 2),
]


@pytest.mark.parametrize("sched", ["decode", "prefill"])
@pytest.mark.parametrize("case", range(len(CASES)), ids=[f"case{i}" for i in range(len(CASES))])
def test_shared_prefix_pages(oracle_lib, case, sched):
    import torch
    Bn, H_q, H_kv, L, ps, ctx, n = CASES[case]
    inp = synth.generate(B=Bn, H_q=H_q, H_kv=H_kv, L=L, D=128, page_size=ps, context_lens=ctx,
                         seed=90 + case, name=f"shared{case}")
    private, shared = share_prefix(inp, n)
    schedule = {"decode": B.PA_SCHED_DECODE, "prefill": B.PA_SCHED_PREFILL}[sched]
    a, _ = gu.run(with_pool(inp, *private), schedule)  # both schedules take every case
    sh_inp = with_pool(inp, *shared)
    b, _ = gu.run(sh_inp, schedule)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "page sharing changed the output"
    gu.assert_parity(gu.out_to_f64(b), gu.oracle_full(oracle_lib, sh_inp), "bf16",
                     f"shared{case}/{sched}")


@pytest.mark.parametrize("schedule", [B.PA_SCHED_AUTO, B.PA_SCHED_DECODE, B.PA_SCHED_PREFILL],
                         ids=["auto", "decode", "tiles"])
def test_shared_prefix_pages_in_a_ragged_batch(oracle_lib, schedule):
    import torch
    from test_varlen_gpu import oracle_varlen, run_varlen, to_device
    inp = synth.generate_ragged(8, 2, 128, 16, [1, 37, 1, 130, 4], [90, 300, 64, 700, 129],
                                seed=95)
    private, shared = share_prefix(inp, 4)
    outs = []
    for kp, vp, bt in (private, shared):
        r = synth.RaggedInputs(inp.query, kp, vp, bt, inp.context_lens, inp.cu_q, inp.page_size,
                               inp.scale, inp.causal, inp.dtype, inp.name)
        res = run_varlen(r, schedule, dev=to_device(r))
        assert res is not None, "the forced schedule refused a shape it takes"
        outs.append((r, res[0]))
    assert torch.equal(outs[0][1].view(torch.int16), outs[1][1].view(torch.int16))
    r, out = outs[1]
    gu.assert_parity(gu.out_to_f64(out), oracle_varlen(oracle_lib, r), "bf16", "shared/ragged")
