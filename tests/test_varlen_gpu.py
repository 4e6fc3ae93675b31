"""Ragged batches on the GPU (pa_paged_attention_varlen) vs the oracle.

A ragged batch mixes decode steps (one query), prefill chunks and
continuations (many queries) and sequences without new queries in one call;
queries and outputs are packed by token.  Every case runs the automatic
routing (short sequences to the page walk, long ones to the tensor-core
tiles, in the same call) and both forced schedules, and compares every output
row with the oracle's ragged-batch function.  Further tests: a batch of equal
query counts gives bitwise the rows of the [B, H_q, L, D] path, the
full-size continuous-batching step, fp32, empty sequences with junk metadata,
broken offsets (flagged, nothing written outside the output) and argument
checks.
"""
import numpy as np
import pytest

import gpu_util as gu
from paged_kv_cache_03_gb300 import binding as B
from paged_kv_cache_03_gb300 import synth

pytestmark = pytest.mark.gpu

SCHEDULES = [B.PA_SCHED_AUTO, B.PA_SCHED_DECODE, B.PA_SCHED_PREFILL]
SCHED_IDS = ["auto", "decode", "tiles"]


def to_device(inp):
    import torch

    def conv(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if inp.dtype == "bf16":
            t = t.view(torch.bfloat16)
        return t.cuda()

    return dict(query=conv(inp.query), key_pages=conv(inp.key_pages),
                value_pages=conv(inp.value_pages),
                block_table=torch.from_numpy(np.ascontiguousarray(inp.block_table)).cuda(),
                context_lens=torch.from_numpy(np.ascontiguousarray(inp.context_lens)).cuda(),
                cu_q=torch.from_numpy(np.ascontiguousarray(inp.cu_q)).cuda())


def run_varlen(inp, schedule=B.PA_SCHED_AUTO, dev=None, max_L=None, cu_q=None, total_q=None,
               check_flag=True, out=None):
    """Runs the ragged-batch entry point; returns (out tensor, flag) or None
    when a forced schedule cannot take the shape."""
    import torch
    dev = dev or to_device(inp)
    max_L = inp.max_L if max_L is None else max_L
    shape = B.shape_of_varlen(dev["query"], dev["key_pages"], dev["block_table"], max_L)
    ws = B.new_workspace(shape)
    if out is None:
        out = torch.zeros_like(dev["query"])
    st = B.pa_paged_attention_varlen(
        shape, dev["query"], dev["key_pages"], dev["value_pages"], dev["block_table"],
        dev["context_lens"], dev["cu_q"] if cu_q is None else cu_q,
        dev["query"].shape[0] if total_q is None else total_q, inp.scale, inp.causal, out, ws,
        ws.numel(), None, schedule)
    if st == B.PA_ERR_UNSUPPORTED and schedule != B.PA_SCHED_AUTO:
        return None
    assert st == B.PA_OK, B.status_str(st)
    torch.cuda.synchronize()
    _, flag = B.pa_check_device_flag(ws)
    if check_flag:
        assert flag == 0, f"device flag {flag:#x}"
    return out, flag


def oracle_varlen(lib, inp):
    return lib.paged_attention_varlen(inp.query, inp.key_pages, inp.value_pages,
                                      inp.block_table, inp.context_lens, inp.cu_q, inp.scale,
                                      inp.causal)


CASES = [
    # (name, H_q, H_kv, page_size, query counts, context lengths, causal, seed)
    ("gqa4-mixed", 8, 2, 16, [1, 0, 37, 1, 5, 130, 1, 2], [50, 9, 300, 1, 5, 700, 2048, 129],
     True, 401),
    ("gqa1-rows-around-4", 4, 4, 16, [1, 2, 3, 4, 5, 200, 4], [10, 64, 3, 400, 5, 900, 33],
     True, 402),
    ("gqa8-all-tiles", 16, 2, 64, [1, 1, 65, 3], [77, 1000, 65, 8], True, 403),
    ("full-visibility", 8, 2, 16, [1, 7, 40, 1], [30, 7, 500, 2], False, 404),
    ("page128-long", 32, 8, 128, [1, 128, 1, 256], [4000, 1500, 129, 3000], True, 405),
    ("page8-tiles-edge", 8, 2, 8, [33, 1, 64], [33, 17, 200], True, 406),
    # page sizes the tiles do not take: the page walk serves every sequence,
    # a tile of keys spanning many page pieces
    ("page3-walk-only", 8, 2, 3, [1, 0, 9, 2], [40, 5, 100, 7], True, 407),
    ("page1-walk-only", 4, 4, 1, [3, 1], [50, 20], True, 408),
    # mask=None with more queries than keys in some sequences: every row sees
    # the whole context
    ("no-causal-more-queries-than-keys", 8, 2, 16, [40, 1, 130, 3, 9], [7, 3, 50, 1, 200],
     False, 409),
    ("no-causal-L-over-S-page128", 32, 8, 128, [300, 1, 65], [129, 1, 64], False, 410),
]


@pytest.mark.parametrize("case", [c for c in CASES if not gu.tiles_take("bf16", *c[1:4])],
                         ids=lambda c: c[0])
def test_varlen_tiles_refuse_page_sizes_they_do_not_take(case):
    name, H_q, H_kv, ps, q_lens, ctx, causal, seed = case
    inp = synth.generate_ragged(H_q, H_kv, 128, ps, q_lens, ctx, seed=seed, causal=causal,
                                name=name)
    assert run_varlen(inp, B.PA_SCHED_PREFILL) is None


def _case_schedules():
    """Every case on AUTO and the forced page walk; the forced tiles only
    where the tiles take the page size (the walk-only cases check, in
    test_varlen_tiles_refuse_page_sizes_they_do_not_take, that the library
    refuses them)."""
    for c in CASES:
        for s, sid in zip(SCHEDULES, SCHED_IDS):
            if s == B.PA_SCHED_PREFILL and not gu.tiles_take("bf16", c[1], c[2], c[3]):
                continue
            yield pytest.param(c, s, id=f"{c[0]}-{sid}")


@pytest.mark.parametrize("case,schedule", list(_case_schedules()))
def test_varlen_matches_oracle(oracle_lib, case, schedule):
    name, H_q, H_kv, ps, q_lens, ctx, causal, seed = case
    inp = synth.generate_ragged(H_q, H_kv, 128, ps, q_lens, ctx, seed=seed, causal=causal,
                                name=name)
    res = run_varlen(inp, schedule)
    assert res is not None, "the forced schedule refused a shape it takes"
    got = gu.out_to_f64(res[0])
    gu.assert_parity(got, oracle_varlen(oracle_lib, inp), "bf16", f"{name} sched {schedule}")


def test_varlen_uniform_batch_equals_uniform_path_bitwise():
    """Equal query counts: the ragged call gives bitwise the [B, H_q, L, D]
    path's rows, on both schedules (the same arithmetic over the same data)."""
    import torch
    for L, sched in ((1, B.PA_SCHED_DECODE), (3, B.PA_SCHED_DECODE), (70, B.PA_SCHED_PREFILL),
                     (70, B.PA_SCHED_DECODE)):
        u = synth.generate(3, 8, 2, L, 128, 16, context_lens=[L + 20, 300, L], seed=410 + L)
        r = synth.RaggedInputs(np.ascontiguousarray(u.query.transpose(0, 2, 1, 3).reshape(
                                   -1, u.query.shape[1], u.query.shape[3])),
                               u.key_pages, u.value_pages, u.block_table, u.context_lens,
                               np.arange(0, 3 * L + 1, L, dtype=np.int32), u.page_size, u.scale,
                               u.causal, u.dtype, "uniform-as-ragged")
        out_u, _ = gu.run(u, sched)
        out_r, _ = run_varlen(r, sched)
        a = out_u.view(torch.int16).cpu().numpy().transpose(0, 2, 1, 3).reshape(out_r.shape)
        assert np.array_equal(a, out_r.view(torch.int16).cpu().numpy()), (L, sched)


def test_varlen_continuous_batching_step(oracle_lib):
    """The full-size mixed step: 56 decodes and 8 chunks of 128 tokens."""
    inp = synth.mixed_workload()
    ref = oracle_varlen(oracle_lib, inp)
    for sched in SCHEDULES:
        got = gu.out_to_f64(run_varlen(inp, sched)[0])
        gu.assert_parity(got, ref, "bf16", f"mixed step sched {sched}")


def test_varlen_fp32_control(oracle_lib):
    inp = synth.generate_ragged(8, 2, 128, 16, [1, 9, 0, 3], [40, 9, 5, 100], seed=420,
                                dtype="f32")
    for sched in (B.PA_SCHED_AUTO, B.PA_SCHED_DECODE):
        got = gu.out_to_f64(run_varlen(inp, sched)[0])
        gu.assert_parity(got, oracle_varlen(oracle_lib, inp), "f32", f"fp32 sched {sched}")
    assert run_varlen(inp, B.PA_SCHED_PREFILL) is None  # the tiles take bf16 only


def test_varlen_empty_sequences_are_never_read(oracle_lib):
    """Sequences with no new queries may carry any context length and table
    row: nothing of them is read and nothing is flagged."""
    inp = synth.generate_ragged(8, 2, 128, 16, [2, 0, 70, 0, 1], [20, 10, 200, 10, 5], seed=430)
    ref = oracle_varlen(oracle_lib, inp)
    bt = inp.block_table.copy()
    ctx = inp.context_lens.copy()
    bt[1, :] = 10 ** 6
    bt[3, :] = -7
    ctx[1] = -3
    ctx[3] = 10 ** 7
    junk = synth.RaggedInputs(inp.query, inp.key_pages, inp.value_pages, bt, ctx, inp.cu_q,
                              inp.page_size, inp.scale, inp.causal, inp.dtype, "junk")
    for sched in SCHEDULES:
        got = gu.out_to_f64(run_varlen(junk, sched)[0])
        gu.assert_parity(got, ref, "bf16", f"empty sequences sched {sched}")


def test_varlen_broken_offsets_are_flagged_and_skipped(oracle_lib):
    """An offset array that runs past total_q or backwards, or a query count
    above shape.L, sets PA_FLAG_BAD_CONTEXT; the other sequences are exact and
    nothing is written outside [0, total_q) (guard rows stay intact)."""
    import torch
    inp = synth.generate_ragged(8, 2, 128, 16, [3, 70, 1], [30, 300, 9], seed=440)
    ref = oracle_varlen(oracle_lib, inp)
    T = int(inp.cu_q[-1])
    dev = to_device(inp)
    for cu_bad, bad_seq in (([0, 3, 73, 80], 2),     # runs past total_q
                            ([0, 3, 1, 74], 1),      # backwards
                            ([0, 3, 73, 74], None)):  # valid, but max_L = 60 < 70
        for sched in SCHEDULES:
            guard = torch.full((T + 16, inp.H_q, inp.D), 7.0, dtype=torch.bfloat16,
                               device="cuda")
            out = guard[:T]
            max_L = 60 if bad_seq is None else inp.max_L
            res = run_varlen(inp, sched, dev=dev, max_L=max_L,
                             cu_q=torch.tensor(cu_bad, dtype=torch.int32, device="cuda"),
                             total_q=T, check_flag=False, out=out)
            if res is None:
                continue
            _, flag = res
            assert flag & B.PA_FLAG_BAD_CONTEXT, (cu_bad, sched)
            tail = guard[T:].float().cpu().numpy()
            assert np.all(tail == 7.0), "a write landed past total_q"
            got = gu.out_to_f64(out)
            if bad_seq is None:
                keep = [0, 2]  # sequence 1 (70 queries > max_L 60) is skipped
            elif bad_seq == 2:
                keep = [0, 1]
            else:  # sequence 1 runs backwards, sequence 2 then holds 73 > max_L queries
                keep = [0]
            for b in keep:
                lo, hi = cu_bad[b], cu_bad[b + 1]
                gu.assert_parity(got[lo:hi], ref[inp.cu_q[b]:inp.cu_q[b + 1]], "bf16",
                                 f"sequence {b} beside broken offsets {cu_bad}")


def test_varlen_argument_checks():
    import torch
    inp = synth.generate_ragged(8, 2, 128, 16, [1, 2], [5, 9], seed=450)
    dev = to_device(inp)
    shape = B.shape_of_varlen(dev["query"], dev["key_pages"], dev["block_table"], 2)
    ws = B.new_workspace(shape)
    out = torch.empty_like(dev["query"])
    args = (dev["query"], dev["key_pages"], dev["value_pages"], dev["block_table"],
            dev["context_lens"])

    def call(cu_q=dev["cu_q"], total_q=3, wsb=ws.numel(), sched=B.PA_SCHED_AUTO, o=out):
        return B.pa_paged_attention_varlen(shape, *args, cu_q, total_q, inp.scale, True, o, ws,
                                           wsb, None, sched)

    assert call() == B.PA_OK
    assert call(cu_q=None) == B.PA_ERR_INVALID_ARG
    assert call(total_q=-1) == B.PA_ERR_INVALID_ARG
    assert call(wsb=64) == B.PA_ERR_WORKSPACE
    assert call(sched=7) == B.PA_ERR_INVALID_ARG
    assert call(o=None) == B.PA_ERR_INVALID_ARG
    assert call(total_q=0) == B.PA_OK
    torch.cuda.synchronize()


def test_varlen_many_sequences(oracle_lib):
    """1500 sequences (more than one 1024-wide scan block in the tile plan and
    several in the page walk's prologue): decode steps, empty sequences and
    a 40-token chunk every 50th sequence."""
    rng = np.random.default_rng(460)
    B = 1500
    q_lens = np.ones(B, dtype=np.int64)
    q_lens[::50] = 40
    q_lens[7::97] = 0
    ctx = rng.integers(40, 401, size=B)
    inp = synth.generate_ragged(8, 2, 128, 16, q_lens, ctx, seed=461, name="many")
    ref = oracle_varlen(oracle_lib, inp)
    for sched in SCHEDULES:
        got = gu.out_to_f64(run_varlen(inp, sched)[0])
        gu.assert_parity(got, ref, "bf16", f"1500 sequences sched {sched}")


def test_varlen_validate_metadata():
    """The host-side check of a ragged batch's metadata accepts what the oracle
    accepts and rejects the same broken offsets, lengths and table entries."""
    import torch
    inp = synth.generate_ragged(8, 2, 128, 16, [2, 0, 70, 1], [20, 5, 300, 9], seed=470)
    dev = to_device(inp)
    shape = B.shape_of_varlen(dev["query"], dev["key_pages"], dev["block_table"], inp.max_L)
    T = int(inp.cu_q[-1])

    def check(cu=None, ctx=None, bt=None, total=T, causal=True):
        t = lambda a: torch.tensor(np.asarray(a), dtype=torch.int32, device="cuda")  # noqa: E731
        return B.pa_validate_metadata_varlen(
            shape, dev["block_table"] if bt is None else t(bt),
            dev["context_lens"] if ctx is None else t(ctx),
            dev["cu_q"] if cu is None else t(cu), total, causal)

    assert check() == B.PA_OK
    assert check(ctx=[20, -9, 300, 9]) == B.PA_OK  # the empty sequence is not read
    assert check(cu=[1, 3, 3, 73, 74]) == B.PA_ERR_INVALID_ARG
    assert check(cu=[0, 2, 1, 73, 74]) == B.PA_ERR_INVALID_ARG
    assert check(total=T + 1) == B.PA_ERR_INVALID_ARG
    assert check(ctx=[1, 5, 300, 9]) == B.PA_ERR_INVALID_ARG  # 2 queries, 1 key, causal
    assert check(ctx=[1, 5, 300, 9], causal=False) == B.PA_OK
    bt = inp.block_table.copy()
    bt[2, 5] = inp.num_pages
    assert check(bt=bt) == B.PA_ERR_BAD_BLOCK_TABLE
