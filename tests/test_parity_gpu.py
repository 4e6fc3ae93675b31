"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Bars: bf16 max-abs <= 1e-2 and mean-abs <= 1e-3; fp32 control max-abs
<= 1e-5; page translation (debug gather) bit-exact; outputs bitwise equal
under physical page permutation and under junk in unused block-table entries.
"""
import functools

import numpy as np
import pytest

import gpu_util as gu
import pins
from paged_kv_cache_03_gb300 import binding as B
from paged_kv_cache_03_gb300 import synth

pytestmark = pytest.mark.gpu

SCHEDULES = {"decode": B.PA_SCHED_DECODE, "prefill": B.PA_SCHED_PREFILL}


@functools.lru_cache(maxsize=None)
def workload(name, dtype="bf16"):
    return synth.workload(name, dtype=dtype)


def check(oracle_lib, inp, schedule=B.PA_SCHED_AUTO, rows=None, what=""):
    """Runs one schedule and compares with the oracle.  A forced tile call on
    a shape outside the tiles' rule is refused by the library (checked here)
    and compares nothing; inside the rule it must run."""
    try:
        out, _ = gu.run(inp, schedule)
    except gu.Unsupported:
        assert schedule == B.PA_SCHED_PREFILL and not gu.tiles_take(
            inp.dtype, inp.H_q, inp.H_kv, inp.page_size), f"{what}: refused a shape it takes"
        return None
    got = gu.out_to_f64(out)
    if rows is None:
        ref = gu.oracle_full(oracle_lib, inp)
    else:
        ref = gu.oracle_rows(oracle_lib, inp, rows)
        got = got[rows[:, 0], rows[:, 1], rows[:, 2]]
    return gu.assert_parity(got, ref, inp.dtype, what or inp.name)


# ---- the five named workloads ------------------------------------------------
@pytest.mark.parametrize("name", ["tiny", "decode", "tails", "long_decode"])
def test_workload_auto_schedule(oracle_lib, name):
    check(oracle_lib, workload(name))


@functools.lru_cache(maxsize=None)
def oracle_of_workload(name, dtype="bf16"):
    """The oracle's full output for a named workload (computed once per run:
    the causal prefill takes about 7e10 fp64 multiply-adds)."""
    import oracle
    return gu.oracle_full(oracle.load(), workload(name, dtype))


@pytest.mark.parametrize("sched", ["auto", "decode", "prefill"])
def test_prefill_workload_every_element(sched):
    """The causal prefill (B=4, L=S=2048, 32/8 heads, pages of 128, keys x2)
    compared with the oracle element by element, all 33.5M outputs, on the
    automatic choice and both forced schedules."""
    inp = workload("prefill")
    out, _ = gu.run(inp, {"auto": B.PA_SCHED_AUTO, **SCHEDULES}[sched])
    gu.assert_parity(gu.out_to_f64(out), oracle_of_workload("prefill"), "bf16",
                     f"prefill/{sched}")


@pytest.mark.parametrize("name", ["tiny", "tails"])
@pytest.mark.parametrize("sched", ["decode", "prefill"])
def test_workload_forced_schedule(oracle_lib, name, sched):
    check(oracle_lib, workload(name), SCHEDULES[sched], what=f"{name}/{sched}")


# ---- the page's required fixtures ("Week 3 Day 5", Task 3) --------------------
FIXTURES = pins.golden("paged_fixtures.json")["fixtures"]


def fixture_inputs(fx, dtype="bf16"):
    kw = {k: fx[k] for k in ("B", "H_q", "H_kv", "L", "page_size", "context_lens", "causal")}
    if "num_pages" in fx:
        kw["num_pages"] = fx["num_pages"]
    seed = sum(ord(c) for c in fx["name"])
    return synth.generate(D=128, seed=seed, dtype=dtype, name=fx["name"], **kw)


@pytest.mark.parametrize("fx", FIXTURES, ids=[f["name"] for f in FIXTURES])
@pytest.mark.parametrize("sched", ["auto", "decode", "prefill"])
def test_page_fixture(oracle_lib, fx, sched):
    inp = fixture_inputs(fx)
    check(oracle_lib, inp, {"auto": B.PA_SCHED_AUTO, **SCHEDULES}[sched])


def test_output_dtype_stays_bf16():
    import torch
    inp = fixture_inputs(FIXTURES[-1])
    out, _ = gu.run(inp)
    assert out.dtype == torch.bfloat16 and tuple(out.shape) == inp.query.shape


def test_non_consecutive_pages_are_scattered():
    inp = fixture_inputs(next(f for f in FIXTURES if f["name"] == "non_consecutive_physical_pages"))
    used = inp.block_table[inp.block_table >= 0]
    assert np.any(np.diff(used) != 1)


# ---- the operator grid of "Week 2 Day 5", Task 3, restated on pages -----------
GRID = pins.golden("week2_operator_grid.json")


def grid_cases():
    for ctx in GRID["contexts"]:
        for L in GRID["query_lengths"]:
            for gqa in GRID["gqa_ratios"]:
                for causal in (True, False):
                    if causal and L > ctx:
                        continue
                    yield ctx, L, gqa, causal


@pytest.mark.parametrize("ctx,L,gqa,causal", list(grid_cases()))
def test_operator_grid(oracle_lib, ctx, L, gqa, causal):
    inp = synth.generate(B=2, H_q=2 * gqa, H_kv=2, L=L, D=128, page_size=16,
                         context_lens=[ctx, max(ctx, L) + 3], seed=1000 + ctx * 7 + L + gqa,
                         causal=causal, name=f"grid{ctx}")
    for s in (B.PA_SCHED_AUTO, B.PA_SCHED_DECODE, B.PA_SCHED_PREFILL):
        check(oracle_lib, inp, s, what=f"grid ctx={ctx} L={L} gqa={gqa} causal={causal}")


# ---- edge shapes -------------------------------------------------------------
EDGE = [
    # (name, kwargs)
    ("page_size_1", dict(B=2, H_q=4, H_kv=2, L=2, page_size=1, context_lens=[37, 5])),
    ("page_size_3", dict(B=2, H_q=4, H_kv=4, L=3, page_size=3, context_lens=[50, 3])),
    ("page_size_256", dict(B=2, H_q=8, H_kv=2, L=1, page_size=256, context_lens=[700, 256])),
    ("full_block_table", dict(B=2, H_q=4, H_kv=1, L=4, page_size=16, context_lens=[64, 64],
                              max_pages_per_seq=4)),
    ("context_equals_L", dict(B=2, H_q=2, H_kv=2, L=9, page_size=4, context_lens=[9, 12])),
    ("one_key", dict(B=3, H_q=2, H_kv=1, L=1, page_size=16, context_lens=[1, 1, 2])),
    ("gqa8_rows8", dict(B=2, H_q=16, H_kv=2, L=1, page_size=16, context_lens=[300, 33])),
    ("gqa16_two_chunks", dict(B=1, H_q=16, H_kv=1, L=1, page_size=64, context_lens=[1000])),
    ("mha_single_row", dict(B=4, H_q=4, H_kv=4, L=1, page_size=32, context_lens=[10, 900, 33, 1])),
    ("rows_not_multiple_of_8", dict(B=2, H_q=6, H_kv=2, L=3, page_size=8, context_lens=[77, 40])),
    ("many_short_sequences", dict(B=300, H_q=4, H_kv=1, L=1, page_size=16,
                                  ctx_range=(1, 40))),
    ("long_and_short_mixed", dict(B=5, H_q=8, H_kv=2, L=1, page_size=16,
                                  context_lens=[20000, 3, 700, 1, 9000])),
]


@pytest.mark.parametrize("name,kw", EDGE, ids=[e[0] for e in EDGE])
@pytest.mark.parametrize("causal", [True, False])
def test_edge_shapes(oracle_lib, name, kw, causal):
    inp = synth.generate(D=128, seed=sum(map(ord, name)), causal=causal, name=name, **kw)
    for s in (B.PA_SCHED_AUTO, B.PA_SCHED_DECODE, B.PA_SCHED_PREFILL):
        check(oracle_lib, inp, s, what=f"{name}/{s}")


# ---- fp32 control ---------------------------------------------------------------
@pytest.mark.parametrize("name", ["decode", "long_decode"])
def test_fp32_control_full_size_workload(oracle_lib, name):
    """The fp32 control build at the workloads' full size: the batched decode
    (64 contexts up to 4096 keys, segments split across CTAs and merged by the
    combine kernel) and the long decode (16 x 32768 keys over 16-slot pages),
    every element within 1e-5 of the oracle."""
    inp = synth.workload(name, dtype="f32")
    for sched in (B.PA_SCHED_AUTO, B.PA_SCHED_DECODE):
        check(oracle_lib, inp, sched, what=f"fp32 {name} sched {sched}")


@pytest.mark.parametrize("name", ["tiny", "fixture_L65", "fixture_crossing", "short_decode"])
def test_fp32_control(oracle_lib, name):
    if name == "tiny":
        inp = workload("tiny", "f32")
    elif name == "fixture_L65":
        inp = fixture_inputs(FIXTURES[3], "f32")
    elif name == "fixture_crossing":
        inp = fixture_inputs(FIXTURES[1], "f32")
    else:
        inp = synth.generate(B=8, H_q=32, H_kv=8, L=1, D=128, page_size=128,
                             ctx_range=(128, 2048), seed=77, dtype="f32")
    check(oracle_lib, inp, B.PA_SCHED_DECODE, what=f"fp32 {name}")


# ---- bit-exact page translation ---------------------------------------------------
@pytest.mark.parametrize("case", ["tiny", "crossing", "page1"])
def test_gather_is_bit_exact(oracle_lib, case):
    import torch
    if case == "tiny":
        inp = workload("tiny")
    elif case == "crossing":
        inp = fixture_inputs(FIXTURES[1])
    else:
        inp = synth.generate(B=2, H_q=2, H_kv=2, L=1, D=128, page_size=1, context_lens=[9, 4],
                             seed=5)
    dev = gu.to_device(inp)
    shape = B.shape_of(dev["query"], dev["key_pages"], dev["block_table"])
    max_S = int(inp.context_lens.max()) + 5
    kd = torch.empty((inp.B, inp.H_kv, max_S, inp.D), dtype=dev["key_pages"].dtype,
                     device="cuda")
    vd = torch.empty_like(kd)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    st = B.pa_gather_debug(shape, dev["key_pages"], dev["value_pages"], dev["block_table"],
                           dev["context_lens"], max_S, kd, vd, ws)
    assert st == B.PA_OK
    torch.cuda.synchronize()
    k_ref, v_ref = oracle_lib.gather(inp.key_pages, inp.value_pages, inp.block_table,
                                     inp.context_lens, max_S)
    assert np.array_equal(gu.out_to_f64(kd), k_ref)
    assert np.array_equal(gu.out_to_f64(vd), v_ref)
    assert B.pa_check_device_flag(ws)[1] == 0


def permuted(inp, seed):
    """Same logical K/V, different physical placement of every page."""
    perm = np.random.default_rng(seed).permutation(inp.num_pages).astype(np.int32)
    kp = np.empty_like(inp.key_pages)
    vp = np.empty_like(inp.value_pages)
    kp[perm] = inp.key_pages
    vp[perm] = inp.value_pages
    bt = inp.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    return synth.PagedInputs(inp.query, kp, vp, bt, inp.context_lens, inp.page_size,
                             inp.scale, inp.causal, inp.dtype, inp.name + "-perm")


@pytest.mark.parametrize("name", ["tiny", "decode", "tails"])
def test_page_permutation_is_bitwise_invisible(name):
    import torch
    inp = workload(name)
    a, _ = gu.run(inp)
    b, _ = gu.run(permuted(inp, 11))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_unused_block_table_entries_are_never_read():
    import torch
    inp = workload("decode")
    a, _ = gu.run(inp)
    for fill in (-1, 2 ** 31 - 1, inp.num_pages, -12345):
        bt = inp.block_table.copy()
        for b in range(inp.B):
            npg = (int(inp.context_lens[b]) + inp.page_size - 1) // inp.page_size
            bt[b, npg:] = fill
        out, flag = gu.run(inp, block_table=torch.from_numpy(bt).cuda())
        assert flag == 0
        assert torch.equal(a.view(torch.int16), out.view(torch.int16))


def test_repeatable_bitwise():
    import torch
    inp = workload("tails")
    a, _ = gu.run(inp)
    b, _ = gu.run(inp)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---- errors the kernels record instead of faulting ---------------------------------
def test_bad_page_id_sets_flag(oracle_lib):
    import torch
    inp = workload("tiny")
    bt = inp.block_table.copy()
    bt[0, 0] = inp.num_pages + 5
    out, flag = gu.run(inp, block_table=torch.from_numpy(bt).cuda(), check_flag=False)
    assert flag & B.PA_FLAG_BAD_PAGE
    # the other sequence is untouched by the bad entry
    ref = gu.oracle_full(oracle_lib, inp)
    gu.assert_parity(gu.out_to_f64(out)[1], ref[1], "bf16", "untouched sequence")


@pytest.mark.parametrize("bad", [0, -3, 10 ** 6, 2])
def test_bad_context_length_sets_flag_and_zeros(oracle_lib, bad):
    import torch
    inp = workload("tiny")  # L = 5, so a context of 2 breaks the causal contract
    ctx = inp.context_lens.copy()
    ctx[1] = bad
    out, flag = gu.run(inp, context_lens=torch.from_numpy(ctx).cuda(), check_flag=False)
    assert flag & B.PA_FLAG_BAD_CONTEXT
    got = gu.out_to_f64(out)
    assert not got[1].any()
    ref = gu.oracle_full(oracle_lib, inp)
    gu.assert_parity(got[0], ref[0], "bf16", "valid sequence")


def test_validate_metadata():
    import torch
    inp = workload("tiny")
    dev = gu.to_device(inp)
    sh = B.shape_of(dev["query"], dev["key_pages"], dev["block_table"])
    assert B.pa_validate_metadata(sh, dev["block_table"], dev["context_lens"], True) == B.PA_OK
    bt = inp.block_table.copy()
    bt[1, 2] = -1
    assert B.pa_validate_metadata(sh, torch.from_numpy(bt).cuda(), dev["context_lens"],
                                  True) == B.PA_ERR_BAD_BLOCK_TABLE
    ctx = inp.context_lens.copy()
    ctx[0] = 3
    assert B.pa_validate_metadata(sh, dev["block_table"], torch.from_numpy(ctx).cuda(),
                                  True) == B.PA_ERR_INVALID_ARG


def test_output_guard_bands_untouched():
    import torch
    inp = workload("tails")
    dev = gu.to_device(inp)
    n = dev["query"].numel()
    g = 4096
    big = torch.full((n + 2 * g,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big[g:g + n].view(dev["query"].shape)
    shape = B.shape_of(dev["query"], dev["key_pages"], dev["block_table"])
    ws = B.new_workspace(shape)
    st = B.pa_paged_attention(shape, dev["query"], dev["key_pages"], dev["value_pages"],
                              dev["block_table"], dev["context_lens"], inp.scale, True, out, ws,
                              ws.numel())
    assert st == B.PA_OK
    torch.cuda.synchronize()
    assert bool((big[:g] == 7.0).all()) and bool((big[g + n:] == 7.0).all())


def test_small_workspace_is_rejected():
    import torch
    inp = workload("decode")
    dev = gu.to_device(inp)
    shape = B.shape_of(dev["query"], dev["key_pages"], dev["block_table"])
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dev["query"])
    st = B.pa_paged_attention_sched(shape, dev["query"], dev["key_pages"], dev["value_pages"],
                                    dev["block_table"], dev["context_lens"], inp.scale, True, out,
                                    ws, ws.numel(), None, B.PA_SCHED_DECODE)
    assert st == B.PA_ERR_WORKSPACE


def test_side_stream(oracle_lib):
    import torch
    inp = workload("tiny")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, _ = gu.run(inp)
    gu.assert_parity(gu.out_to_f64(out), gu.oracle_full(oracle_lib, inp), "bf16", "side stream")


def test_paged_attention_wrapper(oracle_lib):
    import torch
    inp = workload("tiny")
    dev = gu.to_device(inp)
    out = B.paged_attention(dev["query"], dev["key_pages"], dev["value_pages"],
                            dev["block_table"], dev["context_lens"], inp.page_size,
                            scale=inp.scale, causal=True)
    torch.cuda.synchronize()
    gu.assert_parity(gu.out_to_f64(out), gu.oracle_full(oracle_lib, inp), "bf16", "wrapper")


def test_bounded_wait_gives_up_and_the_context_survives(oracle_lib):
    """The kernels' mbarrier wait on a phase that nothing completes gives up
    after its limit, records PA_FLAG_TIMEOUT and returns; the context stays
    usable (a normal call right after matches the oracle)."""
    import time
    import torch
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert B.pa_selftest_wait_timeout(ws, ws.numel(), 20000) == B.PA_OK
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    _, flag = B.pa_check_device_flag(ws)
    assert flag & B.PA_FLAG_TIMEOUT
    assert waited >= 0.02
    assert B.pa_selftest_wait_timeout(ws, ws.numel(), 3_000_000) == B.PA_ERR_INVALID_ARG
    assert B.pa_selftest_wait_timeout(None, 0, 1000) == B.PA_ERR_WORKSPACE
    inp = synth.workload("tiny")
    out, flag = gu.run(inp)
    assert flag == 0
    gu.assert_parity(gu.out_to_f64(out), gu.oracle_full(oracle_lib, inp), "bf16",
                     "call after a timed-out wait")


def tile_edge_rows(inp, Lt):
    """Every (b, h, l) whose position l is the first or the last of a
    query tile of Lt positions: every query tile of every head."""
    ls = sorted({l for t0 in range(0, inp.L, Lt) for l in (t0, min(t0 + Lt, inp.L) - 1)})
    return np.array([(b, h, l) for b in range(inp.B) for h in range(inp.H_q) for l in ls],
                    dtype=np.int32)


def test_long_prefill_8192(oracle_lib):
    """One causal prefill of 8192 tokens (tile kernel: 128 query-tile pairs
    per kv head, up to 64 key tiles each), checked on the first and last
    position of every query tile (32 positions of 4 heads) for all 32 heads:
    16384 rows, each against its own oracle row."""
    inp = synth.generate(B=1, H_q=32, H_kv=8, L=8192, D=128, page_size=128,
                         context_lens=[8192], k_scale=2.0, seed=701, name="prefill-8192")
    out, _ = gu.run(inp)
    rows = tile_edge_rows(inp, 128 // (inp.H_q // inp.H_kv))
    got = gu.out_to_f64(out)[rows[:, 0], rows[:, 1], rows[:, 2]]
    gu.assert_parity(got, gu.oracle_rows(oracle_lib, inp, rows), "bf16", "prefill 8192")


# ---- the tile schedule's key split and last-tile rows -----------------------------
SPLIT_CASES = [
    # (name, kwargs): few query-tile pairs (keys split into chunks), and a last
    # query tile of at most 8 rows taken by the last full pair's CTA
    ("L65_G4_remainder4", dict(B=3, H_q=16, H_kv=4, L=65, page_size=64,
                               context_lens=[65, 700, 2000])),
    ("L66_G4_remainder8", dict(B=2, H_q=8, H_kv=2, L=66, page_size=128,
                               context_lens=[66, 1500])),
    ("L33_G8_remainder8", dict(B=2, H_q=16, H_kv=2, L=33, page_size=32,
                               context_lens=[40, 900])),
    ("L257_G1_remainder1", dict(B=1, H_q=2, H_kv=2, L=257, page_size=64, context_lens=[600])),
    ("L65_many_pairs_no_split", dict(B=40, H_q=32, H_kv=8, L=65, page_size=128,
                                     ctx_range=(65, 400))),
    ("L200_split_only", dict(B=1, H_q=8, H_kv=2, L=200, page_size=16, context_lens=[3000])),
    # contexts of 128 k + 1 keys: only the last tile's rows see the final key tile
    ("L65_last_key_tile_remainder_only", dict(B=3, H_q=32, H_kv=8, L=65, page_size=128,
                                              context_lens=[129, 257, 1025])),
]


@pytest.mark.parametrize("name,kw", SPLIT_CASES, ids=[c[0] for c in SPLIT_CASES])
@pytest.mark.parametrize("causal", [True, False])
def test_tile_key_split_and_last_tile_rows(oracle_lib, name, kw, causal):
    """Shapes on which the tile schedule splits each pair's keys into chunks
    merged by the combine kernel, and/or gives the rows of a short last query
    tile to the warp-level tensor cores of the last full pair: every element
    against the oracle, on the automatic choice and the forced tiles."""
    inp = synth.generate(D=128, seed=sum(map(ord, name)) + 31, causal=causal, name=name, **kw)
    for sched in (B.PA_SCHED_AUTO, B.PA_SCHED_PREFILL):
        check(oracle_lib, inp, sched, what=f"{name} causal={causal} sched {sched}")


# ---- every GQA group size the tiles take ---------------------------------------
GROUP_CASES = [
    # (name, kwargs): G = H_q / H_kv from 1 to 16, so a query tile holds 128, 64,
    # 32, 16 or 8 positions; the epilogue's tiled stores take rounds of 16 rows of
    # one head (G <= 8) or fall back to direct stores (G = 16), and tiles past
    # the last query rows take the direct path too
    ("G1_Lt128", dict(B=1, H_q=4, H_kv=4, L=300, page_size=128, context_lens=[1000])),
    ("G2_Lt64", dict(B=2, H_q=8, H_kv=4, L=150, page_size=64, context_lens=[150, 700])),
    ("G8_Lt16", dict(B=2, H_q=16, H_kv=2, L=100, page_size=32, context_lens=[100, 300])),
    ("G16_Lt8", dict(B=2, H_q=16, H_kv=1, L=40, page_size=16, context_lens=[40, 200])),
]


@pytest.mark.parametrize("name,kw", GROUP_CASES, ids=[c[0] for c in GROUP_CASES])
@pytest.mark.parametrize("causal", [True, False])
def test_tile_schedule_every_group_size(oracle_lib, name, kw, causal):
    """The tile schedule forced on each GQA group size it takes, causal and
    not: every element against the oracle."""
    inp = synth.generate(D=128, seed=sum(map(ord, name)) + 53, causal=causal, name=name, **kw)
    check(oracle_lib, inp, B.PA_SCHED_PREFILL, what=f"{name} causal={causal}")


# ---- mask=None with more queries than keys ---------------------------------------
NONCAUSAL_LONG_L = [
    # (name, kwargs): L > context_len for some or all sequences, causal off
    ("ps16", dict(B=3, H_q=32, H_kv=8, L=200, page_size=16, context_lens=[50, 130, 7])),
    ("ps128", dict(B=2, H_q=32, H_kv=8, L=300, page_size=128, context_lens=[129, 1])),
    ("gqa1", dict(B=2, H_q=4, H_kv=4, L=40, page_size=8, context_lens=[17, 3])),
    ("decode_rows", dict(B=4, H_q=8, H_kv=2, L=2, page_size=16, context_lens=[1, 1, 5, 2])),
]


@pytest.mark.parametrize("name,kw", NONCAUSAL_LONG_L, ids=[c[0] for c in NONCAUSAL_LONG_L])
@pytest.mark.parametrize("sched", ["auto", "decode", "prefill"])
def test_no_causal_rule_with_more_queries_than_keys(oracle_lib, name, kw, sched):
    """mask=None ("Week 3 Day 5", Keep the Day 4 Interface) lets every query
    row see every key of its context, so L > context_len is a valid call:
    every row is the same softmax over all context_len keys."""
    inp = synth.generate(D=128, seed=sum(map(ord, name)) + 17, causal=False,
                         name=f"nocausal-{name}", **kw)
    assert (inp.context_lens < inp.L).any()
    check(oracle_lib, inp, {"auto": B.PA_SCHED_AUTO, **SCHEDULES}[sched],
          what=f"no causal, L > S, {name}/{sched}")


def test_decode_1024_sequences(oracle_lib):
    """1024 single-token decodes (the page walk's prologue scans 4 blocks of
    sequences; many short segments), checked in full."""
    inp = synth.generate(B=1024, H_q=32, H_kv=8, L=1, D=128, page_size=16,
                         ctx_range=(16, 512), seed=703, name="decode-1024")
    for sched in (B.PA_SCHED_AUTO, B.PA_SCHED_DECODE):
        out, _ = gu.run(inp, sched)
        gu.assert_parity(gu.out_to_f64(out), gu.oracle_full(oracle_lib, inp), "bf16",
                         f"decode 1024 sched {sched}")
