"""K/V append on the GPU (pa_append_kv) vs the oracle's append, bitwise.

The append is a copy through the block table, so the pools after the call
must equal the oracle's pools bit for bit: on the shapes of the named
workloads (the new tokens are the last L positions of each context), on
page-crossing and one-slot pages, fp32, with junk in unused block-table
entries, and with the errors the kernel records instead of faulting.  A last
test appends and then attends: the path reads back exactly what was written.
"""
import numpy as np
import pytest

import gpu_util as gu
from paged_kv_cache_03_gb300 import binding as B
from paged_kv_cache_03_gb300 import synth

pytestmark = pytest.mark.gpu


def _torch(a):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def _bits(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def gpu_append(inp, kn, vn, block_table=None, context_lens=None):
    """Runs pa_append_kv on copies of the pools; returns (k, v, flag)."""
    import torch
    kp, vp = _torch(inp.key_pages), _torch(inp.value_pages)
    bt = _torch(inp.block_table if block_table is None else block_table)
    ctx = _torch(inp.context_lens if context_lens is None else context_lens)
    H_kv = inp.key_pages.shape[1]
    L = kn.shape[2]
    sh = B.make_shape(inp.B, H_kv, H_kv, L, inp.D, inp.num_pages, inp.page_size,
                      bt.shape[1], B.PA_BF16 if inp.dtype == "bf16" else B.PA_F32)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    st = B.pa_append_kv(sh, _torch(kn), _torch(vn), kp, vp, bt, ctx, ws, ws.numel())
    assert st == B.PA_OK, B.status_str(st)
    torch.cuda.synchronize()
    _, flag = B.pa_check_device_flag(ws)
    return _bits(kp), _bits(vp), flag


CASES = [
    # (workload, overrides, new tokens L, seed)
    ("tiny", {}, 5, 301),
    ("decode", {}, 1, 302),
    ("prefill", {}, 2048, 303),
    ("tails", {}, 65, 304),
    ("tiny", dict(page_size=1, num_pages=None), 3, 305),
    ("tiny", dict(page_size=3, num_pages=None), 5, 306),
    ("long_decode", dict(B=2, context_lens=[32768] * 2, num_pages=4096), 1, 307),
]


@pytest.mark.parametrize("name,kw,L,seed", CASES, ids=[f"{c[0]}-L{c[2]}-{c[3]}" for c in CASES])
def test_append_matches_oracle_bitwise(oracle_lib, name, kw, L, seed):
    inp = synth.workload(name, **kw)
    kn, vn = synth.new_kv(inp.B, inp.key_pages.shape[1], L, inp.D, seed)
    k_ref, v_ref, st = oracle_lib.append_kv(kn, vn, inp.key_pages, inp.value_pages,
                                            inp.block_table, inp.context_lens)
    assert st == 0
    k, v, flag = gpu_append(inp, kn, vn)
    assert flag == 0
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def test_append_fp32(oracle_lib):
    inp = synth.workload("tails", dtype="f32", B=3, ctx_range=(100, 700), num_pages=None)
    kn, vn = synth.new_kv(inp.B, inp.key_pages.shape[1], 65, inp.D, 311, dtype="f32")
    k_ref, v_ref, st = oracle_lib.append_kv(kn, vn, inp.key_pages, inp.value_pages,
                                            inp.block_table, inp.context_lens)
    assert st == 0
    k, v, flag = gpu_append(inp, kn, vn)
    assert flag == 0
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def test_append_never_reads_unused_table_entries(oracle_lib):
    inp = synth.workload("decode")
    kn, vn = synth.new_kv(inp.B, inp.key_pages.shape[1], 1, inp.D, 321)
    bt = inp.block_table.copy()
    for b in range(inp.B):
        npg = (int(inp.context_lens[b]) + inp.page_size - 1) // inp.page_size
        bt[b, npg:] = -123456
    k_ref, v_ref, _ = oracle_lib.append_kv(kn, vn, inp.key_pages, inp.value_pages,
                                           inp.block_table, inp.context_lens)
    k, v, flag = gpu_append(inp, kn, vn, block_table=bt)
    assert flag == 0
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def test_append_errors_are_recorded_and_skipped(oracle_lib):
    inp = synth.workload("tiny")  # contexts 13 and 40, L = 5 new tokens
    kn, vn = synth.new_kv(inp.B, inp.key_pages.shape[1], 5, inp.D, 331)
    ctx = inp.context_lens.copy()
    ctx[0] = 4  # shorter than the new tokens
    k_ref, v_ref, st = oracle_lib.append_kv(kn, vn, inp.key_pages, inp.value_pages,
                                            inp.block_table, ctx)
    assert st == 1
    k, v, flag = gpu_append(inp, kn, vn, context_lens=ctx)
    assert flag & B.PA_FLAG_BAD_CONTEXT
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)
    bt = inp.block_table.copy()
    bt[1, 2] = inp.num_pages + 9  # positions 35..39 of sequence 1 lie on logical page 2
    k_ref, v_ref, st = oracle_lib.append_kv(kn, vn, inp.key_pages, inp.value_pages, bt,
                                            inp.context_lens)
    assert st == 3
    k, v, flag = gpu_append(inp, kn, vn, block_table=bt)
    assert flag & B.PA_FLAG_BAD_PAGE
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def test_append_rejects_bad_arguments():
    import torch
    sh = B.make_shape(2, 4, 2, 1, 64, 16, 16, 3)  # D != 128
    t = torch.zeros(64, dtype=torch.uint8, device="cuda")
    assert B.pa_append_kv(sh, t, t, t, t, t, t, t, 256) == B.PA_ERR_UNSUPPORTED
    sh = B.make_shape(2, 4, 2, 1, 128, 16, 16, 3)
    assert B.pa_append_kv(sh, t, t, t, t, t, t, None, 0) == B.PA_ERR_WORKSPACE
    assert B.pa_append_kv(sh, None, t, t, t, t, t, t, 256) == B.PA_ERR_INVALID_ARG


def test_append_then_attend(oracle_lib):
    """Append the new tokens' K/V, then run the path over the appended pool:
    the output matches the oracle over the oracle-appended pool."""
    import torch
    inp = synth.workload("tails")
    H_kv = inp.key_pages.shape[1]
    kn, vn = synth.new_kv(inp.B, H_kv, inp.L, inp.D, 341)
    k_ref, v_ref, st = oracle_lib.append_kv(kn, vn, inp.key_pages, inp.value_pages,
                                            inp.block_table, inp.context_lens)
    assert st == 0
    dev = gu.to_device(inp)
    sh = B.make_shape(inp.B, H_kv, H_kv, inp.L, inp.D, inp.num_pages, inp.page_size,
                      inp.block_table.shape[1])
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert B.pa_append_kv(sh, _torch(kn), _torch(vn), dev["key_pages"], dev["value_pages"],
                          dev["block_table"], dev["context_lens"], ws, 256) == B.PA_OK
    appended = synth.PagedInputs(inp.query, k_ref, v_ref, inp.block_table, inp.context_lens,
                                 inp.page_size, inp.scale, inp.causal, inp.dtype, "appended")
    out, _ = gu.run(appended, dev=dev)
    gu.assert_parity(gu.out_to_f64(out), gu.oracle_full(oracle_lib, appended), "bf16",
                     "append then attend")


def test_prefill_then_decode_through_the_library(oracle_lib):
    """The serving flow on one pool, every step through the library: append
    the prompts' K/V and attend over them (causal prefill), then append one
    token per sequence and attend again (decode), then a ragged step where one
    sequence decodes and the other takes a prefill chunk.  Each output matches
    the oracle over the oracle's own appended pools."""
    import torch
    H_q, H_kv, D, ps = 8, 2, 128, 16
    B_, L0 = 2, 70                            # two prompts of 70 tokens
    npg = 8                                   # pages per sequence: room for 128 tokens
    rng = np.random.default_rng(480)
    pool = synth.generate(B_, H_q, H_kv, 1, D, ps, context_lens=[npg * ps] * B_, seed=481)
    kp_ref, vp_ref = pool.key_pages.copy(), pool.value_pages.copy()
    bt = pool.block_table.copy()
    kp_dev, vp_dev = _torch(kp_ref), _torch(vp_ref)
    bt_dev = _torch(bt)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")

    def append(ctx, L, seed):
        nonlocal kp_ref, vp_ref
        kn, vn = synth.new_kv(B_, H_kv, L, D, seed)
        kp_ref, vp_ref, st = oracle_lib.append_kv(kn, vn, kp_ref, vp_ref, bt, ctx)
        assert st == 0
        sh = B.make_shape(B_, H_kv, H_kv, L, D, kp_ref.shape[0], ps, bt.shape[1])
        assert B.pa_append_kv(sh, _torch(kn), _torch(vn), kp_dev, vp_dev, bt_dev, _torch(ctx),
                              ws, 256) == B.PA_OK

    def attend(ctx, L, seed, what):
        q = synth._normal(rng, (B_, H_q, L, D), "bf16")
        inp = synth.PagedInputs(q, kp_ref, vp_ref, bt, ctx, ps, float(np.float32(D ** -0.5)),
                                True, "bf16", what)
        dev = dict(query=_torch(q), key_pages=kp_dev, value_pages=vp_dev, block_table=bt_dev,
                   context_lens=_torch(ctx))
        out, flag = gu.run(inp, dev=dev)
        assert flag == 0
        gu.assert_parity(gu.out_to_f64(out), gu.oracle_full(oracle_lib, inp), "bf16", what)

    # prefill: both prompts' K/V appended, then causal attention over them
    ctx = np.array([L0, L0], dtype=np.int32)
    append(ctx, L0, 482)
    attend(ctx, L0, 483, "prefill")
    for step in range(3):                     # three decode steps
        ctx = ctx + 1
        append(ctx, 1, 484 + step)
        attend(ctx, 1, 490 + step, f"decode step {step}")
    # ragged step: sequence 0 decodes one token, sequence 1 takes 20 tokens
    lens = np.array([1, 20])
    kn_all, vn_all = [], []
    new_ctx = ctx + lens.astype(np.int32)
    for b in range(B_):
        kn, vn = synth.new_kv(1, H_kv, int(lens[b]), D, 500 + b)
        one = np.ascontiguousarray(bt[b:b + 1])
        kp_ref, vp_ref, st = oracle_lib.append_kv(kn, vn, kp_ref, vp_ref, one, new_ctx[b:b + 1])
        assert st == 0
        sh = B.make_shape(1, H_kv, H_kv, int(lens[b]), D, kp_ref.shape[0], ps, bt.shape[1])
        assert B.pa_append_kv(sh, _torch(kn), _torch(vn), kp_dev, vp_dev, _torch(one),
                              _torch(new_ctx[b:b + 1]), ws, 256) == B.PA_OK
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = synth._normal(rng, (int(cu[-1]), H_q, D), "bf16")
    r = synth.RaggedInputs(q, kp_ref, vp_ref, bt, new_ctx, cu, ps, float(np.float32(D ** -0.5)),
                           True, "bf16", "ragged step")
    ref = oracle_lib.paged_attention_varlen(q, kp_ref, vp_ref, bt, new_ctx, cu, r.scale, True)
    shape = B.shape_of_varlen(_torch(q), kp_dev, bt_dev, int(lens.max()))
    out = torch.zeros((int(cu[-1]), H_q, D), dtype=torch.bfloat16, device="cuda")
    wsv = B.new_workspace(shape)
    assert B.pa_paged_attention_varlen(shape, _torch(q), kp_dev, vp_dev, bt_dev, _torch(new_ctx),
                                       _torch(cu), int(cu[-1]), r.scale, True, out, wsv,
                                       wsv.numel()) == B.PA_OK
    torch.cuda.synchronize()
    gu.assert_parity(gu.out_to_f64(out), ref, "bf16", "ragged step after decode")
