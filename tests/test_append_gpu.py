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
