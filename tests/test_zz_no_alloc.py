"""The allocation-free decode entry point (pa_paged_attention_decode_noalloc).

Some callers cannot allocate device memory: a serving process whose free HBM
is all owned by its K/V page pool and caching allocator, or a latency-bound
decode loop that cannot afford the device-wide synchronisation cudaMalloc and
cudaFree may cause.  For them the library keeps its decode scratch in one
fixed device array.  These tests call that entry point through the C ABI and
check it against the regular entry point running the same decode schedule,
on consecutive calls that reuse the shared scratch, and check that a shape
needing more scratch than the fixed maximum is refused.  This file is
collected last on purpose.
"""
import numpy as np
import pytest

import gpu_util as gu
from paged_kv_cache_03_gb300 import binding as B
from paged_kv_cache_03_gb300 import synth

pytestmark = pytest.mark.gpu


def _inputs():
    return [
        synth.workload("decode"),
        synth.generate(B=3, H_q=8, H_kv=2, L=65, D=128, page_size=128,
                       context_lens=[1000, 777, 65], seed=21, name="tails-small"),
        synth.workload("tiny"),
    ]


def test_noalloc_matches_regular_entry_point_on_consecutive_calls(oracle_lib):
    """Two calls in a row per input (the second reuses the scratch the first
    left behind), for three inputs in turn: each output is bitwise the
    regular entry point's on the same (decode) schedule, whose split does
    not depend on which block runs a chunk, and within the bf16 bars of the
    oracle."""
    import torch
    for inp in _inputs():
        dev = gu.to_device(inp)
        shape = B.shape_of(dev["query"], dev["key_pages"], dev["block_table"])
        ref, _ = gu.run(inp, B.PA_SCHED_DECODE, dev=dev)
        want = gu.oracle_full(oracle_lib, inp)
        for call in range(2):
            out = torch.full_like(dev["query"], float("nan"))
            flag = torch.full((1,), -1, dtype=torch.int32, device="cuda")
            st = B.pa_paged_attention_decode_noalloc(
                shape, dev["query"], dev["key_pages"], dev["value_pages"], dev["block_table"],
                dev["context_lens"], inp.scale, inp.causal, out, flag)
            assert st == B.PA_OK, B.status_str(st)
            torch.cuda.synchronize()
            assert int(flag.item()) == 0
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
                f"{inp.name} call {call}: differs from the regular entry point"
            gu.assert_parity(gu.out_to_f64(out), want, "bf16", f"{inp.name} call {call}")


def test_noalloc_reports_this_calls_errors_only():
    import torch
    inp = synth.workload("tiny")
    dev = gu.to_device(inp)
    shape = B.shape_of(dev["query"], dev["key_pages"], dev["block_table"])
    out = torch.empty_like(dev["query"])
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = dev["context_lens"].clone()
    bad[1] = 0
    st = B.pa_paged_attention_decode_noalloc(shape, dev["query"], dev["key_pages"],
                                             dev["value_pages"], dev["block_table"], bad,
                                             inp.scale, True, out, flag)
    assert st == B.PA_OK
    torch.cuda.synchronize()
    assert int(flag.item()) & B.PA_FLAG_BAD_CONTEXT
    st = B.pa_paged_attention_decode_noalloc(shape, dev["query"], dev["key_pages"],
                                             dev["value_pages"], dev["block_table"],
                                             dev["context_lens"], inp.scale, True, out, flag)
    assert st == B.PA_OK
    torch.cuda.synchronize()
    assert int(flag.item()) == 0


def test_noalloc_refuses_shapes_beyond_its_scratch():
    import torch
    # 20000 sequences x 8 kv heads need far more than the fixed 8 MiB of partials
    shape = B.make_shape(20000, 32, 8, 1, 128, 64, 128, 2, B.PA_BF16)
    assert B.pa_workspace_bytes(shape) > (8 << 20)
    t = torch.zeros(16, dtype=torch.uint8, device="cuda")
    st = B.pa_paged_attention_decode_noalloc(shape, t, t, t, t, t, 0.1, True, t, None)
    assert st == B.PA_ERR_WORKSPACE


def test_noalloc_rejected_calls_enqueue_nothing():
    """A call refused by the argument checks writes neither the caller's flag
    nor the shared scratch: the flag word a previous call left (here: a bad
    context length) is still there for the next flag copy to see."""
    import torch
    inp = synth.workload("tiny")
    dev = gu.to_device(inp)
    shape = B.shape_of(dev["query"], dev["key_pages"], dev["block_table"])
    out = torch.empty_like(dev["query"])
    flag = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for scale in (float("nan"), -1.0, float("inf")):
        st = B.pa_paged_attention_decode_noalloc(shape, dev["query"], dev["key_pages"],
                                                 dev["value_pages"], dev["block_table"],
                                                 dev["context_lens"], scale, True, out, flag)
        assert st == B.PA_ERR_INVALID_ARG
    st = B.pa_paged_attention_decode_noalloc(shape, dev["query"][..., 1:], dev["key_pages"],
                                             dev["value_pages"], dev["block_table"],
                                             dev["context_lens"], inp.scale, True, out, flag)
    assert st == B.PA_ERR_INVALID_ARG  # query not 16-byte aligned
    torch.cuda.synchronize()
    assert int(flag.item()) == 12345
