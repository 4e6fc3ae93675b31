"""The C-ABI calls can be captured in a CUDA graph and replayed (a serving
loop captures its decode step once): each path -- the page walk with its
combine, the tensor-core tiles, and a mixed ragged batch (pair plan, tiles
and the page walk launched as their programmatic dependent) -- gives bitwise
the output of a direct call, replay after replay."""
import numpy as np
import pytest

import gpu_util as gu
from paged_kv_cache_03_gb300 import binding as B
from paged_kv_cache_03_gb300 import synth

pytestmark = pytest.mark.gpu


def _bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy()


def _capture(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


@pytest.mark.parametrize("name,sched", [("decode", B.PA_SCHED_DECODE),
                                        ("tails", B.PA_SCHED_PREFILL)])
def test_uniform_call_in_a_graph(name, sched):
    import torch
    inp = synth.workload(name)
    dev = gu.to_device(inp)
    shape = B.shape_of(dev["query"], dev["key_pages"], dev["block_table"])
    ws = B.new_workspace(shape)
    out = torch.empty_like(dev["query"])
    stream = torch.cuda.Stream()

    def call():
        st = B.pa_paged_attention_sched(shape, dev["query"], dev["key_pages"],
                                        dev["value_pages"], dev["block_table"],
                                        dev["context_lens"], inp.scale, inp.causal, out, ws,
                                        ws.numel(), torch.cuda.current_stream(), sched)
        assert st == B.PA_OK

    with torch.cuda.stream(stream):
        call()  # first call outside the capture (one-time kernel attributes)
    torch.cuda.synchronize()
    ref = _bits(out)
    out.zero_()
    g = _capture(call, stream)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(_bits(out), ref)
    assert B.pa_check_device_flag(ws)[1] == 0


def test_mixed_ragged_call_in_a_graph():
    import torch
    r = synth.mixed_workload()
    conv = lambda a, bf=False: (torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16)  # noqa: E731
                                if bf else torch.from_numpy(np.ascontiguousarray(a))).cuda()
    q, kp, vp = conv(r.query, True), conv(r.key_pages, True), conv(r.value_pages, True)
    bt, ctx, cu = conv(r.block_table), conv(r.context_lens), conv(r.cu_q)
    shape = B.shape_of_varlen(q, kp, bt, r.max_L)
    ws = B.new_workspace(shape)
    out = torch.empty_like(q)
    T = int(r.cu_q[-1])
    stream = torch.cuda.Stream()

    def call():
        st = B.pa_paged_attention_varlen(shape, q, kp, vp, bt, ctx, cu, T, r.scale, r.causal,
                                         out, ws, ws.numel(), torch.cuda.current_stream())
        assert st == B.PA_OK

    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    ref = _bits(out)
    g = _capture(call, stream)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(_bits(out), ref)
    assert B.pa_check_device_flag(ws)[1] == 0
