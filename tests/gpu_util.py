"""Helpers shared by the GPU tests: move seeded inputs to the device, call the
C ABI through the binding, compare with the oracle."""
from __future__ import annotations

import numpy as np

from paged_kv_cache_03_gb300 import binding as B
from paged_kv_cache_03_gb300.synth import PagedInputs, bf16_to_f32

# Parity bars: bf16 outputs within 1e-2 max-abs and 1e-3 mean-abs of the fp64
# oracle; the fp32 control within 1e-5 max-abs.
BF16_MAX_ABS = 1e-2
BF16_MEAN_ABS = 1e-3
F32_MAX_ABS = 1e-5


def to_device(inp: PagedInputs, device="cuda"):
    import torch

    def conv(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if inp.dtype == "bf16":
            t = t.view(torch.bfloat16)
        return t.to(device)

    return dict(query=conv(inp.query), key_pages=conv(inp.key_pages),
                value_pages=conv(inp.value_pages),
                block_table=torch.from_numpy(inp.block_table).to(device),
                context_lens=torch.from_numpy(inp.context_lens).to(device))


def out_to_f64(out) -> np.ndarray:
    import torch
    if out.dtype == torch.bfloat16:
        return bf16_to_f32(out.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    return out.cpu().numpy().astype(np.float64)


class Unsupported(Exception):
    pass


def tiles_take(dtype: str, H_q: int, H_kv: int, page_size: int) -> bool:
    """Whether the tensor-core tile schedule takes a shape (the library's
    documented rule): bf16, H_q/H_kv a divisor of 128 of at most 16, and a
    page size that is a multiple of 8.  A forced tile call outside the rule
    returns PA_ERR_UNSUPPORTED; one inside it must run."""
    G = H_q // H_kv
    return dtype == "bf16" and 1 <= G <= 16 and 128 % G == 0 and page_size % 8 == 0


def run(inp: PagedInputs, schedule=B.PA_SCHED_AUTO, dev=None, workspace=None, check_flag=True,
        block_table=None, context_lens=None):
    """Runs the CUDA path; returns (out tensor, flag word).  Raises
    Unsupported when a forced schedule cannot run this shape."""
    import torch
    dev = dev or to_device(inp)
    bt = dev["block_table"] if block_table is None else block_table
    ctx = dev["context_lens"] if context_lens is None else context_lens
    shape = B.shape_of(dev["query"], dev["key_pages"], bt)
    ws = workspace if workspace is not None else B.new_workspace(shape)
    out = torch.empty_like(dev["query"])
    st = B.pa_paged_attention_sched(shape, dev["query"], dev["key_pages"], dev["value_pages"],
                                    bt, ctx, inp.scale, inp.causal, out, ws, ws.numel(), None,
                                    schedule)
    if st == B.PA_ERR_UNSUPPORTED and schedule != B.PA_SCHED_AUTO:
        raise Unsupported(B.status_str(st))
    assert st == B.PA_OK, f"launch status {st} ({B.status_str(st)})"
    torch.cuda.synchronize()
    st, flag = B.pa_check_device_flag(ws)
    if check_flag:
        assert flag == 0, f"device flag {flag:#x}"
    return out, flag


def oracle_full(lib, inp: PagedInputs) -> np.ndarray:
    return lib.paged_attention(inp.query, inp.key_pages, inp.value_pages, inp.block_table,
                               inp.context_lens, inp.scale, inp.causal)


def oracle_rows(lib, inp: PagedInputs, rows) -> np.ndarray:
    return lib.paged_attention_rows(inp.query, inp.key_pages, inp.value_pages, inp.block_table,
                                    inp.context_lens, inp.scale, inp.causal, rows)


def errors(got: np.ndarray, ref: np.ndarray):
    d = np.abs(got - ref)
    return float(d.max()), float(d.mean())


def assert_parity(got: np.ndarray, ref: np.ndarray, dtype: str, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mx, mean = errors(got, ref)
    if dtype == "bf16":
        assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS, \
            f"{what}: max-abs {mx:.3e} mean-abs {mean:.3e}"
    else:
        assert mx <= F32_MAX_ABS, f"{what}: max-abs {mx:.3e}"
    return mx, mean


def sample_rows(inp: PagedInputs, n: int, seed: int = 0):
    """n (b, h, l) rows: the first and last query of every sequence and head
    band plus uniform random rows."""
    rng = np.random.default_rng(seed)
    rows = set()
    for b in range(inp.B):
        for h in (0, inp.H_q - 1):
            for l in {0, inp.L - 1, inp.L // 2}:
                rows.add((b, h, l))
    while len(rows) < n:
        rows.add((int(rng.integers(inp.B)), int(rng.integers(inp.H_q)),
                  int(rng.integers(inp.L))))
    return np.array(sorted(rows), dtype=np.int32)
