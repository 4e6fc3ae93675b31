"""ctypes binding of libpaged_attn.so (the C ABI in include/paged_attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  There is no fallback; if the library is missing or
cannot be built, every call raises.  PyTorch provides device memory and
streams.

The functions named ``pa_*`` mirror the C entry points one to one.
``paged_attention`` is the pages' model-facing call ("Week 3 Day 5: Paged
FlashAttention", Keep the Day 4 Interface): it allocates the output and a
workspace with torch and calls ``pa_paged_attention_sched``.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import build as _build

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_BAD_BLOCK_TABLE = 3
PA_ERR_WORKSPACE = 4
PA_ERR_CUDA = 5
PA_ERR_DEVICE_FLAG = 6

PA_BF16 = 0
PA_F32 = 1

PA_SCHED_AUTO = 0
PA_SCHED_DECODE = 1
PA_SCHED_PREFILL = 2

PA_FLAG_BAD_PAGE = 0x1
PA_FLAG_BAD_CONTEXT = 0x2
PA_FLAG_TIMEOUT = 0x4

_lock = threading.Lock()
_lib = None


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        super().__init__(f"{what}: status {status} ({status_str(status)})" if what else
                         f"status {status} ({status_str(status)})")
        self.status = status


class pa_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H_q", ctypes.c_int), ("H_kv", ctypes.c_int),
                ("L", ctypes.c_int), ("D", ctypes.c_int), ("num_pages", ctypes.c_int),
                ("page_size", ctypes.c_int), ("max_pages_per_seq", ctypes.c_int),
                ("dtype", ctypes.c_int)]


def library_path() -> str:
    return _build.LIB


def load(auto_build: bool = True):
    """Loads libpaged_attn.so (building it first if it is stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if auto_build and not _build.up_to_date():
            _build.build()
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        vp, i32p, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t
        sp = ctypes.POINTER(pa_shape)
        lib.pa_workspace_bytes.argtypes = [sp]
        lib.pa_workspace_bytes.restype = sz
        common = [sp, vp, vp, vp, i32p, i32p, ctypes.c_float, ctypes.c_int, vp, vp, sz, vp]
        lib.pa_paged_attention.argtypes = common
        lib.pa_paged_attention.restype = ctypes.c_int
        lib.pa_paged_attention_sched.argtypes = common + [ctypes.c_int]
        lib.pa_paged_attention_sched.restype = ctypes.c_int
        lib.pa_paged_attention_profiled.argtypes = common + [ctypes.c_int, vp, vp]
        lib.pa_paged_attention_profiled.restype = ctypes.c_int
        lib.pa_paged_attention_decode_noalloc.argtypes = [sp, vp, vp, vp, i32p, i32p,
                                                          ctypes.c_float, ctypes.c_int, vp, vp,
                                                          vp]
        lib.pa_paged_attention_decode_noalloc.restype = ctypes.c_int
        lib.pa_gather_debug.argtypes = [sp, vp, vp, i32p, i32p, ctypes.c_int, vp, vp, vp, vp]
        lib.pa_gather_debug.restype = ctypes.c_int
        lib.pa_check_device_flag.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int,
                                             vp]
        lib.pa_check_device_flag.restype = ctypes.c_int
        lib.pa_validate_metadata.argtypes = [sp, i32p, i32p, ctypes.c_int, vp]
        lib.pa_validate_metadata.restype = ctypes.c_int
        lib.pa_choose_schedule.argtypes = [sp]
        lib.pa_choose_schedule.restype = ctypes.c_int
        lib.pa_launch_count.argtypes = [sp, ctypes.c_int]
        lib.pa_launch_count.restype = ctypes.c_int
        lib.pa_paged_attention_masked.argtypes = [sp, vp, vp, vp, i32p, i32p, ctypes.c_float,
                                                  ctypes.c_int, vp, ctypes.c_longlong, vp, vp,
                                                  sz, vp, ctypes.c_int]
        lib.pa_paged_attention_masked.restype = ctypes.c_int
        lib.pa_paged_attention_varlen.argtypes = [sp, vp, vp, vp, i32p, i32p, i32p, ctypes.c_int,
                                                  ctypes.c_float, ctypes.c_int, vp, vp, sz, vp,
                                                  ctypes.c_int]
        lib.pa_paged_attention_varlen.restype = ctypes.c_int
        lib.pa_validate_metadata_varlen.argtypes = [sp, i32p, i32p, i32p, ctypes.c_int,
                                                    ctypes.c_int, vp]
        lib.pa_validate_metadata_varlen.restype = ctypes.c_int
        lib.pa_selftest_wait_timeout.argtypes = [vp, sz, ctypes.c_uint, vp]
        lib.pa_selftest_wait_timeout.restype = ctypes.c_int
        lib.pa_append_kv.argtypes = [sp, vp, vp, vp, vp, i32p, i32p, vp, sz, vp]
        lib.pa_append_kv.restype = ctypes.c_int
        lib.pa_status_str.argtypes = [ctypes.c_int]
        lib.pa_status_str.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_str(status: int) -> str:
    try:
        return load().pa_status_str(int(status)).decode()
    except Exception:  # pragma: no cover - library missing
        return "?"


def _ptr(x):
    """Device/host address of a torch tensor, or an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_shape(B, H_q, H_kv, L, D, num_pages, page_size, max_pages_per_seq, dtype=PA_BF16):
    return pa_shape(int(B), int(H_q), int(H_kv), int(L), int(D), int(num_pages),
                    int(page_size), int(max_pages_per_seq), int(dtype))


def shape_of(query, key_pages, block_table) -> pa_shape:
    """pa_shape of torch tensors laid out as in include/paged_attn.h."""
    import torch
    B, H_q, L, D = query.shape
    P, H_kv, ps, D2 = key_pages.shape
    if D2 != D:
        raise ValueError("query and pages disagree on head dim")
    if query.dtype != key_pages.dtype:
        raise ValueError("query and pages must share a dtype")
    dt = {torch.bfloat16: PA_BF16, torch.float32: PA_F32}.get(query.dtype)
    if dt is None:
        raise ValueError(f"unsupported dtype {query.dtype}")
    return make_shape(B, H_q, H_kv, L, D, P, ps, block_table.shape[1], dt)


# ---- one-to-one C entry points ---------------------------------------------
def pa_workspace_bytes(shape: pa_shape) -> int:
    return int(load().pa_workspace_bytes(ctypes.byref(shape)))


def pa_paged_attention(shape, query, key_pages, value_pages, block_table, context_lens, scale,
                       causal, out, workspace, workspace_bytes, stream=None) -> int:
    return load().pa_paged_attention(
        ctypes.byref(shape), _ptr(query), _ptr(key_pages), _ptr(value_pages), _ptr(block_table),
        _ptr(context_lens), float(scale), int(bool(causal)), _ptr(out), _ptr(workspace),
        int(workspace_bytes), _stream(stream))


def pa_paged_attention_sched(shape, query, key_pages, value_pages, block_table, context_lens,
                             scale, causal, out, workspace, workspace_bytes, stream=None,
                             schedule=PA_SCHED_AUTO) -> int:
    return load().pa_paged_attention_sched(
        ctypes.byref(shape), _ptr(query), _ptr(key_pages), _ptr(value_pages), _ptr(block_table),
        _ptr(context_lens), float(scale), int(bool(causal)), _ptr(out), _ptr(workspace),
        int(workspace_bytes), _stream(stream), int(schedule))


def pa_paged_attention_profiled(shape, query, key_pages, value_pages, block_table, context_lens,
                                scale, causal, out, workspace, workspace_bytes, stream=None,
                                schedule=PA_SCHED_AUTO, event_before=None,
                                event_after=None) -> int:
    """event_before / event_after: raw cudaEvent_t handles (int) or None."""
    return load().pa_paged_attention_profiled(
        ctypes.byref(shape), _ptr(query), _ptr(key_pages), _ptr(value_pages), _ptr(block_table),
        _ptr(context_lens), float(scale), int(bool(causal)), _ptr(out), _ptr(workspace),
        int(workspace_bytes), _stream(stream), int(schedule), event_before, event_after)


def pa_paged_attention_decode_noalloc(shape, query, key_pages, value_pages, block_table,
                                      context_lens, scale, causal, out, device_flag_out=None,
                                      stream=None) -> int:
    """Decode schedule with the library's fixed scratch array instead of a
    caller workspace (for callers that cannot allocate device memory).
    device_flag_out: optional device tensor of one 32-bit word that receives
    this call's PA_FLAG_* bits."""
    return load().pa_paged_attention_decode_noalloc(
        ctypes.byref(shape), _ptr(query), _ptr(key_pages), _ptr(value_pages), _ptr(block_table),
        _ptr(context_lens), float(scale), int(bool(causal)), _ptr(out), _ptr(device_flag_out),
        _stream(stream))


def pa_gather_debug(shape, key_pages, value_pages, block_table, context_lens, max_S, k_dense,
                    v_dense, workspace, stream=None) -> int:
    return load().pa_gather_debug(
        ctypes.byref(shape), _ptr(key_pages), _ptr(value_pages), _ptr(block_table),
        _ptr(context_lens), int(max_S), _ptr(k_dense), _ptr(v_dense), _ptr(workspace),
        _stream(stream))


def pa_paged_attention_masked(shape, query, key_pages, value_pages, block_table, context_lens,
                              scale, causal, mask, mask_S, out, workspace, workspace_bytes,
                              stream=None, schedule=PA_SCHED_AUTO) -> int:
    """mask: fp32 device tensor [B * H_q, L, mask_S] added to the scaled scores."""
    return load().pa_paged_attention_masked(
        ctypes.byref(shape), _ptr(query), _ptr(key_pages), _ptr(value_pages), _ptr(block_table),
        _ptr(context_lens), float(scale), int(bool(causal)), _ptr(mask), int(mask_S), _ptr(out),
        _ptr(workspace), int(workspace_bytes), _stream(stream), int(schedule))


def pa_paged_attention_varlen(shape, query, key_pages, value_pages, block_table, context_lens,
                              cu_q, total_q, scale, causal, out, workspace, workspace_bytes,
                              stream=None, schedule=PA_SCHED_AUTO) -> int:
    """Ragged batch: query/out [total_q, H_q, D] packed by token, cu_q int32
    device tensor [B + 1]; shape.L bounds every sequence's query count."""
    return load().pa_paged_attention_varlen(
        ctypes.byref(shape), _ptr(query), _ptr(key_pages), _ptr(value_pages), _ptr(block_table),
        _ptr(context_lens), _ptr(cu_q), int(total_q), float(scale), int(bool(causal)),
        _ptr(out), _ptr(workspace), int(workspace_bytes), _stream(stream), int(schedule))


def pa_validate_metadata_varlen(shape, block_table, context_lens, cu_q, total_q, causal,
                                stream=None) -> int:
    return load().pa_validate_metadata_varlen(
        ctypes.byref(shape), _ptr(block_table), _ptr(context_lens), _ptr(cu_q), int(total_q),
        int(bool(causal)), _stream(stream))


def pa_selftest_wait_timeout(workspace, workspace_bytes, timeout_us, stream=None) -> int:
    return load().pa_selftest_wait_timeout(_ptr(workspace), int(workspace_bytes),
                                           int(timeout_us), _stream(stream))


def pa_append_kv(shape, k_new, v_new, key_pages, value_pages, block_table, context_lens,
                 workspace, workspace_bytes, stream=None) -> int:
    return load().pa_append_kv(
        ctypes.byref(shape), _ptr(k_new), _ptr(v_new), _ptr(key_pages), _ptr(value_pages),
        _ptr(block_table), _ptr(context_lens), _ptr(workspace), int(workspace_bytes),
        _stream(stream))


def pa_check_device_flag(workspace, clear=False, stream=None):
    """Returns (status, flag word)."""
    f = ctypes.c_uint32(0)
    st = load().pa_check_device_flag(_ptr(workspace), ctypes.byref(f), int(bool(clear)),
                                     _stream(stream))
    return st, int(f.value)


def pa_validate_metadata(shape, block_table, context_lens, causal, stream=None) -> int:
    return load().pa_validate_metadata(ctypes.byref(shape), _ptr(block_table),
                                       _ptr(context_lens), int(bool(causal)), _stream(stream))


def pa_choose_schedule(shape) -> int:
    return int(load().pa_choose_schedule(ctypes.byref(shape)))


def pa_launch_count(shape, schedule=PA_SCHED_AUTO) -> int:
    return int(load().pa_launch_count(ctypes.byref(shape), int(schedule)))


# ---- the pages' model-facing call ------------------------------------------
def new_workspace(shape: pa_shape, device=None):
    """Zeroed workspace for `shape` on `device` (flag word starts at 0)."""
    import torch
    n = pa_workspace_bytes(shape)
    if n == 0:
        raise PagedAttentionError(PA_ERR_INVALID_ARG, "pa_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def paged_attention(query, key_pages, value_pages, block_table, context_lens, page_size,
                    scale=None, causal=True, *, mask=None, out=None, workspace=None,
                    schedule=PA_SCHED_AUTO, stream=None):
    """out[B, H_q, L, D] = softmax(scale * q.K^T + mask over visible keys) . V,
    with K/V read from the paged pool through block_table.  mask: optional
    fp32 CUDA tensor [B * H_q, L, S_mask] (S_mask >= the table's capacity, a
    multiple of 4) added to the scaled scores."""
    import torch
    shape = shape_of(query, key_pages, block_table)
    if shape.page_size != int(page_size):
        raise ValueError("page_size disagrees with key_pages.shape[2]")
    for name, t in (("query", query), ("key_pages", key_pages), ("value_pages", value_pages),
                    ("block_table", block_table), ("context_lens", context_lens)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if block_table.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_table and context_lens must be int32")
    if scale is None:
        scale = 1.0 / math.sqrt(query.shape[-1])
    if out is None:
        out = torch.empty_like(query)
    if workspace is None:
        workspace = new_workspace(shape, query.device)
    if mask is None:
        st = pa_paged_attention_sched(shape, query, key_pages, value_pages, block_table,
                                      context_lens, scale, causal, out, workspace,
                                      workspace.numel(), stream, schedule)
    else:
        if mask.dtype != torch.float32 or not mask.is_cuda or not mask.is_contiguous():
            raise ValueError("mask must be a contiguous fp32 CUDA tensor")
        if mask.dim() != 3 or mask.shape[0] != shape.B * shape.H_q or mask.shape[1] != shape.L:
            raise ValueError("mask must be [B * H_q, L, S_mask]")
        st = pa_paged_attention_masked(shape, query, key_pages, value_pages, block_table,
                                       context_lens, scale, causal, mask, mask.shape[2], out,
                                       workspace, workspace.numel(), stream, schedule)
    if st != PA_OK:
        raise PagedAttentionError(st, "pa_paged_attention")
    return out


def append_kv(k_new, v_new, key_pages, value_pages, block_table, context_lens, *,
              workspace=None, stream=None):
    """Stores k_new/v_new [B, H_kv, L, D] -- the last L positions of each
    context -- in their pages, through block_table (in place)."""
    import torch
    B_, H_kv, L, D = k_new.shape
    P, Hk, ps, Dk = key_pages.shape
    if Hk != H_kv or Dk != D or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [B, H_kv, L, D] matching the pools")
    if k_new.dtype != key_pages.dtype or v_new.dtype != value_pages.dtype:
        raise ValueError("new rows must have the pools' dtype")
    dtype = PA_BF16 if key_pages.dtype == torch.bfloat16 else PA_F32
    shape = make_shape(B_, H_kv, H_kv, L, D, P, ps, block_table.shape[1], dtype)
    if workspace is None:
        workspace = torch.zeros(256, dtype=torch.uint8, device=key_pages.device)
    st = pa_append_kv(shape, k_new.contiguous(), v_new.contiguous(), key_pages, value_pages,
                      block_table, context_lens, workspace, workspace.numel(), stream)
    if st != PA_OK:
        raise PagedAttentionError(st, "pa_append_kv")
    return workspace


def shape_of_varlen(query, key_pages, block_table, max_L) -> pa_shape:
    """pa_shape of a ragged batch: query [total_q, H_q, D] packed by token,
    B = block_table.shape[0] sequences, L = max_L (bounds every L_b)."""
    import torch
    T, H_q, D = query.shape
    P, H_kv, ps, D2 = key_pages.shape
    if D2 != D:
        raise ValueError("query and pages disagree on head dim")
    if query.dtype != key_pages.dtype:
        raise ValueError("query and pages must share a dtype")
    dt = {torch.bfloat16: PA_BF16, torch.float32: PA_F32}.get(query.dtype)
    if dt is None:
        raise ValueError(f"unsupported dtype {query.dtype}")
    return make_shape(block_table.shape[0], H_q, H_kv, max(1, int(max_L)), D, P, ps,
                      block_table.shape[1], dt)


def paged_attention_varlen(query, key_pages, value_pages, block_table, context_lens, cu_q,
                           max_L, page_size, scale=None, causal=True, *, out=None,
                           workspace=None, schedule=PA_SCHED_AUTO, stream=None):
    """Ragged batch: out[total_q, H_q, D]; sequence b's queries are tokens
    cu_q[b] .. cu_q[b+1]-1 of `query` and the last positions of its context.
    max_L bounds every cu_q[b+1] - cu_q[b]."""
    import torch
    shape = shape_of_varlen(query, key_pages, block_table, max_L)
    if shape.page_size != int(page_size):
        raise ValueError("page_size disagrees with key_pages.shape[2]")
    for name, t in (("query", query), ("key_pages", key_pages), ("value_pages", value_pages),
                    ("block_table", block_table), ("context_lens", context_lens), ("cu_q", cu_q)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if block_table.dtype != torch.int32 or context_lens.dtype != torch.int32 or \
            cu_q.dtype != torch.int32:
        raise ValueError("block_table, context_lens and cu_q must be int32")
    if cu_q.numel() != shape.B + 1 or context_lens.numel() != shape.B:
        raise ValueError("cu_q must hold B + 1 offsets and context_lens B lengths")
    if scale is None:
        scale = 1.0 / math.sqrt(query.shape[-1])
    if out is None:
        out = torch.empty_like(query)
    if workspace is None:
        workspace = new_workspace(shape, query.device)
    st = pa_paged_attention_varlen(shape, query, key_pages, value_pages, block_table,
                                   context_lens, cu_q, query.shape[0], scale, causal, out,
                                   workspace, workspace.numel(), stream, schedule)
    if st != PA_OK:
        raise PagedAttentionError(st, "pa_paged_attention_varlen")
    return out
