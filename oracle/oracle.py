"""ctypes front end of the fp64 CPU oracle (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this module.  It builds
``pa_oracle.c`` with gcc (no CUDA) and calls it on numpy arrays.  Nothing in
the CUDA library imports it, and it imports nothing from that library.

The oracle computes exact paged attention by its plain definition: gather the
history through the block table ("Week 3 Day 5: Paged FlashAttention", Task 1),
then one stable softmax over the visible scores and the weighted value sum
("Week 2 Day 5: Fused Decode Attention", Task 1; causal rule from "Week 3 Day
5", Task 2), all in fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_cache: dict[int, "OracleLib"] = {}

ORACLE_OK = 0
ORACLE_ERR_INVALID_ARG = 1
ORACLE_ERR_BAD_BLOCK_TABLE = 3


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle returned status {code}")
        self.code = code


class _Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("B", "H_q", "H_kv", "L", "D", "num_pages", "page_size",
                 "max_pages_per_seq", "dtype")]


def _lib_path(mutant: int) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mut{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compiles the oracle with gcc into oracle/_build/ and returns the path.

    -ffp-contract=off keeps every multiply and add separately rounded, so the
    x86 and Arm builds give bit-identical results."""
    out = _lib_path(mutant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)
            and os.path.getmtime(out) >= os.path.getmtime(os.path.join(_HERE, "pa_oracle.h"))):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", f"-DORACLE_MUTANT={mutant}", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)  # no OpenMP: serial
    os.replace(tmp, out)
    return out


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleLib:
    def __init__(self, path: str):
        self.path = path
        self.lib = ctypes.CDLL(path)
        vp, ip = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)
        dp = ctypes.POINTER(ctypes.c_double)
        sp = ctypes.POINTER(_Shape)
        self.lib.oracle_gather.argtypes = [sp, vp, vp, ip, ip, ctypes.c_int, dp, dp]
        self.lib.oracle_gather.restype = ctypes.c_int
        self.lib.oracle_paged_attention.argtypes = [sp, vp, vp, vp, ip, ip, ctypes.c_double,
                                                    ctypes.c_int, dp, ctypes.c_int]
        self.lib.oracle_paged_attention.restype = ctypes.c_int
        self.lib.oracle_paged_attention_rows.argtypes = [
            sp, vp, vp, vp, ip, ip, ctypes.c_double, ctypes.c_int, ip, ctypes.c_int, dp,
            ctypes.c_int]
        self.lib.oracle_paged_attention_rows.restype = ctypes.c_int
        fp = ctypes.POINTER(ctypes.c_float)
        self.lib.oracle_paged_attention_masked.argtypes = [
            sp, vp, vp, vp, ip, ip, ctypes.c_double, ctypes.c_int, fp, ctypes.c_int, dp,
            ctypes.c_int]
        self.lib.oracle_paged_attention_masked.restype = ctypes.c_int
        self.lib.oracle_paged_attention_varlen.argtypes = [
            sp, vp, vp, vp, ip, ip, ip, ctypes.c_int, ctypes.c_double, ctypes.c_int, dp,
            ctypes.c_int]
        self.lib.oracle_paged_attention_varlen.restype = ctypes.c_int
        self.lib.oracle_append_kv.argtypes = [sp, vp, vp, vp, vp, ip, ip]
        self.lib.oracle_append_kv.restype = ctypes.c_int

    @staticmethod
    def _shape(query, key_pages, block_table, L=None, H_q=None, B=None):
        dtype = 0 if key_pages.dtype == np.uint16 else 1
        P, H_kv, ps, D = key_pages.shape
        Bq, Hq, Lq, Dq = query.shape
        assert Dq == D
        return _Shape(B=Bq, H_q=Hq, H_kv=H_kv, L=Lq, D=D, num_pages=P, page_size=ps,
                      max_pages_per_seq=block_table.shape[1], dtype=dtype)

    @staticmethod
    def _check_arrays(*arrs):
        for a in arrs:
            assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"

    def paged_attention(self, query, key_pages, value_pages, block_table, context_lens,
                        scale: float, causal: bool, num_threads: int = 0,
                        mask=None) -> np.ndarray:
        """mask: optional float32 additive mask [B * H_q, L, S_mask] over
        logical key positions (S_mask >= every context length)."""
        self._check_arrays(query, key_pages, value_pages, block_table, context_lens)
        sh = self._shape(query, key_pages, block_table)
        out = np.zeros(query.shape, dtype=np.float64)
        if mask is None:
            st = self.lib.oracle_paged_attention(
                ctypes.byref(sh), _ptr(query), _ptr(key_pages), _ptr(value_pages),
                block_table.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                context_lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                float(scale), int(bool(causal)),
                out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(num_threads))
        else:
            mask = np.ascontiguousarray(mask, dtype=np.float32)
            B, Hq, L, _ = query.shape
            assert mask.ndim == 3 and mask.shape[:2] == (B * Hq, L)
            st = self.lib.oracle_paged_attention_masked(
                ctypes.byref(sh), _ptr(query), _ptr(key_pages), _ptr(value_pages),
                block_table.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                context_lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                float(scale), int(bool(causal)),
                mask.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), int(mask.shape[2]),
                out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(num_threads))
        if st != ORACLE_OK:
            raise OracleError(st)
        return out

    def paged_attention_rows(self, query, key_pages, value_pages, block_table, context_lens,
                             scale: float, causal: bool, rows, num_threads: int = 0) -> np.ndarray:
        """rows: int array [n, 3] of (b, q_head, l); returns [n, D] float64."""
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
        self._check_arrays(query, key_pages, value_pages, block_table, context_lens)
        sh = self._shape(query, key_pages, block_table)
        out = np.zeros((rows.shape[0], query.shape[3]), dtype=np.float64)
        st = self.lib.oracle_paged_attention_rows(
            ctypes.byref(sh), _ptr(query), _ptr(key_pages), _ptr(value_pages),
            block_table.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            context_lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            float(scale), int(bool(causal)),
            rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), rows.shape[0],
            out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), int(num_threads))
        if st != ORACLE_OK:
            raise OracleError(st)
        return out

    def gather(self, key_pages, value_pages, block_table, context_lens, max_S: int,
               H_q: int | None = None, L: int = 1):
        """Dense [B, H_kv, max_S, D] float64 K and V gathered through the table."""
        self._check_arrays(key_pages, value_pages, block_table, context_lens)
        P, H_kv, ps, D = key_pages.shape
        B = block_table.shape[0]
        sh = _Shape(B=B, H_q=H_q or H_kv, H_kv=H_kv, L=L, D=D, num_pages=P, page_size=ps,
                    max_pages_per_seq=block_table.shape[1],
                    dtype=0 if key_pages.dtype == np.uint16 else 1)
        k = np.zeros((B, H_kv, max_S, D), dtype=np.float64)
        v = np.zeros_like(k)
        st = self.lib.oracle_gather(
            ctypes.byref(sh), _ptr(key_pages), _ptr(value_pages),
            block_table.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            context_lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), int(max_S),
            k.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            v.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
        if st != ORACLE_OK:
            raise OracleError(st)
        return k, v


    def paged_attention_varlen(self, query, key_pages, value_pages, block_table, context_lens,
                               cu_q, scale: float, causal: bool, max_L: int | None = None,
                               num_threads: int = 0) -> np.ndarray:
        """Ragged batch: query [total_q, H_q, D] packed by token, cu_q [B + 1]
        query offsets (sequence b owns tokens cu_q[b] .. cu_q[b+1]-1, the
        last positions of its context); returns [total_q, H_q, D] float64."""
        cu_q = np.ascontiguousarray(cu_q, dtype=np.int32)
        self._check_arrays(query, key_pages, value_pages, block_table, context_lens)
        P, H_kv, ps, D = key_pages.shape
        T, Hq, Dq = query.shape
        assert Dq == D
        B = block_table.shape[0]
        assert cu_q.shape == (B + 1,) and context_lens.shape == (B,)
        lens = np.diff(cu_q)
        if max_L is None:
            max_L = max(1, int(lens.max()) if B else 1)
        sh = _Shape(B=B, H_q=Hq, H_kv=H_kv, L=int(max_L), D=D, num_pages=P, page_size=ps,
                    max_pages_per_seq=block_table.shape[1],
                    dtype=0 if key_pages.dtype == np.uint16 else 1)
        out = np.zeros(query.shape, dtype=np.float64)
        st = self.lib.oracle_paged_attention_varlen(
            ctypes.byref(sh), _ptr(query), _ptr(key_pages), _ptr(value_pages),
            block_table.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            context_lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            cu_q.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), int(T), float(scale),
            int(bool(causal)), out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            int(num_threads))
        if st != ORACLE_OK:
            raise OracleError(st)
        return out

    def append_kv(self, k_new, v_new, key_pages, value_pages, block_table, context_lens):
        """Copies of the pools after writing the new tokens' K/V rows
        (k_new/v_new [B, H_kv, L, D], the last L positions of each context)
        through the block table.  Returns (key_pages, value_pages, status);
        status is ORACLE_OK or the error of a skipped sequence / token."""
        self._check_arrays(k_new, v_new, key_pages, value_pages, block_table, context_lens)
        assert k_new.dtype == key_pages.dtype and v_new.dtype == value_pages.dtype
        P, H_kv, ps, D = key_pages.shape
        B, Hk, L, Dn = k_new.shape
        assert Hk == H_kv and Dn == D and v_new.shape == k_new.shape
        sh = _Shape(B=B, H_q=H_kv, H_kv=H_kv, L=L, D=D, num_pages=P, page_size=ps,
                    max_pages_per_seq=block_table.shape[1],
                    dtype=0 if key_pages.dtype == np.uint16 else 1)
        kp = key_pages.copy()
        vp = value_pages.copy()
        st = self.lib.oracle_append_kv(
            ctypes.byref(sh), _ptr(k_new), _ptr(v_new), _ptr(kp), _ptr(vp),
            block_table.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            context_lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
        return kp, vp, int(st)


def load(mutant: int = 0) -> OracleLib:
    with _lock:
        if mutant not in _cache:
            _cache[mutant] = OracleLib(build(mutant))
        return _cache[mutant]


def host_cores() -> int:
    """Threads the oracle's OpenMP loops use by default on this host."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
