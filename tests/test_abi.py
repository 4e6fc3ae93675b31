"""The C-ABI library loads, exports every declared entry point, and rejects
bad arguments on the host before any CUDA call (CPU only)."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_03_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            with open(os.path.join(ROOT, "include", fn)) as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(pa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("pa_paged_attention", "pa_paged_attention_sched", "pa_workspace_bytes",
              "pa_gather_debug", "pa_check_device_flag", "pa_validate_metadata",
              "pa_status_str"):
        assert n in names


def test_library_exports_every_declared_symbol():
    B.load()
    lib = ctypes.CDLL(B.library_path())
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def good_shape(**kw):
    d = dict(B=2, H_q=4, H_kv=2, L=5, D=128, num_pages=16, page_size=16, max_pages_per_seq=3,
             dtype=B.PA_BF16)
    d.update(kw)
    return B.make_shape(**d)


FAKE = 1 << 20  # 16-byte aligned non-null addresses: never dereferenced on a failed check


@pytest.mark.parametrize("kw,status", [
    (dict(H_q=3, H_kv=2), B.PA_ERR_INVALID_ARG),
    (dict(B=0), B.PA_ERR_INVALID_ARG),
    (dict(L=0), B.PA_ERR_INVALID_ARG),
    (dict(page_size=0), B.PA_ERR_INVALID_ARG),
    (dict(num_pages=0), B.PA_ERR_INVALID_ARG),
    (dict(dtype=7), B.PA_ERR_INVALID_ARG),
    (dict(D=64), B.PA_ERR_UNSUPPORTED),
    (dict(num_pages=1 << 20, page_size=1 << 12), B.PA_ERR_UNSUPPORTED),
])
def test_bad_shapes_are_rejected_on_host(kw, status):
    sh = good_shape(**kw)
    st = B.pa_paged_attention_sched(sh, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, 1, FAKE, FAKE,
                                    1 << 20, 0, B.PA_SCHED_DECODE)
    assert st == status
    assert B.pa_workspace_bytes(sh) == 0


@pytest.mark.parametrize("which", ["query", "key", "value", "bt", "ctx", "out"])
def test_null_pointers_are_rejected(which):
    ptrs = dict(query=FAKE, key=FAKE, value=FAKE, bt=FAKE, ctx=FAKE, out=FAKE)
    ptrs[which] = 0
    st = B.pa_paged_attention(good_shape(), ptrs["query"], ptrs["key"], ptrs["value"],
                              ptrs["bt"], ptrs["ctx"], 0.1, 1, ptrs["out"], FAKE, 1 << 20, 0)
    assert st == B.PA_ERR_INVALID_ARG


def test_misaligned_pointers_are_rejected():
    st = B.pa_paged_attention(good_shape(), FAKE + 8, FAKE, FAKE, FAKE, FAKE, 0.1, 1, FAKE,
                              FAKE, 1 << 20, 0)
    assert st == B.PA_ERR_INVALID_ARG


def test_missing_workspace_is_rejected():
    st = B.pa_paged_attention(good_shape(), FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, 1, FAKE, 0, 0, 0)
    assert st == B.PA_ERR_WORKSPACE


@pytest.mark.parametrize("scale", [float("nan"), -0.1, -1e-30, float("inf"), float("-inf")])
def test_bad_scale_is_rejected(scale):
    """scale is a softmax temperature: finite and >= 0 (checked on the host,
    before anything is enqueued, in the uniform, masked and ragged calls)."""
    st = B.pa_paged_attention(good_shape(), FAKE, FAKE, FAKE, FAKE, FAKE, scale, 1, FAKE,
                              FAKE, 1 << 20, 0)
    assert st == B.PA_ERR_INVALID_ARG
    st = B.pa_paged_attention_masked(good_shape(), FAKE, FAKE, FAKE, FAKE, FAKE, scale, 1, FAKE,
                                     1 << 12, FAKE, FAKE, 1 << 20, 0, B.PA_SCHED_AUTO)
    assert st == B.PA_ERR_INVALID_ARG
    st = B.pa_paged_attention_varlen(good_shape(), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, scale,
                                     1, FAKE, FAKE, 1 << 20, 0, B.PA_SCHED_AUTO)
    assert st == B.PA_ERR_INVALID_ARG


def test_unknown_schedule_is_rejected():
    st = B.pa_paged_attention_sched(good_shape(), FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, 1, FAKE,
                                    FAKE, 1 << 20, 0, 9)
    assert st == B.PA_ERR_INVALID_ARG


def test_schedule_rule():
    """The dispatch follows the measured crossover of the operator sweep."""
    decode_cfg = dict(B=64, H_q=32, H_kv=8, num_pages=2048, page_size=128, max_pages_per_seq=32)
    # up to 4 query rows per kv head over a real batch: the page walk
    assert B.pa_choose_schedule(good_shape(L=1, **decode_cfg)) == B.PA_SCHED_DECODE
    assert B.pa_choose_schedule(good_shape(L=1, **{**decode_cfg, "H_q": 8})) == B.PA_SCHED_DECODE
    # more than 4 rows per kv head: the tensor-core tiles
    assert B.pa_choose_schedule(good_shape(L=2, **decode_cfg)) == B.PA_SCHED_PREFILL
    assert B.pa_choose_schedule(good_shape(L=2048, **decode_cfg)) == B.PA_SCHED_PREFILL
    # a tiny call: the tile schedule's lower fixed cost wins even for one row
    assert B.pa_choose_schedule(good_shape(L=1)) == B.PA_SCHED_PREFILL
    # at most 8 (sequence, kv head) pairs: the tiles split each pair's keys over
    # SMs of their own, at any context (B = 1, 16384 keys: tiles 33 us, page walk 42 us)
    one_long = dict(B=1, H_q=32, H_kv=8, num_pages=256, page_size=128)
    assert B.pa_choose_schedule(good_shape(L=1, max_pages_per_seq=8, **one_long)) == \
        B.PA_SCHED_PREFILL
    assert B.pa_choose_schedule(good_shape(L=1, max_pages_per_seq=128, **one_long)) == \
        B.PA_SCHED_PREFILL
    # up to 32 pairs over at most 4096 keys: the tiles (B = 4, 4096 keys: 27 us
    # against the page walk's 31 us), beyond that the page walk (B = 4, 16384
    # keys: 69 against 60 us; B = 8, 4096 keys: 44 against 41 us)
    four = dict(B=4, H_q=32, H_kv=8, num_pages=1024, page_size=128)
    assert B.pa_choose_schedule(good_shape(L=1, max_pages_per_seq=32, **four)) == \
        B.PA_SCHED_PREFILL
    assert B.pa_choose_schedule(good_shape(L=1, max_pages_per_seq=128, **four)) == \
        B.PA_SCHED_DECODE
    eight_long = dict(B=8, H_q=32, H_kv=8, num_pages=256, page_size=128)
    assert B.pa_choose_schedule(good_shape(L=1, max_pages_per_seq=32, **eight_long)) == \
        B.PA_SCHED_DECODE
    # fp32 and shapes the tiles do not take (page size not a multiple of 8)
    assert B.pa_choose_schedule(good_shape(L=2048, dtype=B.PA_F32)) == B.PA_SCHED_DECODE
    assert B.pa_choose_schedule(good_shape(L=64, page_size=12, num_pages=40)) == B.PA_SCHED_DECODE
    assert B.pa_choose_schedule(good_shape(D=64)) == -1
    assert B.pa_launch_count(good_shape(L=1), B.PA_SCHED_DECODE) == 2


def test_status_strings():
    for st in range(7):
        assert B.status_str(st) not in ("", "unknown status")
