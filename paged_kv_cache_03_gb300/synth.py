"""Seeded synthetic inputs for paged attention.

This module only draws random numbers and lays them out: it holds none of the
attention arithmetic, so the CUDA path and the CPU oracle can both be fed from
it without sharing any of the method.

Recipe (the same for every workload):
  * ``numpy.random.default_rng(seed)``; draws happen in a fixed order:
    context lengths, page permutation, query, key pool, value pool.
  * Values are fp32 N(0, 1), multiplied by ``k_scale`` for keys, then rounded
    to bf16 with round-to-nearest-even (bf16 workloads) or kept fp32 (fp32
    control).  The same bits feed both sides.
  * The physical pool holds ``num_pages`` pages; a random permutation of the
    page ids is cut into consecutive chunks, one per sequence, so physical ids
    are scattered and non-consecutive.  Every pool page, used or not, holds
    N(0, 1) data.  Block-table entries past a sequence's last page are -1.

Layouts: query [B, H_q, L, D]; key/value pages [num_pages, H_kv, page_size, D];
block_table int32 [B, max_pages_per_seq]; context_lens int32 [B].
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# Named workloads.  Head shapes follow Qwen3-4B (32 query heads, 8 KV heads,
# head dim 128), the model the pages measure with.
WORKLOADS = {
    # B=2, pool of 16 pages of 16 slots, contexts 13 and 40, 5 causal queries.
    "tiny": dict(B=2, H_q=4, H_kv=2, L=5, D=128, page_size=16, num_pages=16,
                 context_lens=[13, 40], seed=1),
    # 64 single-token decodes, contexts U{128..4096}, 128-slot pages.
    "decode": dict(B=64, H_q=32, H_kv=8, L=1, D=128, page_size=128,
                   ctx_range=(128, 4096), seed=2),
    # 4 causal prefills of 2048 tokens, keys x2 to widen the score range.
    "prefill": dict(B=4, H_q=32, H_kv=8, L=2048, D=128, page_size=128,
                    context_lens=[2048] * 4, num_pages=64, k_scale=2.0, seed=3),
    # chunked-prefill continuation: 65 new queries on contexts U{1000..8000}.
    "tails": dict(B=8, H_q=32, H_kv=8, L=65, D=128, page_size=128,
                  ctx_range=(1000, 8000), seed=4),
    # 16 decodes over 32768-token contexts in 16-slot pages (whole pool permuted).
    "long_decode": dict(B=16, H_q=32, H_kv=8, L=1, D=128, page_size=16,
                        context_lens=[32768] * 16, num_pages=32768, seed=5),
}


@dataclasses.dataclass
class PagedInputs:
    query: np.ndarray          # [B, H_q, L, D]  uint16 (bf16 bits) or float32
    key_pages: np.ndarray      # [P, H_kv, ps, D]
    value_pages: np.ndarray    # [P, H_kv, ps, D]
    block_table: np.ndarray    # [B, max_pages_per_seq] int32, -1 past the last page
    context_lens: np.ndarray   # [B] int32
    page_size: int
    scale: float               # an fp32-representable value
    causal: bool
    dtype: str                 # "bf16" or "f32"
    name: str = ""

    @property
    def B(self):
        return self.query.shape[0]

    @property
    def H_q(self):
        return self.query.shape[1]

    @property
    def L(self):
        return self.query.shape[2]

    @property
    def D(self):
        return self.query.shape[3]

    @property
    def H_kv(self):
        return self.key_pages.shape[1]

    @property
    def num_pages(self):
        return self.key_pages.shape[0]

    @property
    def max_pages_per_seq(self):
        return self.block_table.shape[1]


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(rng, shape, dtype: str, mult: float = 1.0, chunk: int = 1 << 24):
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = rng.standard_normal(e - s, dtype=np.float32)
        if mult != 1.0:
            v *= np.float32(mult)
        out[s:e] = bf16_bits(v) if dtype == "bf16" else v
    return out.reshape(shape)


def generate(B, H_q, H_kv, L, D, page_size, context_lens=None, ctx_range=None,
             num_pages=None, max_pages_per_seq=None, seed=0, dtype="bf16",
             k_scale=1.0, causal=True, scale=None, name="") -> PagedInputs:
    rng = np.random.default_rng(seed)
    if context_lens is None:
        lo, hi = ctx_range
        context_lens = rng.integers(lo, hi + 1, size=B)
    ctx = np.asarray(context_lens, dtype=np.int64)
    assert ctx.shape == (B,)
    npg = [(int(s) + page_size - 1) // page_size for s in ctx]
    if max_pages_per_seq is None:
        top = ctx_range[1] if ctx_range is not None else int(ctx.max())
        max_pages_per_seq = max(1, (top + page_size - 1) // page_size, max(npg))
    need = sum(npg)
    if num_pages is None:
        num_pages = max(need, 1)
    assert num_pages >= need, "pool too small for the contexts"
    perm = rng.permutation(num_pages).astype(np.int32)
    block_table = np.full((B, max_pages_per_seq), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        block_table[b, :npg[b]] = perm[off:off + npg[b]]
        off += npg[b]
    query = _normal(rng, (B, H_q, L, D), dtype)
    key_pages = _normal(rng, (num_pages, H_kv, page_size, D), dtype, k_scale)
    value_pages = _normal(rng, (num_pages, H_kv, page_size, D), dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    scale = float(np.float32(scale))
    return PagedInputs(query, key_pages, value_pages, block_table,
                       ctx.astype(np.int32), page_size, scale, bool(causal), dtype, name)


def workload(name: str, dtype: str = "bf16", **overrides) -> PagedInputs:
    """One of the named workloads, optionally with fields overridden."""
    kw = dict(WORKLOADS[name])
    kw.update(overrides)
    return generate(dtype=dtype, name=name, **kw)


def new_kv(B: int, H_kv: int, L: int, D: int, seed: int, dtype: str = "bf16"):
    """Seeded N(0,1) rows of the new tokens' keys and values, [B, H_kv, L, D]
    each (bf16 bit patterns or fp32), for the K/V append."""
    rng = np.random.default_rng(seed)
    return _normal(rng, (B, H_kv, L, D), dtype), _normal(rng, (B, H_kv, L, D), dtype)


def additive_mask(rows: int, L: int, S_mask: int, seed: int, removed: float = 1.0 / 3.0):
    """Seeded fp32 additive mask [rows, L, S_mask] (rows = B * H_q): N(0,1)
    biases, a `removed` fraction of the positions at -inf."""
    rng = np.random.default_rng(seed)
    m = rng.standard_normal((rows, L, S_mask), dtype=np.float32)
    m[rng.random(m.shape) < removed] = -np.inf
    return m


def additive_mask_device(rows: int, L: int, S_mask: int, seed: int, device,
                         removed: float = 1.0 / 3.0):
    """additive_mask's recipe (N(0,1) biases, a `removed` fraction at -inf)
    drawn on a CUDA device with torch's seeded generator, for the gigabyte
    masks of the full-size workloads; the values differ from additive_mask's."""
    import torch
    g = torch.Generator(device=device).manual_seed(seed)
    m = torch.randn((rows, L, S_mask), generator=g, device=device, dtype=torch.float32)
    drop = torch.rand((rows, L, S_mask), generator=g, device=device) < removed
    return m.masked_fill_(drop, float("-inf"))


@dataclasses.dataclass
class RaggedInputs:
    query: np.ndarray          # [T, H_q, D] packed by token (bf16 bits or float32)
    key_pages: np.ndarray      # [P, H_kv, ps, D]
    value_pages: np.ndarray
    block_table: np.ndarray    # [B, max_pages_per_seq] int32
    context_lens: np.ndarray   # [B] int32
    cu_q: np.ndarray           # [B + 1] int32 query offsets
    page_size: int
    scale: float
    causal: bool
    dtype: str
    name: str = ""

    @property
    def B(self):
        return int(self.block_table.shape[0])

    @property
    def H_q(self):
        return int(self.query.shape[1])

    @property
    def H_kv(self):
        return int(self.key_pages.shape[1])

    @property
    def D(self):
        return int(self.query.shape[2])

    @property
    def num_pages(self):
        return int(self.key_pages.shape[0])

    @property
    def q_lens(self):
        return np.diff(self.cu_q)

    @property
    def max_L(self):
        return max(1, int(self.q_lens.max()))


def generate_ragged(H_q, H_kv, D, page_size, q_lens, context_lens, seed=0, dtype="bf16",
                    num_pages=None, max_pages_per_seq=None, k_scale=1.0, causal=True,
                    scale=None, name="") -> RaggedInputs:
    """A ragged batch: sequence b has q_lens[b] new queries (its last
    positions) and context_lens[b] keys; pools and block table as in
    generate(), queries packed by token."""
    q_lens = np.asarray(q_lens, dtype=np.int64)
    B = len(q_lens)
    base = generate(B, H_q, H_kv, 1, D, page_size, context_lens=context_lens,
                    num_pages=num_pages, max_pages_per_seq=max_pages_per_seq, seed=seed,
                    dtype=dtype, k_scale=k_scale, causal=causal, scale=scale, name=name)
    rng = np.random.default_rng(seed + 7919)
    T = int(q_lens.sum())
    query = _normal(rng, (T, H_q, D), dtype)
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return RaggedInputs(query, base.key_pages, base.value_pages, base.block_table,
                        base.context_lens, cu_q, page_size, base.scale, bool(causal), dtype, name)


# A continuous-batching step (Qwen3-4B heads): 56 single-token decodes over
# contexts U{128..4096} and 8 prefill chunks of 128 tokens (the serving
# trace's prefill step) over contexts U{128..2048}, in one batch.
def mixed_workload(seed=6, dtype="bf16") -> RaggedInputs:
    rng = np.random.default_rng(seed)
    n_dec, n_pre, chunk = 56, 8, 128
    ctx_dec = rng.integers(128, 4096 + 1, size=n_dec)
    ctx_pre = rng.integers(chunk, 2048 + 1, size=n_pre)
    order = rng.permutation(n_dec + n_pre)  # decodes and chunks interleaved
    q_lens = np.concatenate([np.ones(n_dec, np.int64), np.full(n_pre, chunk)])[order]
    ctx = np.concatenate([ctx_dec, ctx_pre])[order]
    return generate_ragged(32, 8, 128, 128, q_lens, ctx, seed=seed, dtype=dtype,
                           max_pages_per_seq=4096 // 128, name="mixed")
