"""Pins for the fp64 oracle: checks against facts fixed by the pages and by
mathematics, not against the oracle itself.

Each ``pin_*`` function takes an ``oracle.OracleLib`` and raises
``AssertionError`` (or ``oracle.OracleError``) when the oracle disagrees.
They are used twice: by test_oracle_pins.py on the real oracle, and by
test_oracle_mutants.py on builds with one planted mistake, to show that every
planted mistake trips at least one pin.

The facts:
  * brute force: a separately written dense attention on the *logical* K/V
    (never paged), with the visibility mask materialised as an L x S matrix
    ("Week 2 Day 5: Fused Decode Attention", Task 1 normalises masks to
    [B*H_q, L, S]) and scipy's softmax;
  * a library routine: torch's scaled_dot_product_attention in float64 where
    its causal convention coincides with the pages' (non-causal, or L == S);
  * invariants: physical page permutation ("Week 3 Day 5: Paged
    FlashAttention", Task 1: physical ids need not be consecutive), block-table
    entries past the last page are never read, GQA equals explicit head
    repetition ("Week 2 Day 5", Task 1: broadcasting pairs heads without
    repeating K/V);
  * tile-size independence of a streaming online-softmax fold ("Day 22: the
    fused paged-attention kernel", What I learned 1 and 3);
  * closed forms: a dominant key gives exactly its value row; identical keys
    give the mean of exactly the visible value rows, which fixes the causal
    boundary s <= l + context_len - L ("Week 3 Day 5", Task 2) to the key.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.special

import oracle as oracle_mod
from paged_kv_cache_03_gb300.synth import bf16_bits, bf16_to_f32

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TOL = 1e-12


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# Paged case built from logical tensors (test side, independent of synth's
# pool generator): logical K/V are drawn first, then scattered into a pool.
# --------------------------------------------------------------------------
class Case:
    pass


def make_case(seed, B, H_q, H_kv, L, D, ps, ctx, *, num_pages=None, dtype="bf16",
              perm=None, k_mult=1.0, q=None, K=None, V=None, causal=True, scale=None):
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, dtype=np.int32)
    Smax = int(ctx.max())

    def draw(shape, mult=1.0):
        v = rng.standard_normal(shape).astype(np.float32) * np.float32(mult)
        if dtype == "bf16":
            bits = bf16_bits(v)
            return bits, bf16_to_f32(bits).astype(np.float64)
        return v, v.astype(np.float64)

    c = Case()
    if q is None:
        c.q_store, c.q = draw((B, H_q, L, D))
    else:
        c.q_store, c.q = q
    if K is None:
        c.K_store, c.K = draw((B, H_kv, Smax, D), k_mult)
    else:
        c.K_store, c.K = K
    if V is None:
        c.V_store, c.V = draw((B, H_kv, Smax, D))
    else:
        c.V_store, c.V = V
    npg = [(int(s) + ps - 1) // ps for s in ctx]
    need = sum(npg)
    P = num_pages if num_pages is not None else need + 3
    if perm is None:
        perm = rng.permutation(P)
    perm = np.asarray(perm)
    maxnpg = max(npg) + 1
    bt = np.full((B, maxnpg), -1, dtype=np.int32)
    sdt = np.uint16 if dtype == "bf16" else np.float32
    # every pool slot starts as noise, so a stray read would show
    kp, _ = draw((P, H_kv, ps, D))
    vp, _ = draw((P, H_kv, ps, D))
    kp = np.ascontiguousarray(kp.astype(sdt))
    vp = np.ascontiguousarray(vp.astype(sdt))
    off = 0
    for b in range(B):
        for lp in range(npg[b]):
            page = int(perm[off])
            off += 1
            bt[b, lp] = page
            for slot in range(ps):
                s = lp * ps + slot
                if s < ctx[b]:
                    kp[page, :, slot, :] = c.K_store[b, :, s, :]
                    vp[page, :, slot, :] = c.V_store[b, :, s, :]
    c.kp, c.vp, c.bt, c.ctx = kp, vp, bt, ctx
    c.q_store = np.ascontiguousarray(c.q_store)
    c.B, c.H_q, c.H_kv, c.L, c.D, c.ps = B, H_q, H_kv, L, D, ps
    c.causal = causal
    c.scale = float(np.float32(1.0 / math.sqrt(D) if scale is None else scale))
    return c


def run_oracle(lib, c, bt=None):
    return lib.paged_attention(c.q_store, c.kp, c.vp, c.bt if bt is None else bt, c.ctx,
                               c.scale, c.causal)


def visible_mask(L, S, causal):
    s = np.arange(S)[None, :]
    l = np.arange(L)[:, None]
    return (s <= l + S - L) if causal else np.ones((L, S), dtype=bool)


def dense_bruteforce(c):
    """Dense attention on the logical tensors with a materialised mask."""
    G = c.H_q // c.H_kv
    out = np.zeros((c.B, c.H_q, c.L, c.D))
    for b in range(c.B):
        S = int(c.ctx[b])
        Kr = np.repeat(c.K[b, :, :S], G, axis=0)  # [H_q, S, D]
        Vr = np.repeat(c.V[b, :, :S], G, axis=0)
        scores = np.einsum("hld,hsd->hls", c.q[b], Kr) * c.scale
        scores = np.where(visible_mask(c.L, S, c.causal)[None], scores, -np.inf)
        P = scipy.special.softmax(scores, axis=-1)
        out[b] = np.einsum("hls,hsd->hld", P, Vr)
    return out


def assert_close(a, b, tol=TOL, what=""):
    err = np.max(np.abs(np.asarray(a) - np.asarray(b)))
    assert np.all(np.isfinite(a)), f"{what}: non-finite output"
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


# --------------------------------------------------------------------------
# Pins
# --------------------------------------------------------------------------
BRUTE_CASES = [
    # (seed, B, H_q, H_kv, L, D, ps, ctx, causal, dtype)
    (11, 2, 4, 2, 5, 128, 16, [13, 40], True, "bf16"),   # the tiny workload's shape
    (12, 2, 4, 2, 3, 8, 3, [7, 20], True, "bf16"),
    (13, 1, 2, 1, 4, 16, 1, [9], True, "bf16"),
    (14, 2, 4, 4, 6, 8, 5, [6, 33], True, "f32"),
    (15, 2, 6, 2, 2, 8, 4, [17, 2], False, "bf16"),
    (16, 1, 4, 2, 1, 32, 16, [40], True, "f32"),
    (17, 2, 4, 2, 5, 16, 4, [3, 17], False, "bf16"),  # no causal rule, L > context length
]


def pin_bruteforce(lib):
    for seed, B, Hq, Hkv, L, D, ps, ctx, causal, dt in BRUTE_CASES:
        c = make_case(seed, B, Hq, Hkv, L, D, ps, ctx, dtype=dt, causal=causal)
        assert_close(run_oracle(lib, c), dense_bruteforce(c), what=f"bruteforce seed {seed}")


def pin_torch_sdpa(lib):
    import torch
    import torch.nn.functional as F
    for seed, B, Hq, Hkv, L, D, ps, S, causal in [
        (21, 1, 4, 2, 24, 16, 5, 24, True),    # L == S: torch's causal convention agrees
        (22, 2, 2, 1, 3, 32, 4, 19, False),
        (23, 1, 8, 2, 9, 128, 16, 9, True),
    ]:
        c = make_case(seed, B, Hq, Hkv, L, D, ps, [S] * B, causal=causal)
        G = Hq // Hkv
        q = torch.from_numpy(c.q)
        K = torch.from_numpy(np.repeat(c.K[:, :, :S], G, axis=1))
        V = torch.from_numpy(np.repeat(c.V[:, :, :S], G, axis=1))
        ref = F.scaled_dot_product_attention(q, K, V, is_causal=causal, scale=c.scale)
        assert_close(run_oracle(lib, c), ref.numpy(), what=f"sdpa seed {seed}")


def pin_page_permutation(lib):
    base = dict(B=2, H_q=4, H_kv=2, L=3, D=16, ps=4, ctx=[15, 9])
    outs = []
    need = 4 + 3
    for perm in (np.arange(need), np.random.default_rng(5).permutation(need),
                 np.random.default_rng(6).permutation(need)[::-1].copy()):
        c = make_case(31, num_pages=need, perm=perm, **base)
        outs.append(run_oracle(lib, c))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0]), "output depends on physical page placement"
    assert_close(outs[0], dense_bruteforce(c), what="permutation case")


def pin_shared_pages(lib):
    """Several table rows may name one physical page (a common prefix held
    once; the translation of "Week 3 Day 5", Task 1 only reads the pool):
    the result is bitwise that of private copies, and the dense brute force."""
    c = make_case(37, 3, 4, 2, 3, 16, 4, [13, 10, 9])
    # give sequences 1 and 2 sequence 0's first two pages (8 positions)
    K_store, K = c.K_store.copy(), c.K.copy()
    V_store, V = c.V_store.copy(), c.V.copy()
    for b in (1, 2):
        K_store[b, :, :8], K[b, :, :8] = c.K_store[0, :, :8], c.K[0, :, :8]
        V_store[b, :, :8], V[b, :, :8] = c.V_store[0, :, :8], c.V[0, :, :8]
    c = make_case(37, 3, 4, 2, 3, 16, 4, [13, 10, 9], q=(c.q_store, c.q), K=(K_store, K),
                  V=(V_store, V))
    private = run_oracle(lib, c)
    bt = c.bt.copy()
    bt[1:, :2] = c.bt[0, :2]
    assert np.array_equal(run_oracle(lib, c, bt), private), "page sharing changed the result"
    assert_close(private, dense_bruteforce(c), what="shared-prefix case")


def pin_unused_table_entries(lib):
    c = make_case(41, 2, 2, 1, 2, 16, 8, [17, 8])
    ref = run_oracle(lib, c)
    for fill in (-1, 0, 2 ** 31 - 1, c.kp.shape[0]):
        bt = c.bt.copy()
        for b in range(c.B):
            npg = (int(c.ctx[b]) + c.ps - 1) // c.ps
            bt[b, npg:] = fill
        assert np.array_equal(run_oracle(lib, c, bt), ref), f"unused entry {fill} was read"


def _online_fold(q, K, V, last, scale, tile):
    """Streaming fold of the keys 0..last in tiles, keeping a running max,
    running denominator and running weighted-V sum; the old state is
    rescaled by exp(m_old - m_new) whenever the max moves up."""
    D = q.shape[0]
    m, den, acc = -np.inf, 0.0, np.zeros(D)
    S = K.shape[0]
    for t0 in range(0, S, tile):
        idx = np.arange(t0, min(t0 + tile, S))
        valid = idx <= last
        x = np.where(valid, scale * (K[idx] @ q), -np.inf)
        m_new = max(m, float(x.max()))
        if m_new == -np.inf:
            continue
        corr = math.exp(m - m_new) if m > -np.inf else 0.0
        p = np.where(valid, np.exp(x - m_new), 0.0)
        den = den * corr + p.sum()
        acc = acc * corr + p @ V[idx]
        m = m_new
    return acc / den


def pin_tile_size_invariance(lib):
    g = golden("tile_size_invariance.json")
    S = g["history"]
    d = golden("fused_kernel_diagram.json")
    for seed, S_, L, tiles in ((51, S, 3, g["block_sizes"]), (52, d["history"], 1, [d["tile"]])):
        c = make_case(seed, 1, 2, 1, L, 16, 4, [S_])
        ref = run_oracle(lib, c)
        for tile in tiles:
            for h in range(c.H_q):
                for l in range(L):
                    last = l + S_ - L
                    got = _online_fold(c.q[0, h, l], c.K[0, 0, :S_], c.V[0, 0, :S_],
                                       last, c.scale, tile)
                    assert_close(ref[0, h, l], got, what=f"tile {tile}")


def pin_single_page(lib):
    # context inside one page: the result is plain attention over that page's
    # first S slots, read straight from the pool array
    rng = np.random.default_rng(61)
    ps, S, D = 16, 11, 32
    c = make_case(61, 1, 2, 2, 1, D, ps, [S], num_pages=5, causal=False)
    page = int(c.bt[0, 0])
    got = run_oracle(lib, c)
    for h in range(2):
        Kp = bf16_to_f32(c.kp[page, h, :S]).astype(np.float64)
        Vp = bf16_to_f32(c.vp[page, h, :S]).astype(np.float64)
        w = scipy.special.softmax(c.scale * (Kp @ c.q[0, h, 0]))
        assert_close(got[0, h, 0], w @ Vp, what="single page")
    del rng


def pin_one_hot(lib):
    # one key's score exceeds all others by > 745, so every other weight is
    # below exp(-745) ~ 5e-324: the output is exactly that key's value row
    D, S, j = 128, 37, 23
    rng = np.random.default_rng(71)
    qf = rng.standard_normal((1, 1, 1, D)).astype(np.float32)
    qb = bf16_bits(qf)
    qv = bf16_to_f32(qb).astype(np.float64)
    Kf = rng.standard_normal((1, 1, S, D)).astype(np.float32) * np.float32(0.01)
    Kf[0, 0, j] = bf16_to_f32(qb[0, 0, 0]) * np.float32(120.0)
    Kb = bf16_bits(Kf)
    c = make_case(71, 1, 1, 1, 1, D, 8, [S], q=(qb, qv),
                  K=(Kb, bf16_to_f32(Kb).astype(np.float64)), causal=False)
    x = c.scale * (c.K[0, 0, :S] @ c.q[0, 0, 0])
    assert x[j] - np.delete(x, j).max() > 745.0
    got = run_oracle(lib, c)
    assert np.array_equal(got[0, 0, 0], c.V[0, 0, j]), "dominant key must return its value row"


def pin_uniform_visible_mean(lib):
    # identical keys -> equal scores -> each row averages exactly its visible
    # value rows; with causal, row l sees keys 0 .. l + S - L
    for seed, L, S, ps, causal in ((81, 5, 13, 4, True), (82, 7, 40, 16, True),
                                   (83, 3, 9, 2, False), (84, 9, 9, 3, True)):
        D = 16
        rng = np.random.default_rng(seed)
        row = bf16_bits(rng.standard_normal(D).astype(np.float32))
        Kb = np.broadcast_to(row, (1, 1, S, D)).copy()
        c = make_case(seed, 1, 1, 1, L, D, ps, [S],
                      K=(Kb, bf16_to_f32(Kb).astype(np.float64)), causal=causal)
        got = run_oracle(lib, c)
        for l in range(L):
            n = (l + S - L + 1) if causal else S
            assert_close(got[0, 0, l], c.V[0, 0, :n].mean(axis=0), what=f"uniform row {l}")


def pin_gqa_equals_repeat(lib):
    B, Hq, Hkv, L, D, ps, ctx = 2, 6, 2, 3, 16, 4, [14, 7]
    c = make_case(91, B, Hq, Hkv, L, D, ps, ctx)
    G = Hq // Hkv
    rep = make_case(91, B, Hq, Hq, L, D, ps, ctx, q=(c.q_store, c.q),
                    K=(np.repeat(c.K_store, G, axis=1), np.repeat(c.K, G, axis=1)),
                    V=(np.repeat(c.V_store, G, axis=1), np.repeat(c.V, G, axis=1)))
    assert np.array_equal(run_oracle(lib, c), run_oracle(lib, rep)), "GQA map differs from repetition"


def pin_gather(lib):
    c = make_case(101, 2, 2, 2, 1, 16, 3, [10, 4])
    k, v = lib.gather(c.kp, c.vp, c.bt, c.ctx, 12)
    for b in range(c.B):
        S = int(c.ctx[b])
        assert np.array_equal(k[b, :, :S], c.K[b, :, :S])
        assert np.array_equal(v[b, :, :S], c.V[b, :, :S])
        assert not k[b, :, S:].any() and not v[b, :, S:].any()


def pin_errors(lib):
    c = make_case(111, 1, 2, 1, 2, 16, 4, [6])
    bt = c.bt.copy()
    bt[0, 0] = c.kp.shape[0]
    for args, code in (
        (dict(bt=bt), oracle_mod.oracle.ORACLE_ERR_BAD_BLOCK_TABLE),
        (dict(ctx=np.array([1], np.int32)), oracle_mod.oracle.ORACLE_ERR_INVALID_ARG),
        (dict(ctx=np.array([0], np.int32)), oracle_mod.oracle.ORACLE_ERR_INVALID_ARG),
        (dict(ctx=np.array([10 ** 6], np.int32)), oracle_mod.oracle.ORACLE_ERR_INVALID_ARG),
    ):
        try:
            lib.paged_attention(c.q_store, c.kp, c.vp, args.get("bt", c.bt),
                                args.get("ctx", c.ctx), c.scale, True)
        except oracle_mod.OracleError as e:
            assert e.code == code, (args, e.code)
        else:
            raise AssertionError(f"expected error {code} for {list(args)}")


def pin_rows_api(lib):
    c = make_case(121, 2, 4, 2, 3, 16, 4, [9, 12])
    full = run_oracle(lib, c)
    rows = [(0, 3, 2), (1, 0, 0), (1, 2, 1)]
    got = lib.paged_attention_rows(c.q_store, c.kp, c.vp, c.bt, c.ctx, c.scale, True, rows)
    for i, (b, h, l) in enumerate(rows):
        assert np.array_equal(got[i], full[b, h, l])


# ---- K/V append ---------------------------------------------------------------
# The append writes the new tokens' rows at the last L positions of each
# context through the block table.  Facts that fix it:
#   * with pages handed out in order, the pool is a plain reshape of a dense
#     [B, H_kv, capacity, D] cache (numpy transpose/reshape), so the append is
#     a slice assignment dense[b, :, S-L:S, :] = new[b];
#   * physical page permutation is invisible: appending into a permuted pool
#     and un-permuting gives the in-order result, bitwise;
#   * nothing outside the targeted (page, slot) rows changes.
def _append_case(seed, B, H_kv, L, D, ps, ctx, npg_cap, dtype="bf16", perm=True):
    from paged_kv_cache_03_gb300.synth import new_kv
    rng = np.random.default_rng(seed)
    P = B * npg_cap
    order = rng.permutation(P).astype(np.int32) if perm else np.arange(P, dtype=np.int32)
    bt = order.reshape(B, npg_cap).copy()
    if dtype == "bf16":
        kp = bf16_bits(rng.standard_normal((P, H_kv, ps, D), dtype=np.float32))
        vp = bf16_bits(rng.standard_normal((P, H_kv, ps, D), dtype=np.float32))
    else:
        kp = rng.standard_normal((P, H_kv, ps, D), dtype=np.float32)
        vp = rng.standard_normal((P, H_kv, ps, D), dtype=np.float32)
    kn, vn = new_kv(B, H_kv, L, D, seed + 7, dtype)
    return kn, vn, kp, vp, bt, np.asarray(ctx, dtype=np.int32)


def _dense_view(pool, bt, B, H_kv, ps, D):
    """[B, H_kv, npg*ps, D] view of a pool whose sequence b owns pages
    bt[b, 0], bt[b, 1], ... in order."""
    npg = bt.shape[1]
    out = np.empty((B, H_kv, npg * ps, D), dtype=pool.dtype)
    for b in range(B):
        pages = pool[bt[b]]                      # [npg, H_kv, ps, D]
        out[b] = pages.transpose(1, 0, 2, 3).reshape(H_kv, npg * ps, D)
    return out


def pin_append_dense_slice(lib):
    for seed, B, H_kv, L, ps, ctx, cap in ((201, 2, 2, 3, 4, [7, 12], 3),
                                           (202, 3, 1, 1, 1, [1, 5, 2], 5),
                                           (203, 2, 2, 5, 3, [5, 9], 4)):
        for dtype in ("bf16", "f32"):
            kn, vn, kp, vp, bt, c = _append_case(seed, B, H_kv, L, 16, ps, ctx, cap, dtype,
                                                 perm=False)
            k2, v2, st = lib.append_kv(kn, vn, kp, vp, bt, c)
            assert st == oracle_mod.ORACLE_OK
            for pool, new, after in ((kp, kn, k2), (vp, vn, v2)):
                want = _dense_view(pool, bt, B, H_kv, ps, 16)
                for b in range(B):
                    want[b, :, c[b] - L:c[b], :] = new[b]
                got = _dense_view(after, bt, B, H_kv, ps, 16)
                assert np.array_equal(got, want), (seed, dtype)


def pin_append_page_permutation(lib):
    B, H_kv, L, ps, ctx, cap = 3, 2, 4, 4, [6, 11, 4], 3
    kn, vn, kp, vp, bt, c = _append_case(211, B, H_kv, L, 16, ps, ctx, cap, perm=False)
    k_ref, v_ref, st = lib.append_kv(kn, vn, kp, vp, bt, c)
    assert st == oracle_mod.ORACLE_OK
    perm = np.random.default_rng(212).permutation(kp.shape[0])
    kpp = np.empty_like(kp)
    vpp = np.empty_like(vp)
    kpp[perm] = kp
    vpp[perm] = vp
    k2, v2, st = lib.append_kv(kn, vn, kpp, vpp, perm[bt].astype(np.int32), c)
    assert st == oracle_mod.ORACLE_OK
    assert np.array_equal(k2[perm], k_ref) and np.array_equal(v2[perm], v_ref)


def pin_append_touches_only_new_rows(lib):
    B, H_kv, L, ps, ctx, cap = 2, 2, 3, 4, [9, 3], 4
    kn, vn, kp, vp, bt, c = _append_case(221, B, H_kv, L, 16, ps, ctx, cap)
    bt[:, 3] = -7  # entries past each context's pages: never read
    k2, v2, st = lib.append_kv(kn, vn, kp, vp, bt, c)
    assert st == oracle_mod.ORACLE_OK
    changed = np.any(k2 != kp, axis=-1) | np.any(v2 != vp, axis=-1)  # [P, H_kv, ps]
    want = np.zeros_like(changed)
    for b in range(B):
        for t in range(L):
            s = int(c[b]) - L + t
            want[bt[b, s // ps], :, s % ps] = True
    assert np.array_equal(changed, want)
    # and the gather of the appended pools returns the new rows there
    kd, vd = lib.gather(k2, v2, bt, c, int(c.max()))
    for b in range(B):
        assert np.array_equal(kd[b, :, c[b] - L:c[b]], bf16_to_f32(kn[b]).astype(np.float64))
        assert np.array_equal(vd[b, :, c[b] - L:c[b]], bf16_to_f32(vn[b]).astype(np.float64))


def pin_append_errors(lib):
    B, H_kv, L, ps, ctx, cap = 2, 1, 3, 4, [2, 7], 2  # sequence 0 is shorter than L
    kn, vn, kp, vp, bt, c = _append_case(231, B, H_kv, L, 16, ps, ctx, cap)
    k2, v2, st = lib.append_kv(kn, vn, kp, vp, bt, c)
    assert st == oracle_mod.ORACLE_ERR_INVALID_ARG
    assert np.array_equal(k2[bt[0]], kp[bt[0]])  # nothing of sequence 0 written
    kd, _ = lib.gather(k2, v2, bt[1:], c[1:], 7)
    assert np.array_equal(kd[0, :, 4:7], bf16_to_f32(kn[1]).astype(np.float64))
    bt2 = bt.copy()
    bt2[1, 1] = kp.shape[0] + 3  # position 4..6 of sequence 1 sit on a bad page
    c2 = np.array([3, 7], dtype=np.int32)
    k3, _, st = lib.append_kv(kn, vn, kp, vp, bt2, c2)
    assert st == oracle_mod.ORACLE_ERR_BAD_BLOCK_TABLE
    kd, _ = lib.gather(k3, k3, bt2[:1], c2[:1], 3)
    assert np.array_equal(kd[0, :, 0:3], bf16_to_f32(kn[0]).astype(np.float64))


# ---- explicit additive masks -------------------------------------------------
# "Week 2 Day 5: Fused Decode Attention", Task 1 normalises explicit masks to
# [B * H_q, L, S] and keeps the causal flag next to them; the mask is added to
# the scaled scores before the softmax.  Facts that fix the masked oracle:
#   * brute force: the dense attention above with the mask added to its logits;
#   * a zero mask is no mask (bitwise), a per-row constant mask cancels in the
#     softmax (closed form);
#   * a mask that lifts one visible key far above the rest gives exactly that
#     key's value row; a row with every key at -inf outputs 0.
def _mask_for(c, S_mask, seed, dense=True):
    rng = np.random.default_rng(seed)
    m = rng.standard_normal((c.B * c.H_q, c.L, S_mask)).astype(np.float32)
    if dense:  # knock out a random third of the positions as well
        m[rng.random(m.shape) < 0.33] = -np.inf
    return m


def _dense_masked(c, mask):
    G = c.H_q // c.H_kv
    out = np.zeros((c.B, c.H_q, c.L, c.D))
    for b in range(c.B):
        S = int(c.ctx[b])
        Kr = np.repeat(c.K[b, :, :S], G, axis=0)
        Vr = np.repeat(c.V[b, :, :S], G, axis=0)
        scores = np.einsum("hld,hsd->hls", c.q[b], Kr) * c.scale
        scores = scores + mask[b * c.H_q:(b + 1) * c.H_q, :, :S].astype(np.float64)
        scores = np.where(visible_mask(c.L, S, c.causal)[None], scores, -np.inf)
        for h in range(c.H_q):
            for l in range(c.L):
                row = scores[h, l]
                if np.all(row == -np.inf):
                    continue  # nothing visible: 0
                P = scipy.special.softmax(row)
                out[b, h, l] = P @ Vr[h]
    return out


def pin_mask_bruteforce(lib):
    for seed, B, Hq, Hkv, L, D, ps, ctx, causal, dt in BRUTE_CASES[:5]:
        c = make_case(seed + 500, B, Hq, Hkv, L, D, ps, ctx, dtype=dt, causal=causal)
        S_mask = int(max(ctx)) + 3
        mask = _mask_for(c, S_mask, seed + 600)
        got = lib.paged_attention(c.q_store, c.kp, c.vp, c.bt, c.ctx, c.scale, c.causal,
                                  mask=mask)
        assert_close(got, _dense_masked(c, mask), what=f"masked brute force {seed}")


def pin_mask_zero_and_row_constant(lib):
    c = make_case(701, 2, 4, 2, 3, 16, 4, [11, 6])
    ref = run_oracle(lib, c)
    zero = np.zeros((c.B * c.H_q, c.L, 12), dtype=np.float32)
    got = lib.paged_attention(c.q_store, c.kp, c.vp, c.bt, c.ctx, c.scale, c.causal, mask=zero)
    assert np.array_equal(got, ref), "a zero mask must be no mask"
    rowc = np.random.default_rng(702).standard_normal((c.B * c.H_q, c.L, 1)).astype(np.float32)
    const = np.broadcast_to(rowc * 7, (c.B * c.H_q, c.L, 12)).copy()
    got = lib.paged_attention(c.q_store, c.kp, c.vp, c.bt, c.ctx, c.scale, c.causal, mask=const)
    assert_close(got, ref, what="per-row constant mask")


def pin_mask_dominant_and_empty_rows(lib):
    c = make_case(711, 1, 2, 1, 4, 16, 4, [10])
    mask = np.zeros((2, 4, 10), dtype=np.float32)
    j = 3  # visible to every row (rows see keys 0..6+l)
    mask[:, :, j] = 800.0
    got = lib.paged_attention(c.q_store, c.kp, c.vp, c.bt, c.ctx, c.scale, True, mask=mask)
    for h in range(2):
        for l in range(4):
            assert_close(got[0, h, l], c.V[0, 0, j], what="dominant masked key")
    mask = np.zeros((2, 4, 10), dtype=np.float32)
    mask[1, 2, :] = -np.inf  # every key of row (h=1, l=2)
    got = lib.paged_attention(c.q_store, c.kp, c.vp, c.bt, c.ctx, c.scale, True, mask=mask)
    assert np.array_equal(got[0, 1, 2], np.zeros(16)), "a fully masked row outputs 0"
    ref = run_oracle(lib, c)
    keep = np.ones((2, 4), dtype=bool)
    keep[1, 2] = False
    assert np.array_equal(got[0][keep], ref[0][keep])


# --------------------------------------------------------------------------
# Ragged batches: per-sequence query counts, tokens packed [T, H_q, D]
# --------------------------------------------------------------------------
VARLEN_CASES = [
    # (seed, H_q, H_kv, D, ps, L_b per sequence, context lengths, causal, dtype)
    (81, 4, 2, 8, 3, [1, 7, 1, 3, 2], [9, 20, 1, 40, 2], True, "bf16"),
    (82, 2, 2, 16, 16, [5, 1, 1], [5, 33, 17], True, "f32"),
    (83, 6, 2, 8, 4, [2, 4, 1], [11, 6, 30], False, "bf16"),
    (84, 4, 1, 128, 16, [1, 6], [13, 40], True, "bf16"),
]


def _varlen_case(seed, H_q, H_kv, D, ps, lens, ctx, causal, dtype):
    """A ragged batch on the logical tensors of make_case: sequence b's
    queries are the first L_b query rows drawn for it, packed by token."""
    Lmax = max(lens)
    c = make_case(seed, len(lens), H_q, H_kv, Lmax, D, ps, ctx, dtype=dtype, causal=causal)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q_store = np.zeros((T, H_q, D), dtype=c.q_store.dtype)
    q = np.zeros((T, H_q, D))
    for b, Lb in enumerate(lens):
        q_store[cu[b]:cu[b + 1]] = c.q_store[b, :, :Lb, :].transpose(1, 0, 2)
        q[cu[b]:cu[b + 1]] = c.q[b, :, :Lb, :].transpose(1, 0, 2)
    c.vq_store, c.vq, c.cu, c.lens = np.ascontiguousarray(q_store), q, cu, list(lens)
    return c


def _varlen_dense(c):
    """Dense attention per sequence on the logical K/V: sequence b's L_b
    queries are the last L_b of its S_b positions."""
    G = c.H_q // c.H_kv
    out = np.zeros(c.vq.shape)
    for b, Lb in enumerate(c.lens):
        if Lb == 0:
            continue
        S = int(c.ctx[b])
        Kr = np.repeat(c.K[b, :, :S], G, axis=0)
        Vr = np.repeat(c.V[b, :, :S], G, axis=0)
        qb = c.vq[c.cu[b]:c.cu[b + 1]].transpose(1, 0, 2)  # [H_q, L_b, D]
        scores = np.einsum("hld,hsd->hls", qb, Kr) * c.scale
        scores = np.where(visible_mask(Lb, S, c.causal)[None], scores, -np.inf)
        P = scipy.special.softmax(scores, axis=-1)
        out[c.cu[b]:c.cu[b + 1]] = np.einsum("hls,hsd->hld", P, Vr).transpose(1, 0, 2)
    return out


def _run_varlen(lib, c, **kw):
    return lib.paged_attention_varlen(c.vq_store, c.kp, c.vp, c.bt, c.ctx, c.cu, c.scale,
                                      c.causal, **kw)


def pin_varlen_bruteforce(lib):
    for case in VARLEN_CASES:
        c = _varlen_case(*case)
        assert_close(_run_varlen(lib, c), _varlen_dense(c), what=f"varlen seed {case[0]}")


def pin_varlen_equals_single_sequences(lib):
    """Each sequence of a ragged batch gives exactly the rows of a batch of
    that sequence alone with L = L_b (the uniform path, pinned above)."""
    for case in VARLEN_CASES:
        c = _varlen_case(*case)
        got = _run_varlen(lib, c)
        for b, Lb in enumerate(c.lens):
            q1 = np.ascontiguousarray(c.vq_store[c.cu[b]:c.cu[b + 1]].transpose(1, 0, 2)[None])
            one = lib.paged_attention(q1, c.kp, c.vp, np.ascontiguousarray(c.bt[b:b + 1]),
                                      np.ascontiguousarray(c.ctx[b:b + 1]), c.scale, c.causal)
            assert np.array_equal(got[c.cu[b]:c.cu[b + 1]], one[0].transpose(1, 0, 2)), \
                f"varlen seed {case[0]}: sequence {b} differs from its single-sequence batch"


def pin_varlen_empty_sequences_and_errors(lib):
    """Sequences with no new queries are not read (their context length and
    table row may be anything); a broken offset array or a query count above
    the context (causal) is rejected."""
    c = _varlen_case(85, 4, 2, 8, 3, [2, 3], [7, 12], True, "bf16")
    ref = _run_varlen(lib, c)
    # insert an empty sequence with junk metadata between the two
    bt = np.concatenate([c.bt[:1], np.full((1, c.bt.shape[1]), 10 ** 6, np.int32), c.bt[1:]])
    ctx = np.array([c.ctx[0], -5, c.ctx[1]], dtype=np.int32)
    cu = np.array([0, 2, 2, 5], dtype=np.int32)
    got = lib.paged_attention_varlen(c.vq_store, c.kp, c.vp, bt, ctx, cu, c.scale, True)
    assert np.array_equal(got, ref), "an empty sequence changed the batch"
    for cu_bad, what in (([1, 2, 5], "cu_q[0] != 0"), ([0, 4, 5], "L_b > max_L"),
                         ([0, 3, 2], "decreasing offsets")):
        try:
            lib.paged_attention_varlen(c.vq_store, c.kp, c.vp, c.bt, c.ctx,
                                       np.array(cu_bad, np.int32), c.scale, True, max_L=3)
        except oracle_mod.OracleError as e:
            assert e.code == oracle_mod.ORACLE_ERR_INVALID_ARG, what
        else:
            raise AssertionError(f"accepted {what}")
    short = np.array([2, 2], dtype=np.int32)  # sequence 1: 3 queries, 2 keys
    try:
        lib.paged_attention_varlen(c.vq_store, c.kp, c.vp, c.bt, short, c.cu, c.scale, True)
    except oracle_mod.OracleError as e:
        assert e.code == oracle_mod.ORACLE_ERR_INVALID_ARG
    else:
        raise AssertionError("accepted L_b > context length under causal")


ALL_PINS = [pin_bruteforce, pin_torch_sdpa, pin_page_permutation, pin_shared_pages,
            pin_unused_table_entries,
            pin_tile_size_invariance, pin_single_page, pin_one_hot, pin_uniform_visible_mean,
            pin_gqa_equals_repeat, pin_gather, pin_errors, pin_rows_api,
            pin_append_dense_slice, pin_append_page_permutation, pin_append_touches_only_new_rows,
            pin_append_errors, pin_mask_bruteforce, pin_mask_zero_and_row_constant,
            pin_mask_dominant_and_empty_rows, pin_varlen_bruteforce,
            pin_varlen_equals_single_sequences, pin_varlen_empty_sequences_and_errors]
