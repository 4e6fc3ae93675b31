// prefill.cu -- schedule (b): long causal prefills on tcgen05 tensor cores.
//
// What it computes is the same exact paged attention as the page walk
// ("Week 3 Day 5: Paged FlashAttention"): Task 1's page translation while
// staging K/V tiles, Task 2's tiled online softmax (Q.K^T -> scale and causal
// bounds -> merge the max -> rescale sum and accumulator -> exponentials and
// sum -> P.V), whole K/V tiles past the causal frontier skipped, and the
// normalised bf16 output written once.
//
// How it is laid out on GB300 (one CTA per pair of 128-row query tiles):
//   * The 128 rows of a tile are Lt = 128/G consecutive positions l of all G
//     query heads that share one kv head (GQA packing), so one K/V tile feeds
//     128 rows and the causal frontier moves by only Lt keys across the tile.
//     A CTA owns two consecutive tiles, A and B, which share every K/V tile.
//   * Warp 0 stages tiles with 2-D TMA loads (128-byte swizzle): both query
//     tiles once (one box per head), then 128-key K and V tiles into 2-slot
//     rings.  Every box lies inside one page: box height
//     = gcd(page_size, 128) rows, its row coordinate (physical_page * H_kv +
//     kv_head) * page_size + slot comes from the block table, so a tile that
//     crosses pages is just several boxes.
//   * Warp 1 allocates all 512 TMEM columns (S_A, S_B, O_A, O_B, 128 each)
//     and one thread issues tcgen05.mma in the order PV_A(j), S_A(j+1),
//     PV_B(j), S_B(j+1): while one softmax warpgroup works on its tile the
//     tensor core runs the other tile's products.  S = Q.K^T uses K-major
//     operands; O += P.V reads V MN-major from its natural [key][dim] layout.
//   * Warps 4-7 (tile A) and 8-11 (tile B) run the softmax, one TMEM lane
//     (query row) per thread: S row from TMEM, causal/length mask, row max of
//     the raw scores, running max moved only when it grows by more than 2^8
//     (then O is rescaled in TMEM), p = 2^(s*scale*log2 e - m) with one packed
//     FMA and one exp2 per score, P rounded to bf16 into swizzled shared
//     memory for the P.V MMA (one buffer, written by A and B in turn), running
//     sum in fp32; at the end O/l -> bf16 -> global.  Whole K/V tiles past a
//     tile's last causal frontier are skipped.
//   * Boxes are copied whole, so a sequence's last K/V tile can carry page
//     rows past its context (unused slots, any contents).  Their scores are
//     masked to -inf.  Their V rows would still meet a weight of exactly 0,
//     and 0 * NaN is NaN, so the producer lands that V tile on a barrier of
//     its own, zeroes those rows and only then releases the tile to the MMA.
//   * All waits are bounded; on a timeout the CTA records PA_FLAG_TIMEOUT,
//     lets its copies and MMAs finish, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace pa {
namespace {

constexpr int kD = kHeadDim;
constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per K/V tile
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S of tile t at 128 t, O of tile t at 256 + 128 t
__host__ __device__ constexpr uint32_t col_s(int t) { return 128u * static_cast<uint32_t>(t); }
__host__ __device__ constexpr uint32_t col_o(int t) { return 256u + 128u * static_cast<uint32_t>(t); }
constexpr float kLazyRescaleLog2 = 8.0f;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kHalf = BM * 128;   // 128 rows x 64 bf16 (one 128-byte swizzle column block)
constexpr int kTile = 2 * kHalf;  // 128 rows x 128 bf16
constexpr int kOffQ = 0;                    // tile t at kOffQ + t * kTile
constexpr int kOffK = kOffQ + 2 * kTile;    // slot s at kOffK + s * kTile
constexpr int kOffV = kOffK + 2 * kTile;    // slot s at kOffV + s * kTile
constexpr int kOffP = kOffV + 2 * kTile;    // one P buffer, used by A and B in turn
constexpr int kOffBar = kOffP + kTile;
enum Bar {
    kQFull = 0,
    kKFull = 1,   // + slot
    kKEmpty = 3,  // + slot
    kVFull = 5,   // + slot
    kVEmpty = 7,  // + slot
    kSFull = 9,   // + tile
    kPFull = 11,  // + tile
    kODone = 13,  // + tile
    kMmaDone = 15,
    kVTail = 16,  // the V tile that holds rows past the context
    kNumBars = 18  // (even: what follows stays 16-byte aligned)
};
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kOffRows = kOffAbort + 8;  // output row (b, h, l) = base + h * sh + l * sl
constexpr int kSmemUsed = kOffRows + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack to align the base

struct PrefillParams {
    const int32_t* bt;
    const int32_t* ctx;
    void* out;
    uint32_t* flag;
    int B, H_q, H_kv, L, G, Lt, nM, nPairs, num_pages, ps, max_npg, box_rows, causal;
    long long max_S;
    float scale_log2;
    const float* mask;  // optional additive mask [B * H_q, L, mask_S], or null
    long long mask_S;   // >= the table's capacity, a multiple of 4
    // ragged batch (null cu_q: the [B, H_q, L, D] layout): rows packed by
    // token [total_q, H_q, D]; sequence b owns tokens cu_q[b] .. cu_q[b+1]-1;
    // pair_prefix[b] = query-tile pairs of sequences before b, [B] = all
    const int32_t* cu_q;
    const int* pair_prefix;
    int total_q;
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Output rows of one CTA's sequence, in units of D elements: row (b, h, l)
// is base + h * sh + l * sl ([B, H_q, L, D], or [tokens, H_q, D] from token
// q0 on).  Kept in shared memory between the set-up and the epilogue.
struct alignas(16) OutRows {
    long long base;
    int sh, sl;
};

// All 32 lanes wait; the warp agrees on the outcome (a lane that timed out
// makes the whole warp give up, so warp-collective instructions stay uniform).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __all_sync(0xffffffffu, ok);
}

// Warp-uniform read of the CTA's abort flag.
__device__ __forceinline__ bool aborted(volatile int* f) {
    return __any_sync(0xffffffffu, *f != 0);
}

__device__ __forceinline__ void give_up(const PrefillParams& p, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(p.flag, PA_FLAG_TIMEOUT);
}

// The block-table row coordinates of the boxes of K/V tile j (lane i: box i
// and i + 32 ...); -1 for boxes past the context or with a bad page id.
__device__ __forceinline__ void tile_boxes(const PrefillParams& p, int b, int kvh, int S, int j,
                                           int lane, int (&row)[4], uint32_t& bytes) {
    const int nbox = BN / p.box_rows;
    bytes = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const int bi = lane + 32 * w;
        row[w] = -1;
        const int key = j * BN + bi * p.box_rows;
        if (bi < nbox && key < S) {
            const int lp = key / p.ps, slot = key - lp * p.ps;
            const int pp = __ldg(p.bt + static_cast<long long>(b) * p.max_npg + lp);
            if (pp >= 0 && pp < p.num_pages) {
                row[w] = (pp * p.H_kv + kvh) * p.ps + slot;
                bytes += 2u * static_cast<uint32_t>(p.box_rows) * 128u;  // two 64-dim halves
            } else {
                atomicOr(p.flag, PA_FLAG_BAD_PAGE);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
}

__device__ __forceinline__ void issue_boxes(const CUtensorMap* map, uint32_t dst, const int (&row)[4],
                                            int lane, int box_rows, uint32_t bar, uint64_t pol) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        if (row[w] < 0) continue;
        const uint32_t off = static_cast<uint32_t>(lane + 32 * w) * box_rows * 128u;
        tc::tma_load_2d(dst + off, map, 0, row[w], bar, pol);
        tc::tma_load_2d(dst + kHalf + off, map, 64, row[w], bar, pol);
    }
}

// p = 2^(s * c - m) for one 128-key row: rounded to bf16 pairs in pw (the
// P.V operand) and summed in fp32 into ts.  The row sum adds the rounded
// weights, the same ones P.V applies to V, so the output stays a weighted
// mean of value rows: o = sum bf16(p) v / sum bf16(p).  Summing the unrounded
// p instead would scale a row dominated by one key by that key's rounding
// error (up to 2^-9 relative), which on the causal prefill workload's peaky
// rows reached 1.4e-2 absolute after the output's own rounding.
__device__ __forceinline__ void exp_pack(const float (&x)[4][32], float2 c2, float2 nm2,
                                         uint32_t (&pw)[64], float2& ts) {
#pragma unroll
    for (int k = 0; k < 64; ++k) {
        const int cc = k >> 4, e = (k & 15) * 2;
        const float2 y = __ffma2_rn(make_float2(x[cc][e], x[cc][e + 1]), c2, nm2);
        const uint32_t w = pack_bf16x2(fast_exp2(y.x), fast_exp2(y.y));
        ts = __fadd2_rn(ts, bf16x2_to_float2(w));
        pw[k] = w;
    }
}

// kMask: an explicit additive mask is read; kVarlen: a ragged batch (queries
// packed by token, per-sequence query counts).  Separate instantiations, so
// the plain kernel carries none of their code or registers.
template <bool kMask, bool kVarlen>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tile_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const sbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + kOffBar;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(sbase + kOffAbort);
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + kOffTmemSlot);
    OutRows* const out_rows = reinterpret_cast<OutRows*>(sbase + kOffRows);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- which tiles ----------------------------------------------------------
    // (b, kv head, pair mp of 128-row query tiles); Lb query positions of
    // sequence b, the first at token q0 (ragged batch)
    int b, kvh, mp, Lb = p.L, q0 = 0, nM = p.nM;
    if constexpr (kVarlen) {
        // a page walk over the batch's other sequences may start beside us
        pdl_launch_dependents();
        const int i = static_cast<int>(blockIdx.x) / p.H_kv;
        kvh = static_cast<int>(blockIdx.x) % p.H_kv;
        if (i >= p.pair_prefix[p.B]) return;  // past the batch's pairs: before any set-up
        int lo = 0, hi = p.B - 1;  // the last sequence whose pairs start at or before i
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.pair_prefix[mid] <= i) lo = mid;
            else hi = mid - 1;
        }
        b = lo;
        q0 = p.cu_q[b];
        Lb = p.cu_q[b + 1] - q0;
        nM = (Lb + p.Lt - 1) / p.Lt;
        mp = (nM + 1) / 2 - 1 - (i - p.pair_prefix[b]);  // heavy pairs of a sequence first
    } else {
        const int per_m = p.H_kv * p.B;
        mp = p.nPairs - 1 - static_cast<int>(blockIdx.x) / per_m;  // heavy pairs first
        const int rest = static_cast<int>(blockIdx.x) % per_m;
        b = rest / p.H_kv;
        kvh = rest % p.H_kv;
    }
    const int S = p.ctx[b];
    const bool valid_seq =
        S >= 1 && static_cast<long long>(S) <= p.max_S && !(p.causal && S < Lb);
    int nk_t[2], lim_min_t[2], l0_t[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int m = 2 * mp + t;
        l0_t[t] = m * p.Lt;
        const bool exists = m < nM && valid_seq;
        const int l_last = min(l0_t[t] + p.Lt, Lb) - 1;
        const int lim_max = p.causal ? l_last + S - Lb : S - 1;  // last key any row sees
        lim_min_t[t] = p.causal ? l0_t[t] + S - Lb : S - 1;      // last key row l0 sees
        nk_t[t] = exists ? lim_max / BN + 1 : 0;
    }
    const int nk = max(nk_t[0], nk_t[1]);
    const int ntiles = (2 * mp + 1 < nM) ? 2 : 1;
    // The producer's block-table lookup of K/V tile 0 goes out before the
    // set-up below, so its latency overlaps the set-up instead of delaying
    // the first copies.
    int rows_cur[4] = {-1, -1, -1, -1};
    uint32_t bytes_cur = 0;
    if (warp == 0 && nk > 0) tile_boxes(p, b, kvh, S, 0, lane, rows_cur, bytes_cur);

    // ---- set-up: barriers, V zeroed, TMEM --------------------------------------
    if (tid == 0) {
        mbar_init(bar(kQFull), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(kKFull + s), 1);
            mbar_init(bar(kKEmpty + s), 1);
            mbar_init(bar(kSFull + s), 1);
            mbar_init(bar(kPFull + s), 4);
            mbar_init(bar(kODone + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(kVFull + s), 1);
            mbar_init(bar(kVEmpty + s), 1);
        }
        mbar_init(bar(kMmaDone), 1);
        mbar_init(bar(kVTail), 1);
        *abort_flag = 0;
        if constexpr (kVarlen) {
            out_rows->base = static_cast<long long>(q0) * p.H_q;
            out_rows->sh = 1;
            out_rows->sl = p.H_q;
        } else {
            out_rows->base = static_cast<long long>(b) * p.H_q * p.L;
            out_rows->sh = p.L;
            out_rows->sl = 1;
        }
        fence_mbar_init();
    }
    // V rows that are never loaded must hold finite values (their weight is
    // exactly 0, and 0 * NaN would not be).  Only a last key tile that ends
    // past the context has such rows, and only in a slot no earlier tile of
    // this CTA filled (tiles 0 and 1); a tile whose last box runs past the
    // context is zeroed after its copy lands (kVTail).  Rows of a later slot
    // past the context still hold the finite rows of the tile two before.
    if (nk <= 2 && S < nk * BN && S % p.box_rows == 0) {
        uint4* v = reinterpret_cast<uint4*>(sbase + kOffV);
        for (int i = tid; i < 2 * kTile / 16; i += kThreads) v[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    if (warp == 1) {
        tc::tmem_alloc(base + kOffTmemSlot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    if (!valid_seq && tid == 0) atomicOr(p.flag, PA_FLAG_BAD_CONTEXT);

    if (warp == 0 && nk > 0) {
        // ============================ TMA producer ============================
        const uint64_t pol_q = l2_policy_evict_first();
        const uint64_t pol_kv = l2_policy_evict_last();
        if (lane == 0) {
            tc::prefetch_tensormap(&tm_q);
            tc::prefetch_tensormap(&tm_k);
            tc::prefetch_tensormap(&tm_v);
            mbar_arrive_expect_tx(bar(kQFull),
                                  static_cast<uint32_t>(ntiles * p.G * p.Lt * 128 * 2));
            for (int t = 0; t < ntiles; ++t)
                for (int g = 0; g < p.G; ++g) {
                    const uint32_t dst = base + kOffQ + t * kTile + g * p.Lt * 128;
                    if constexpr (kVarlen) {  // map (D, H_q, tokens): Lt tokens of head kvh*G + g
                        for (int h = 0; h < 2; ++h)
                            tc::tma_load_3d(dst + h * kHalf, &tm_q, h * 64, kvh * p.G + g,
                                            q0 + l0_t[t], bar(kQFull), pol_q);
                    } else {
                        const int row = ((b * p.H_q) + kvh * p.G + g) * p.L + l0_t[t];
                        for (int h = 0; h < 2; ++h)
                            tc::tma_load_2d(dst + h * kHalf, &tm_q, h * 64, row, bar(kQFull),
                                            pol_q);
                    }
                }
        }
        __syncwarp();
        // the K/V tile whose last box runs past the context (its V rows past
        // the context are zeroed before the MMA may read the tile), or -1
        const int tail_tile = (S % p.box_rows != 0) ? (S - 1) / BN : -1;
        int rows_next[4] = {-1, -1, -1, -1};
        uint32_t bytes_next = 0;
        int issued = 0;
        for (int t = 0; t < nk; ++t) {
            const int s = t & 1;
            if (t >= 2 && !warp_wait(bar(kKEmpty + s), ((t >> 1) - 1) & 1)) {
                if (lane == 0) give_up(p, abort_flag);
                break;
            }
            if (aborted(abort_flag)) break;
            if (lane == 0) mbar_arrive_expect_tx(bar(kKFull + s), bytes_cur);
            __syncwarp();
            issue_boxes(&tm_k, base + kOffK + s * kTile, rows_cur, lane, p.box_rows,
                        bar(kKFull + s), pol_kv);
            if (t >= 2 && !warp_wait(bar(kVEmpty + s), ((t >> 1) - 1) & 1)) {
                if (lane == 0) give_up(p, abort_flag);
                issued = -(t + 1);  // K(t) issued, V(t) not
                break;
            }
            const bool vtail = t == tail_tile;
            const uint32_t vbar = vtail ? bar(kVTail) : bar(kVFull + s);
            if (lane == 0) mbar_arrive_expect_tx(vbar, bytes_cur);
            __syncwarp();
            issue_boxes(&tm_v, base + kOffV + s * kTile, rows_cur, lane, p.box_rows, vbar, pol_kv);
            issued = t + 1;
            // rows of the next tile, looked up before waiting for a free slot
            if (t + 1 < nk) tile_boxes(p, b, kvh, S, t + 1, lane, rows_next, bytes_next);
            if (vtail) {  // the last tile this CTA loads: nothing waits behind it
                if (!warp_wait(bar(kVTail), 0)) {
                    if (lane == 0) give_up(p, abort_flag);
                    break;
                }
                for (int r = S - t * BN + lane; r < BN; r += 32) {
                    uint4* const vrow =
                        reinterpret_cast<uint4*>(sbase + kOffV + s * kTile + r * 128);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        vrow[q] = make_uint4(0u, 0u, 0u, 0u);
                        vrow[kHalf / 16 + q] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();  // the MMA reads them through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kVFull + s));
            }
#pragma unroll
            for (int w = 0; w < 4; ++w) rows_cur[w] = rows_next[w];
            bytes_cur = bytes_next;
        }
        // let every copy into this CTA's shared memory land before leaving
        if (!mbar_wait(bar(kQFull), 0)) give_up(p, abort_flag);
        const int kdone = issued < 0 ? -issued : issued, vdone = issued < 0 ? -issued - 1 : issued;
        for (int t = max(0, kdone - 2); t < kdone; ++t)
            if (!mbar_wait(bar(kKFull + (t & 1)), (t >> 1) & 1)) give_up(p, abort_flag);
        for (int t = max(0, vdone - 2); t < vdone; ++t)
            if (!(t == tail_tile ? mbar_wait(bar(kVTail), 0)
                                 : mbar_wait(bar(kVFull + (t & 1)), (t >> 1) & 1)))
                give_up(p, abort_flag);
    } else if (warp == 1 && nk > 0) {
        // ============================ MMA issuer =============================
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_bf16(BM, BN, 0, 0);  // Q, K both K-major
            constexpr uint32_t idO = tc::idesc_bf16(BM, kD, 0, 1);  // P K-major, V MN-major
            auto qk = [&](int t, int j) {
                const uint32_t kaddr = base + kOffK + (j & 1) * kTile;
                const uint32_t qaddr = base + kOffQ + t * kTile;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * kHalf + (kk & 3) * 32;
                    tc::mma_bf16(tmem + col_s(t), tc::smem_desc_sw128(qaddr + koff, 16, 1024),
                                 tc::smem_desc_sw128(kaddr + koff, 16, 1024), idS, kk > 0);
                }
                tc::commit(bar(kSFull + t));
            };
            auto pv = [&](int t, int j) {
                const uint32_t paddr = base + kOffP;
                const uint32_t vaddr = base + kOffV + (j & 1) * kTile;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {
                    const uint32_t poff = (kk >> 2) * kHalf + (kk & 3) * 32;
                    tc::mma_bf16(tmem + col_o(t), tc::smem_desc_sw128(paddr + poff, 16, 1024),
                                 tc::smem_desc_sw128(vaddr + kk * 16 * 128, kHalf, 1024), idO,
                                 (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::commit(bar(kODone + t));
            };
            bool ok = mbar_wait(bar(kQFull), 0) && mbar_wait(bar(kKFull), 0);
            if (ok) {
                tc::fence_after_sync();
                if (nk_t[0] > 0) qk(0, 0);
                if (nk_t[1] > 0) qk(1, 0);
                tc::commit(bar(kKEmpty));
            }
            for (int j = 0; ok && j < nk; ++j) {
                ok = mbar_wait(bar(kVFull + (j & 1)), (j >> 1) & 1);
                if (!ok || *abort_flag) break;
                const bool more = j + 1 < nk;
                if (j < nk_t[0]) {
                    ok = mbar_wait(bar(kPFull), j & 1);
                    if (!ok || *abort_flag) break;
                    tc::fence_after_sync();
                    pv(0, j);
                }
                if (more) {
                    ok = mbar_wait(bar(kKFull + ((j + 1) & 1)), ((j + 1) >> 1) & 1);
                    if (!ok || *abort_flag) break;
                    tc::fence_after_sync();
                    if (j + 1 < nk_t[0]) qk(0, j + 1);
                }
                if (j < nk_t[1]) {
                    ok = mbar_wait(bar(kPFull + 1), j & 1);
                    if (!ok || *abort_flag) break;
                    tc::fence_after_sync();
                    pv(1, j);
                }
                tc::commit(bar(kVEmpty + (j & 1)));
                if (more) {
                    if (j + 1 < nk_t[1]) qk(1, j + 1);
                    tc::commit(bar(kKEmpty + ((j + 1) & 1)));
                }
            }
            if (!ok) give_up(p, abort_flag);
            // nothing of ours may still be running when TMEM is freed
            tc::commit(bar(kMmaDone));
            if (!mbar_wait(bar(kMmaDone), 0)) give_up(p, abort_flag);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ============================= softmax ===============================
        const int t = (warp - 4) >> 2;      // tile of this warpgroup
        const int q4 = warp & 3;            // TMEM lane quarter of this warp
        const int r = q4 * 32 + lane;       // query row of this thread
        const uint32_t trow = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
        const int g = r / p.Lt, l = l0_t[t] + (r - g * p.Lt);
        const bool row_valid = t < ntiles && g < p.G && l < Lb;
        const int h = kvh * p.G + g;
        const int lim = min(p.causal ? l + S - Lb : S - 1, S - 1);
        const int nkt = nk_t[t];
        const float c = p.scale_log2;
        // with an explicit mask the scores are taken to log2 units (and the
        // mask added) right after the load, so the rest scales by 1
        const float cs = kMask ? 1.f : c;
        const float* const mask_row =
            kMask && row_valid
                ? p.mask + ((static_cast<long long>(b) * p.H_q + h) * p.L + l) * p.mask_S
                : nullptr;
        // the lines holding this row's visible mask entries of key tile jj go
        // to L2 ahead of use: keys [jj * BN, min(jj * BN + BN, lim + 1)), all
        // inside the row (lim < S <= mask_S)
        auto prefetch_mask = [&](int jj) {
            if (!kMask || !mask_row || jj >= nkt) return;
            const int k0 = jj * BN;
            if (k0 > lim) return;
            const int k1 = min(k0 + BN, lim + 1) - 1;  // last visible key of the tile
#pragma unroll
            for (int e = 0; e < 4; ++e) prefetch_l2(mask_row + min(k0 + 32 * e, k1));
            prefetch_l2(mask_row + k1);
        };
        prefetch_mask(0);
        float mrow = neg_inf();
        float2 lsum2 = make_float2(0.f, 0.f);
        bool ok = true;
        for (int j = 0; j < nkt; ++j) {
            prefetch_mask(j + 1);
            ok = warp_wait(bar(kSFull + t), j & 1);
            if (!ok || aborted(abort_flag)) break;
            tc::fence_after_sync();
            float x[4][32];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tc::ld32(trow + col_s(t) + cc * 32, x[cc]);
            tc::wait_ld();
            if constexpr (kMask) {  // s * scale * log2 e + mask * log2 e
                // only the words holding a visible key (k0 + 4q <= lim < mask_S)
                const int k0 = j * BN;
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    float4 mv = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (mask_row && k0 + 4 * q <= lim)
                        mv = __ldg(reinterpret_cast<const float4*>(mask_row + k0) + q);
                    const int cc = q >> 3, e = (q & 7) * 4;
                    x[cc][e + 0] = fmaf(x[cc][e + 0], c, mv.x * 1.4426950408889634f);
                    x[cc][e + 1] = fmaf(x[cc][e + 1], c, mv.y * 1.4426950408889634f);
                    x[cc][e + 2] = fmaf(x[cc][e + 2], c, mv.z * 1.4426950408889634f);
                    x[cc][e + 3] = fmaf(x[cc][e + 3], c, mv.w * 1.4426950408889634f);
                }
            }
            // causal / length mask (frontier tiles only), row max of raw scores
            const bool masking = j * BN + BN - 1 > lim_min_t[t];  // uniform over the CTA
            if (masking) {
                const int cmax = lim - j * BN;  // columns <= cmax are visible
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (cc * 32 + e > cmax) x[cc][e] = neg_inf();
            }
            float mq[4];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                mq[cc] = x[cc][0];
#pragma unroll
                for (int e = 1; e < 31; e += 2) mq[cc] = fmax3(mq[cc], x[cc][e], x[cc][e + 1]);
                mq[cc] = fmaxf(mq[cc], x[cc][31]);
            }
            float mt = fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
            mt *= cs;
            const bool grow = mt > mrow + kLazyRescaleLog2;
            const bool any_grow = __any_sync(0xffffffffu, grow);
            const float mn = grow ? mt : mrow;
            const float alpha = grow ? fast_exp2(mrow - mn) : 1.f;  // 2^-inf = 0 at start
            mrow = mn;
            // P = 2^(s*c - m) packed to bf16 pairs in registers, before any wait
            const float mu = (mrow == neg_inf()) ? 0.f : mrow;
            const float2 c2 = make_float2(cs, cs), nm2 = make_float2(-mu, -mu);
            float2 ts = make_float2(0.f, 0.f);
            uint32_t pw[64];
            exp_pack(x, c2, nm2, pw, ts);
            lsum2.x = lsum2.x * alpha + ts.x;
            lsum2.y = lsum2.y * alpha + ts.y;
            // O is rescaled once this tile's previous P.V is done
            if (any_grow && j > 0) {
                ok = warp_wait(bar(kODone + t), (j - 1) & 1);
                if (!ok || aborted(abort_flag)) break;
                tc::fence_after_sync();
#pragma unroll 1
                for (int cc = 0; cc < 4; ++cc) {
                    float o[32];
                    tc::ld32(trow + col_o(t) + cc * 32, o);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tc::st32(trow + col_o(t) + cc * 32, o);
                }
                tc::wait_st();
            }
            // the shared P buffer is free once the P.V that read it last is done:
            // A(j) follows B(j-1), B(j) follows A(j) (or its own tile's previous
            // P.V when the other tile has none there)
            {
                int wt = -1, wj = -1;
                if (t == 0) {
                    if (j - 1 >= 0 && j - 1 < nk_t[1]) wt = 1, wj = j - 1;
                    else if (j > 0) wt = 0, wj = j - 1;
                } else {
                    if (j < nk_t[0]) wt = 0, wj = j;
                    else if (j > 0) wt = 1, wj = j - 1;
                }
                if (wt >= 0) {
                    ok = warp_wait(bar(kODone + wt), wj & 1);
                    if (!ok || aborted(abort_flag)) break;
                }
            }
            tc::fence_after_sync();
            uint8_t* const prow = sbase + kOffP + r * 128;
#pragma unroll
            for (int q = 0; q < 16; ++q) {  // 8 keys per 16-byte chunk
                const uint4 w = make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
                const int half = q >> 3, cq = q & 7;
                *reinterpret_cast<uint4*>(prow + half * kHalf + ((cq ^ (r & 7)) << 4)) = w;
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kPFull + t));
        }
        const float lsum = lsum2.x + lsum2.y;
        if (!ok) {
            if (lane == 0) give_up(p, abort_flag);
        } else if (nkt > 0 && warp_wait(bar(kODone + t), (nkt - 1) & 1)) {
            tc::fence_after_sync();
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            uint16_t* const orow = static_cast<uint16_t*>(p.out) +
                                   (out_rows->base + static_cast<long long>(h) * out_rows->sh +
                                    static_cast<long long>(l) * out_rows->sl) * kD;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                float o[32];
                tc::ld32(trow + col_o(t) + cc * 32, o);
                tc::wait_ld();
                if (row_valid) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 w = make_uint4(
                            pack_bf16x2(o[q * 8 + 0] * inv, o[q * 8 + 1] * inv),
                            pack_bf16x2(o[q * 8 + 2] * inv, o[q * 8 + 3] * inv),
                            pack_bf16x2(o[q * 8 + 4] * inv, o[q * 8 + 5] * inv),
                            pack_bf16x2(o[q * 8 + 6] * inv, o[q * 8 + 7] * inv));
                        *reinterpret_cast<uint4*>(orow + cc * 32 + q * 8) = w;
                    }
                }
            }
        } else if (nkt > 0) {
            if (lane == 0) give_up(p, abort_flag);
        }
        if (!valid_seq && row_valid) {
            uint4* orow = reinterpret_cast<uint4*>(
                static_cast<uint16_t*>(p.out) +
                (out_rows->base + static_cast<long long>(h) * out_rows->sh +
                 static_cast<long long>(l) * out_rows->sl) * kD);
            for (int q = 0; q < kD / 8; ++q) orow[q] = make_uint4(0u, 0u, 0u, 0u);
        }
    }

    // ---- tear-down: free TMEM once every role is done -----------------------
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// Ragged batch: pair_prefix[b] = query-tile pairs of the sequences before b
// that the tile schedule takes (L_b > min_L), [B] = all.  A sequence whose
// offsets are broken (cu_q[b] < 0, L_b < 0 or > max_L, cu_q[b+1] > total_q)
// gets none and sets PA_FLAG_BAD_CONTEXT.  One CTA, a block scan per 1024
// sequences.
__global__ void __launch_bounds__(1024) pair_plan_kernel(const int32_t* cu_q, int B, int total_q,
                                                         int Lt, int min_L, int max_L,
                                                         uint32_t* flag, int* pair_prefix) {
    __shared__ int warp_sums[32];
    __shared__ int carry_s;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < B; base += 1024) {
        const int b = base + tid;
        int v = 0;
        if (b < B) {
            const int q0 = cu_q[b], q1 = cu_q[b + 1], Lb = q1 - q0;
            const bool broken = q0 < 0 || Lb < 0 || Lb > max_L || q1 > total_q;
            if (broken) atomicOr(flag, PA_FLAG_BAD_CONTEXT);
            else if (Lb > min_L) v = ((Lb + Lt - 1) / Lt + 1) / 2;
        }
        int x = v;  // inclusive scan: warps, then warp totals
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[w] = x;
        __syncthreads();
        if (w == 0) {
            int t = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            warp_sums[lane] = t;
        }
        __syncthreads();
        const int incl = x + (w > 0 ? warp_sums[w - 1] : 0);
        const int carry = carry_s;
        if (b < B) pair_prefix[b] = carry + incl - v;
        __syncthreads();
        if (tid == 1023) carry_s = carry + incl;
        __syncthreads();
    }
    if (tid == 0) pair_prefix[B] = carry_s;
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

}  // namespace

// 2-D bf16 map over a row-major [rows, 128] matrix, boxes of 64 x box_rows,
// 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* ptr, long long rows, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
    cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// Token-major query map (D, H_q, tokens): one box = box_rows tokens of one
// head, laid out in shared memory exactly like a box of the 2-D map.
bool make_map_tokens(CUtensorMap* map, const void* ptr, int H_q, long long tokens, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H_q),
                          static_cast<cuuint64_t>(tokens)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2,
                             static_cast<cuuint64_t>(H_q) * kD * 2};
    cuuint32_t box[3] = {64u, 1u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gcd_int(int a, int b) {
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

}  // namespace

bool prefill_supported(const pa_shape& sh) {
    if (sh.dtype != PA_BF16 || sh.D != kD) return false;
    const int G = sh.H_q / sh.H_kv;
    // G must divide the 128-row tile, and every TMA box must start on a
    // 1024-byte (8-row) boundary of the 128-byte swizzle: query boxes are
    // 128/G rows, key/value boxes gcd(page_size, 128) rows.
    if (G < 1 || G > 16 || (BM % G) != 0) return false;
    if (sh.page_size % 8 != 0) return false;
    const long long q_rows = static_cast<long long>(sh.B) * sh.H_q * sh.L;
    if (q_rows >= (1ll << 31)) return false;
    const long long nM = (sh.L + BM / G - 1) / (BM / G);
    if (nM * sh.H_kv * sh.B >= (1ll << 31)) return false;
    return true;
}

pa_status prefill_launch(const Call& c) {
    const pa_shape& sh = c.sh;
    if (!prefill_supported(sh)) return PA_ERR_UNSUPPORTED;
    if (c.dev.smem_optin < kSmemBytes) return PA_ERR_UNSUPPORTED;
    const int G = sh.H_q / sh.H_kv;
    const int Lt = BM / G;
    const int box_rows = gcd_int(sh.page_size, BN);
    CUtensorMap tq, tk, tv;
    const long long pool_rows = static_cast<long long>(sh.num_pages) * sh.H_kv * sh.page_size;
    const bool q_ok = c.cu_q ? make_map_tokens(&tq, c.q, sh.H_q, c.total_q, Lt)
                             : make_map(&tq, c.q, static_cast<long long>(sh.B) * sh.H_q * sh.L, Lt);
    if (!q_ok || !make_map(&tk, c.kp, pool_rows, box_rows) ||
        !make_map(&tv, c.vp, pool_rows, box_rows))
        return PA_ERR_CUDA;

    static int attr_done[64] = {0};
    if (c.dev.device >= 0 && c.dev.device < 64 && !attr_done[c.dev.device]) {
        if (cudaFuncSetAttribute(prefill_tile_kernel<false, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(prefill_tile_kernel<true, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(prefill_tile_kernel<false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess)
            return PA_ERR_CUDA;
        attr_done[c.dev.device] = 1;
    }
    PrefillParams p;
    p.bt = c.bt;
    p.ctx = c.ctx;
    p.out = c.out;
    p.flag = static_cast<uint32_t*>(c.ws);
    p.B = sh.B;
    p.H_q = sh.H_q;
    p.H_kv = sh.H_kv;
    p.L = sh.L;
    p.G = G;
    p.Lt = Lt;
    p.nM = (sh.L + Lt - 1) / Lt;
    p.nPairs = (p.nM + 1) / 2;
    p.num_pages = sh.num_pages;
    p.ps = sh.page_size;
    p.max_npg = sh.max_pages_per_seq;
    p.box_rows = box_rows;
    p.causal = c.causal ? 1 : 0;
    p.max_S = static_cast<long long>(sh.max_pages_per_seq) * sh.page_size;
    p.scale_log2 = c.scale * 1.4426950408889634f;
    p.mask = c.mask;
    p.mask_S = c.mask_S;
    p.cu_q = c.cu_q;
    p.total_q = c.total_q;
    p.pair_prefix = nullptr;
    long long pairs = static_cast<long long>(p.nPairs) * sh.B;
    if (c.cu_q) {
        // the pairs of all sequences are at most ceil(L_b / (2 Lt)) each, so at
        // most (total_q + B (2 Lt - 1)) / (2 Lt) together; CTAs past the
        // planned pairs return at once
        pairs = std::min(pairs, (static_cast<long long>(c.total_q) +
                                 static_cast<long long>(sh.B) * (2 * Lt - 1)) / (2 * Lt));
        int* plan = reinterpret_cast<int*>(static_cast<uint8_t*>(c.ws) + c.plan_off);
        p.pair_prefix = plan;
        pair_plan_kernel<<<1, 1024, 0, c.stream>>>(c.cu_q, sh.B, c.total_q, Lt, c.tiles_min_L,
                                                   sh.L, p.flag, plan);
        if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
        if (pairs == 0) return PA_OK;
    }
    const unsigned grid = static_cast<unsigned>(pairs * sh.H_kv);
    if (c.ev_before && cudaEventRecord(c.ev_before, c.stream) != cudaSuccess) return PA_ERR_CUDA;
    if (c.cu_q)  // (a ragged batch takes no explicit mask)
        prefill_tile_kernel<false, true><<<grid, kThreads, kSmemBytes, c.stream>>>(tq, tk, tv, p);
    else if (c.mask)
        prefill_tile_kernel<true, false><<<grid, kThreads, kSmemBytes, c.stream>>>(tq, tk, tv, p);
    else
        prefill_tile_kernel<false, false><<<grid, kThreads, kSmemBytes, c.stream>>>(tq, tk, tv, p);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (c.ev_after && cudaEventRecord(c.ev_after, c.stream) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

}  // namespace pa
