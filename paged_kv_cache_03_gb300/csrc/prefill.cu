// prefill.cu -- schedule (b): long causal prefills on tcgen05 tensor cores.
//
// What it computes is the same exact paged attention as the page walk
// ("Week 3 Day 5: Paged FlashAttention"): Task 1's page translation while
// staging K/V tiles, Task 2's tiled online softmax (Q.K^T -> scale and causal
// bounds -> merge the max -> rescale sum and accumulator -> exponentials and
// sum -> P.V), whole K/V tiles past the causal frontier skipped, and the
// normalised bf16 output written once.
//
// How it is laid out on GB300 (a persistent CTA per SM, each claiming work
// items = pairs of 128-row query tiles from a counter, heaviest first; one
// item's query load and first K/V tiles overlap the previous item's last
// products and epilogue):
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
//     operands; O += P.V takes P from TMEM and reads V MN-major from its
//     natural [key][dim] layout.  S_t(j+1) overwrites the columns that hold
//     P_t(j); it is issued after P.V_t(j), and one thread's MMAs execute in
//     issue order.
//   * Warps 4-7 (tile A) and 8-11 (tile B) run the softmax, one TMEM lane
//     (query row) per thread: S row from TMEM, causal/length mask, row max of
//     the raw scores, running max moved only when it grows by more than 2^8
//     (then O is rescaled in TMEM), p = 2^(s*scale*log2 e - m) with one packed
//     FMA and one exp2 per score, P rounded to bf16 and stored back into
//     Tensor Memory over the first 64 columns of the tile's S, where the P.V
//     MMA reads it as its A operand (so P crosses no shared memory and the
//     two tiles never wait for each other's products), running sum in fp32;
//     at the end O/l -> bf16 -> global.  Whole K/V tiles past a tile's last
//     causal frontier are skipped.
//   * Epilogue: each warp's output rows go out 16 at a time through a 4 KB
//     shared-memory slice and tiled TMA stores (one head's consecutive
//     positions); other rows are stored directly.
//   * Few, long query tiles: each pair's keys are cut into chunks (one wave
//     of items), each writing fp32 partials that tile_combine_kernel merges;
//     a last query tile of at most 8 rows rides on warps 2 and 3 of the last
//     full pair's CTA (warp-level MMA).
//   * With an explicit mask, warp 2 stages the mask tiles into shared memory
//     with TMA, a slot ring of three (the instance keeps one K and one V slot).
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
// Output staging for the tiled stores of the epilogue: 16 rows x 256 bytes
// per warp (two 64-dim halves, 128-byte swizzled), tile t at + t * 16 KB.
constexpr int kOffStage = kOffV + 2 * kTile;
constexpr int kStageRows = 16;
constexpr int kOffBar = kOffStage + 2 * 4 * kStageRows * 256;
// With an explicit mask the kernel keeps one K slot and one V slot and
// stages the mask in three 32 KB slots instead: the second K slot, the
// second V slot and the output staging (whose rows that instance stores
// directly).  A slot holds 64 keys x 128 rows of fp32 as two 32-key column
// blocks of 16 KB, each G boxes of Lt rows x 128 bytes, 128-byte swizzled.
constexpr int kMaskSlots = 3;
__host__ __device__ constexpr int mask_off(int s) {
    return s == 0 ? kOffK + kTile : s == 1 ? kOffV + kTile : kOffStage;
}
constexpr int kMaskHalf = 64;  // keys per mask slot
// K/V ring positions: with a mask one slot, else two
template <bool kOne>
struct KRing {
    static constexpr int kSlots = kOne ? 1 : 2;
    __device__ static int slot(int g) { return kOne ? 0 : (g & 1); }
    __device__ static uint32_t full_parity(int g) { return kOne ? (g & 1) : ((g >> 1) & 1); }
    // the wait for the slot to be free before tile g is loaded into it
    __device__ static uint32_t empty_parity(int g) { return kOne ? ((g - 1) & 1) : (((g >> 1) - 1) & 1); }
};
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
    kVTail = 16,      // the V tile that holds rows past the context
    kQEmpty = 17,     // the item's Q.K^T products are done with the query tiles
    kOFree = 18,      // + tile: the item's epilogue has read O
    kItemFull = 20,   // + slot: a work item is published
    kItemEmpty = 22,  // + slot: every role has read it
    // A slot's fills alternate between the query tiles, so each tile waits on
    // full barriers of its own: it then waits for their phases in order,
    // never for one two phases ahead of the barrier.
    kMaskFull = 24,   // + 3 * tile + slot: the tile's mask half-tile is staged
    kMaskEmpty = 30,  // + slot: the half-tile in the slot has been read
    kNumBars = 34     // (even: what follows stays 16-byte aligned)
};
constexpr int kOffItems = kOffBar + kNumBars * 8;  // 2 slots x 32 bytes
constexpr int kOffTmemSlot = kOffItems + 64;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemUsed = kOffAbort + 8;
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
    int n_items;        // work items (query-tile pairs x kv heads x key splits); a ragged batch's come from its plan
    int* item_counter;  // [next item to claim, CTAs done]: zero between calls
    // key split ([B, H_q, L, D] layout only): each pair's key tiles are cut into
    // nsplit equal chunks, one work item each; with nsplit > 1 every item writes
    // fp32 partials (m, l per row; o[D] per row of a chunk with keys) that
    // tile_combine_kernel merges
    int nsplit;
    float2* part_ml;  // [B * H_q * L][nsplit]
    float* part_o;    // [B * H_q * L][nsplit][D]
    // The last query tile of a sequence, when it holds at most 8 rows (nrem =
    // G x the positions from rem_l0 on), is not a tensor-core item of its own:
    // warps 2 and 3 of the last full pair's CTA take those rows over each
    // staged K/V tile with warp-level MMA, 64 keys each, and write fp32
    // partials per (key chunk, warp) for tile_combine_kernel.  0: none.
    int nrem, rem_l0;
    float2* rem_ml;  // [B * H_kv][nrem][nsplit * 2]
    float* rem_o;    // [B * H_kv][nrem][nsplit * 2][D]
    const void* q;   // the query, [B, H_q, L, D] (read by warps 2 and 3)
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

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

// One work item: query-tile pair mp of sequence b under kv head kvh.
struct Item {
    int b, kvh, mp, S, Lb, q0, nM, live, c;  // c: key chunk of a split pair
};

// Work item i, heaviest pairs first (a CTA claims items from a counter, so
// the heavy ones start early and the light ones fill the gaps at the end).
// Full pairs go in decreasing mp (later queries see more keys under the
// causal rule); an odd last tile, alone in its pair, does half a pair's
// products and goes after the heavier half of the full pairs.
template <bool kVarlen, bool kSplit>
__device__ __forceinline__ Item decode_item(const PrefillParams& p, int i, int n_items) {
    Item it{0, 0, 0, 0, 0, 0, 0, 0, 0};
    if (i >= n_items) return it;
    it.live = 1;
    if constexpr (kVarlen) {
        const int ip = i / p.H_kv;
        it.kvh = i % p.H_kv;
        int lo = 0, hi = p.B - 1;  // the last sequence whose pairs start at or before ip
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.pair_prefix + mid) <= ip) lo = mid;
            else hi = mid - 1;
        }
        it.b = lo;
        it.q0 = __ldg(p.cu_q + lo);
        it.Lb = __ldg(p.cu_q + lo + 1) - it.q0;
        it.nM = (it.Lb + p.Lt - 1) / p.Lt;
        it.mp = (it.nM + 1) / 2 - 1 - (ip - __ldg(p.pair_prefix + lo));  // heavy pairs first
    } else {
        const int ns = kSplit ? p.nsplit : 1;
        const int pi = i / ns;  // the chunks of a pair are consecutive items
        it.c = i - pi * ns;
        const int per_m = p.H_kv * p.B;
        const int q = pi / per_m;  // rank of the pair in the claim order
        const int nfull = p.nM / 2, ins = nfull - nfull / 2;
        if ((p.nM & 1) && q == ins) {
            it.mp = nfull;  // the odd last tile
        } else {
            it.mp = nfull - 1 - ((p.nM & 1) && q > ins ? q - 1 : q);
        }
        const int rest = pi % per_m;
        it.b = rest / p.H_kv;
        it.kvh = rest % p.H_kv;
        it.Lb = p.L;
        it.nM = p.nM;
    }
    it.S = __ldg(p.ctx + it.b);
    return it;
}

// What an item asks of each role: key tiles per query tile (0 for a tile past
// the sequence's queries or a sequence whose context breaks the contract),
// the first query position of each tile and the last key its first row sees.
struct ItemWork {
    int nk_t[2], lim_min_t[2], l0_t[2], nk, ntiles;
    // this item's key tiles: j0 .. j0 + nkc - 1, of which tile t takes the
    // first nkc_t[t] (all of them without a key split)
    int j0, nkc_t[2], nkc;
    bool valid_seq;
};

template <bool kSplit>
__device__ __forceinline__ ItemWork item_work(const PrefillParams& p, const Item& it) {
    ItemWork w;
    w.valid_seq = it.S >= 1 && static_cast<long long>(it.S) <= p.max_S &&
                  !(p.causal && it.S < it.Lb);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int m = 2 * it.mp + t;
        w.l0_t[t] = m * p.Lt;
        const bool exists = m < it.nM && w.valid_seq;
        const int l_last = min(w.l0_t[t] + p.Lt, it.Lb) - 1;
        const int lim_max = p.causal ? l_last + it.S - it.Lb : it.S - 1;  // last key any row sees
        w.lim_min_t[t] = p.causal ? w.l0_t[t] + it.S - it.Lb : it.S - 1;  // last key row l0 sees
        w.nk_t[t] = exists ? lim_max / BN + 1 : 0;
    }
    w.nk = max(w.nk_t[0], w.nk_t[1]);
    // the last full pair also stages every key the remainder rows see
    if (kSplit && p.nrem > 0 && it.mp == p.nPairs - 1 && w.valid_seq)
        w.nk = max(w.nk, (it.S - 1) / BN + 1);
    w.ntiles = (2 * it.mp + 1 < it.nM) ? 2 : 1;
    const int ns = kSplit ? p.nsplit : 1;
    w.j0 = kSplit ? it.c * w.nk / ns : 0;
    const int j1 = kSplit ? (it.c + 1) * w.nk / ns : w.nk;
#pragma unroll
    for (int t = 0; t < 2; ++t) w.nkc_t[t] = max(0, min(j1, w.nk_t[t]) - w.j0);
    // (every tile of the chunk is staged: the last full pair's remainder rows
    // may see a key tile past both of its query tiles' frontiers)
    w.nkc = max(0, j1 - w.j0);
    return w;
}

// The last key any row of the query tile starting at position l0 sees.
__device__ __forceinline__ int tile_last_key(const PrefillParams& p, const Item& it, int l0) {
    const int l_last = min(l0 + p.Lt, it.Lb) - 1;
    return min(p.causal ? l_last + it.S - it.Lb : it.S - 1, it.S - 1);
}

// kMask: an explicit additive mask is read; kVarlen: a ragged batch (queries
// packed by token, per-sequence query counts); kSplit: the keys of each pair
// are cut into p.nsplit chunks that write fp32 partials.  Separate
// instantiations, so the plain kernel carries none of their code or registers.
//
// Persistent: one CTA per SM claims work items (query-tile pairs) from a
// counter in the workspace until none are left, so one item's set-up, query
// load and first K/V tiles overlap the previous item's last products and
// epilogue instead of each CTA paying them alone.  The producer publishes
// each item through a 2-slot ring in shared memory; every role runs the
// item's steps with its own running counts of the barriers' phases.
template <bool kMask, bool kVarlen, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tile_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o,
                        const __grid_constant__ CUtensorMap tm_m, const PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const sbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + kOffBar;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    volatile int* const abort_flag = reinterpret_cast<volatile int*>(sbase + kOffAbort);
    uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(sbase + kOffTmemSlot);
    int4* const item_slot = reinterpret_cast<int4*>(sbase + kOffItems);  // [2][2]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if constexpr (kVarlen) pdl_launch_dependents();  // a page walk may start beside us

    // ---- set-up: barriers, V zeroed, TMEM --------------------------------------
    if (tid == 0) {
        mbar_init(bar(kQFull), 1);
        mbar_init(bar(kQEmpty), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(kKFull + s), 1);
            mbar_init(bar(kKEmpty + s), (kSplit && p.nrem > 0) ? 3 : 1);  // + warps 2, 3
            mbar_init(bar(kSFull + s), 1);
            mbar_init(bar(kPFull + s), 4);
            mbar_init(bar(kODone + s), 1);
            mbar_init(bar(kOFree + s), 4);
            mbar_init(bar(kVFull + s), 1);
            mbar_init(bar(kVEmpty + s), (kSplit && p.nrem > 0) ? 3 : 1);
            mbar_init(bar(kItemFull + s), 1);
            // the MMA thread + 8 softmax warps (+ warps 2 and 3 for remainder
            // rows, + warp 2 that stages the mask)
            mbar_init(bar(kItemEmpty + s), (kSplit && p.nrem > 0) ? 11 : kMask ? 10 : 9);
            if (kMask) {
                for (int t = 0; t < 2; ++t) mbar_init(bar(kMaskFull + 3 * t + s), 1);
                mbar_init(bar(kMaskEmpty + s), 4);
            }
        }
        if (kMask) {  // the third mask slot
            for (int t = 0; t < 2; ++t) mbar_init(bar(kMaskFull + 3 * t + 2), 1);
            mbar_init(bar(kMaskEmpty + 2), 4);
        }
        mbar_init(bar(kMmaDone), 1);
        mbar_init(bar(kVTail), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // V rows that are never loaded must hold finite values (their weight is
    // exactly 0, and 0 * NaN would not be).  A key tile that ends past the
    // context leaves such rows when no box reaches them; later uses of a slot
    // find the finite rows of an earlier tile there, the first use these
    // zeros.  (A tile whose last box runs past the context is zeroed after
    // its copy lands: kVTail.)
    {
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

    // Item k sits in ring slot k & 1 until every reader has arrived on
    // kItemEmpty.
    auto read_item = [&](int k) {
        const int4 a = item_slot[2 * (k & 1)], c = item_slot[2 * (k & 1) + 1];
        return Item{a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w & 1, c.w >> 1};
    };
    using KR = KRing<kMask>;
    using VR = KRing<kMask>;
    auto take_item = [&](int k, Item& it) -> bool {  // a whole warp
        if (!warp_wait(bar(kItemFull + (k & 1)), (k >> 1) & 1)) return false;
        it = read_item(k);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kItemEmpty + (k & 1)));
        return true;
    };

    if (warp == 0) {
        // ============================ TMA producer ============================
        const uint64_t pol_q = l2_policy_evict_first();
        const uint64_t pol_kv = l2_policy_evict_last();
        const int n_items = kVarlen ? __ldg(p.pair_prefix + p.B) * p.H_kv : p.n_items;
        if (lane == 0) {
            tc::prefetch_tensormap(&tm_q);
            tc::prefetch_tensormap(&tm_k);
            tc::prefetch_tensormap(&tm_v);
        }
        auto claim = [&]() {
            return __shfl_sync(0xffffffffu, lane == 0 ? atomicAdd(p.item_counter, 1) : 0, 0);
        };
        int idx = claim();
        int kt = 0;       // K/V tiles issued before this item (ring position)
        int qn = 0;       // items whose queries were loaded
        int vtails = 0;   // tail-tile copies (kVTail phases)
        int kdone = 0, vdone = 0;  // K and V tiles issued in all
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const Item it = decode_item<kVarlen, kSplit>(p, idx, n_items);
            const int next = it.live ? claim() : idx;  // the next item's claim goes out early
            const ItemWork w = item_work<kSplit>(p, it);
            if (k >= 2 && !warp_wait(bar(kItemEmpty + (k & 1)), ((k >> 1) - 1) & 1)) {
                if (lane == 0) give_up(p, abort_flag);
                break;
            }
            if (lane == 0) {
                item_slot[2 * (k & 1)] = make_int4(it.b, it.kvh, it.mp, it.S);
                item_slot[2 * (k & 1) + 1] = make_int4(it.Lb, it.q0, it.nM, it.live | (it.c << 1));
                mbar_arrive(bar(kItemFull + (k & 1)));
            }
            __syncwarp();
            if (!it.live) break;
            idx = next;
            if (!w.valid_seq && lane == 0) atomicOr(p.flag, PA_FLAG_BAD_CONTEXT);
            if (w.nkc == 0) continue;
            // the query tiles, once the previous item's products have read theirs
            if (qn > 0 && !warp_wait(bar(kQEmpty), (qn - 1) & 1)) {
                if (lane == 0) give_up(p, abort_flag);
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(kQFull),
                                      static_cast<uint32_t>(w.ntiles * p.G * p.Lt * 128 * 2));
                for (int t = 0; t < w.ntiles; ++t)
                    for (int g = 0; g < p.G; ++g) {
                        const uint32_t dst = base + kOffQ + t * kTile + g * p.Lt * 128;
                        if constexpr (kVarlen) {  // map (D, H_q, tokens): Lt tokens of one head
                            for (int h = 0; h < 2; ++h)
                                tc::tma_load_3d(dst + h * kHalf, &tm_q, h * 64, it.kvh * p.G + g,
                                                it.q0 + w.l0_t[t], bar(kQFull), pol_q);
                        } else {
                            const int row = ((it.b * p.H_q) + it.kvh * p.G + g) * p.L + w.l0_t[t];
                            for (int h = 0; h < 2; ++h)
                                tc::tma_load_2d(dst + h * kHalf, &tm_q, h * 64, row, bar(kQFull),
                                                pol_q);
                        }
                    }
            }
            __syncwarp();
            ++qn;
            // the K/V tile whose last box runs past the context (its V rows
            // past the context are zeroed before the MMA may read it), or -1
            const int tail_tile = (it.S % p.box_rows != 0) ? (it.S - 1) / BN : -1;
            int rows_cur[4], rows_next[4] = {-1, -1, -1, -1};
            uint32_t bytes_cur, bytes_next = 0;
            tile_boxes(p, it.b, it.kvh, it.S, w.j0, lane, rows_cur, bytes_cur);
            for (int jj = 0; jj < w.nkc; ++jj) {
                const int j = w.j0 + jj;  // key tile
                const int gk = kt + jj, s = gk & 1, ks = KR::slot(gk);
                if (gk >= KR::kSlots && !warp_wait(bar(kKEmpty + ks), KR::empty_parity(gk))) {
                    if (lane == 0) give_up(p, abort_flag);
                    ok = false;
                    break;
                }
                if (aborted(abort_flag)) {
                    ok = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(bar(kKFull + ks), bytes_cur);
                __syncwarp();
                issue_boxes(&tm_k, base + kOffK + ks * kTile, rows_cur, lane, p.box_rows,
                            bar(kKFull + ks), pol_kv);
                kdone = gk + 1;
                const int vs = VR::slot(gk);
                if (gk >= VR::kSlots && !warp_wait(bar(kVEmpty + vs), VR::empty_parity(gk))) {
                    if (lane == 0) give_up(p, abort_flag);
                    ok = false;
                    break;
                }
                const bool vtail = j == tail_tile;
                const uint32_t vbar = vtail ? bar(kVTail) : bar(kVFull + vs);
                if (lane == 0) mbar_arrive_expect_tx(vbar, bytes_cur);
                __syncwarp();
                issue_boxes(&tm_v, base + kOffV + vs * kTile, rows_cur, lane, p.box_rows, vbar,
                            pol_kv);
                // rows of the next tile, looked up before waiting for a free slot
                if (jj + 1 < w.nkc) tile_boxes(p, it.b, it.kvh, it.S, j + 1, lane, rows_next, bytes_next);
                if (vtail) {  // the item's last tile: nothing of this item waits behind it
                    if (!warp_wait(bar(kVTail), vtails & 1)) {
                        if (lane == 0) give_up(p, abort_flag);
                        ok = false;
                        break;
                    }
                    ++vtails;
                    for (int r = it.S - j * BN + lane; r < BN; r += 32) {
                        uint4* const vrow =
                            reinterpret_cast<uint4*>(sbase + kOffV + vs * kTile + r * 128);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            vrow[q] = make_uint4(0u, 0u, 0u, 0u);
                            vrow[kHalf / 16 + q] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    fence_proxy_async_smem();  // the MMA reads them through the async proxy
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kVFull + vs));
                }
                vdone = gk + 1;
#pragma unroll
                for (int q = 0; q < 4; ++q) rows_cur[q] = rows_next[q];
                bytes_cur = bytes_next;
            }
            kt += w.nkc;
        }
        // let every copy into this CTA's shared memory land before leaving
        if (qn > 0 && !mbar_wait(bar(kQFull), (qn - 1) & 1)) give_up(p, abort_flag);
        for (int g = max(0, kdone - KR::kSlots); g < kdone; ++g)
            if (!mbar_wait(bar(kKFull + KR::slot(g)), KR::full_parity(g))) give_up(p, abort_flag);
        for (int g = max(0, vdone - VR::kSlots); g < vdone; ++g)
            if (!mbar_wait(bar(kVFull + VR::slot(g)), VR::full_parity(g))) give_up(p, abort_flag);
        // the last CTA to stop claiming resets the counters for the next call
        if (lane == 0) {
            __threadfence();
            if (atomicAdd(p.item_counter + 1, 1) == static_cast<int>(gridDim.x) - 1) {
                atomicExch(p.item_counter, 0);
                atomicExch(p.item_counter + 1, 0);
                __threadfence();
            }
        }
    } else if (warp == 1) {
        // ============================ MMA issuer =============================
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_bf16(BM, BN, 0, 0);  // Q, K both K-major
            constexpr uint32_t idO = tc::idesc_bf16(BM, kD, 0, 1);  // P K-major, V MN-major
            // Operand descriptors of every tile base, formed once; a k-step's
            // descriptor is the base one advanced by its byte offset.
            const uint64_t dQ0 = tc::smem_desc_sw128(base + kOffQ, 16, 1024);
            const uint64_t dQ1 = tc::smem_desc_sw128(base + kOffQ + kTile, 16, 1024);
            const uint64_t dK0 = tc::smem_desc_sw128(base + kOffK, 16, 1024);
            const uint64_t dK1 = tc::smem_desc_sw128(base + kOffK + kTile, 16, 1024);
            const uint64_t dV0 = tc::smem_desc_sw128(base + kOffV, kHalf, 1024);
            const uint64_t dV1 = tc::smem_desc_sw128(base + kOffV + kTile, kHalf, 1024);
            auto qk = [&](int t, int gk) {
                const uint64_t dq = t ? dQ1 : dQ0, dk = KR::slot(gk) ? dK1 : dK0;
                const uint32_t d = tmem + col_s(t);
                tc::mma_bf16_c<0>(d, dq, dk, idS);
#pragma unroll
                for (int kk = 1; kk < kD / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * kHalf + (kk & 3) * 32;
                    tc::mma_bf16_c<1>(d, tc::desc_advance(dq, koff), tc::desc_advance(dk, koff), idS);
                }
                tc::commit(bar(kSFull + t));
            };
            // P is read from Tensor Memory, where the softmax left it over
            // the first 64 columns of the tile's S (8 columns per 16 keys).
            // The next Q.K^T into those columns is issued after this product,
            // and the tensor core runs one thread's MMAs in issue order.
            auto pv = [&](int t, int j, int gk) {
                const uint64_t dv = VR::slot(gk) ? dV1 : dV0;
                const uint32_t d = tmem + col_o(t), a = tmem + col_s(t);
                if (j > 0) tc::mma_bf16_ts_c<1>(d, a, dv, idO);
                else tc::mma_bf16_ts_c<0>(d, a, dv, idO);
#pragma unroll
                for (int kk = 1; kk < BN / 16; ++kk)
                    tc::mma_bf16_ts_c<1>(d, a + kk * 8, tc::desc_advance(dv, kk * 16 * 128), idO);
                tc::commit(bar(kODone + t));
            };
            int kt = 0, qn = 0;
            int pc[2] = {0, 0};  // P fills consumed per tile (kPFull phases)
            int oe[2] = {0, 0};  // epilogues of each tile so far (kOFree phases)
            bool ok = true;
            Item it;
            for (int k = 0; ok; ++k) {
                ok = mbar_wait(bar(kItemFull + (k & 1)), (k >> 1) & 1);
                if (!ok) break;
                it = read_item(k);
                mbar_arrive(bar(kItemEmpty + (k & 1)));
                if (!it.live) break;
                const ItemWork w = item_work<kSplit>(p, it);
                if (w.nkc == 0) continue;
                const int* nk_t = w.nkc_t;  // this item's tiles (j counts from its first)
                const int nk = w.nkc;
                ok = mbar_wait(bar(kQFull), qn & 1) && mbar_wait(bar(kKFull + KR::slot(kt)), KR::full_parity(kt));
                if (!ok || *abort_flag) break;
                tc::fence_after_sync();
                if (nk_t[0] > 0) qk(0, kt);
                if (nk_t[1] > 0) qk(1, kt);
                tc::commit(bar(kKEmpty + KR::slot(kt)));
                if (nk == 1) tc::commit(bar(kQEmpty));  // all of the item's Q.K^T issued
                for (int j = 0; ok && j < nk; ++j) {
                    const int gk = kt + j;
                    ok = mbar_wait(bar(kVFull + VR::slot(gk)), VR::full_parity(gk));
                    if (!ok || *abort_flag) break;
                    const bool more = j + 1 < nk;
                    if (j < nk_t[0]) {
                        ok = mbar_wait(bar(kPFull), pc[0] & 1);
                        // O_A is overwritten by this item's first P.V: the
                        // previous item's epilogue must have read it
                        if (ok && j == 0 && oe[0] > 0) ok = mbar_wait(bar(kOFree), (oe[0] - 1) & 1);
                        if (!ok || *abort_flag) break;
                        ++pc[0];
                        tc::fence_after_sync();
                        pv(0, j, gk);
                    }
                    if (more) {
                        ok = mbar_wait(bar(kKFull + KR::slot(gk + 1)), KR::full_parity(gk + 1));
                        if (!ok || *abort_flag) break;
                        tc::fence_after_sync();
                        if (j + 1 < nk_t[0]) qk(0, gk + 1);
                    }
                    if (j < nk_t[1]) {
                        ok = mbar_wait(bar(kPFull + 1), pc[1] & 1);
                        if (ok && j == 0 && oe[1] > 0)
                            ok = mbar_wait(bar(kOFree + 1), (oe[1] - 1) & 1);
                        if (!ok || *abort_flag) break;
                        ++pc[1];
                        tc::fence_after_sync();
                        pv(1, j, gk);
                    }
                    tc::commit(bar(kVEmpty + VR::slot(gk)));
                    if (more) {
                        if (j + 1 < nk_t[1]) qk(1, gk + 1);
                        tc::commit(bar(kKEmpty + KR::slot(gk + 1)));
                        if (j + 2 == nk) tc::commit(bar(kQEmpty));  // the item's last Q.K^T
                    }
                }
                if (nk_t[0] > 0) ++oe[0];
                if (nk_t[1] > 0) ++oe[1];
                kt += nk;
                ++qn;
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
        const float c = p.scale_log2;
        // with an explicit mask the scores are taken to log2 units (and the
        // mask added) right after the load, so the rest scales by 1
        const float cs = kMask ? 1.f : c;
        int sc = 0;               // S fills of this tile consumed (kSFull phases)
        int pvA = 0, pvB = 0;     // P.V products of tiles A and B in earlier items (kODone phases)
        int mask_ts = 0;          // mask (query tile, key tile) steps staged for earlier items
        int mf0 = 0, mf1 = 0, mf2 = 0;  // this tile's mask fills consumed per slot
        bool ok = true;
        Item it;
        for (int k = 0; ok; ++k) {
            ok = take_item(k, it);
            if (!ok || !it.live) break;
            const ItemWork w = item_work<kSplit>(p, it);
            const int nkA = w.nkc_t[0], nkB = w.nkc_t[1];
            const int nkt = t == 0 ? nkA : nkB;
            const int pv_own = t == 0 ? pvA : pvB;
            const int lim_min = t == 0 ? w.lim_min_t[0] : w.lim_min_t[1];
            const int g = r / p.Lt, l = (t == 0 ? w.l0_t[0] : w.l0_t[1]) + (r - g * p.Lt);
            const bool row_valid = t < w.ntiles && g < p.G && l < it.Lb;
            const int h = it.kvh * p.G + g;
            const int S = it.S, Lb = it.Lb;
            const int lim = min(p.causal ? l + S - Lb : S - 1, S - 1);
            // output row (b, h, l): [B, H_q, L, D], or [tokens, H_q, D] from token q0
            const long long orow_idx =
                kVarlen ? (static_cast<long long>(it.q0 + l) * p.H_q + h)
                        : ((static_cast<long long>(it.b) * p.H_q + h) * p.L + l);
            // the last key any row of this tile sees: mask columns past it are
            // not staged (no key split with a mask: j0 = 0)
            const int lim_tile = tile_last_key(p, it, t == 0 ? w.l0_t[0] : w.l0_t[1]);
            float mrow = neg_inf();
            float2 lsum2 = make_float2(0.f, 0.f);
            for (int j = 0; j < nkt; ++j) {  // j: this item's tile count, jt the key tile
                const int jt = w.j0 + j;
                ok = warp_wait(bar(kSFull + t), (sc + j) & 1);
                if (!ok || aborted(abort_flag)) break;
                tc::fence_after_sync();
                float x[4][32];
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) tc::ld32(trow + col_s(t) + cc * 32, x[cc]);
                tc::wait_ld();
                if constexpr (kMask) {  // s * scale * log2 e + mask * log2 e
                    // the tile's mask, two staged halves of 64 keys; the stager
                    // fills the slots in turn, per key tile tile A's halves,
                    // then tile B's
                    const int n0 = 2 * (mask_ts + min(j, nkA) + min(j, nkB) + (t == 1 && j < nkA ? 1 : 0));
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int ms = (n0 + hh) % kMaskSlots;
                        const int f = ms == 0 ? mf0 : ms == 1 ? mf1 : mf2;  // this tile's fills of the slot so far
                        ok = warp_wait(bar(kMaskFull + 3 * t + ms), f & 1);
                        if (!ok) break;
                        if (ms == 0) ++mf0;
                        else if (ms == 1) ++mf1;
                        else ++mf2;
                        const uint32_t sb = base + mask_off(ms);
#pragma unroll
                        for (int cb = 0; cb < 2; ++cb) {
                            const int cc = 2 * hh + cb;
                            if (jt * BN + 32 * cc > lim_tile) continue;  // not staged: masked below
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                float4 mv;
                                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                             : "=f"(mv.x), "=f"(mv.y), "=f"(mv.z), "=f"(mv.w)
                                             : "r"(sb + cb * (BM * 128) + r * 128 + ((q ^ (r & 7)) << 4)));
                                const int e = 4 * q;
                                x[cc][e + 0] = fmaf(x[cc][e + 0], c, mv.x * 1.4426950408889634f);
                                x[cc][e + 1] = fmaf(x[cc][e + 1], c, mv.y * 1.4426950408889634f);
                                x[cc][e + 2] = fmaf(x[cc][e + 2], c, mv.z * 1.4426950408889634f);
                                x[cc][e + 3] = fmaf(x[cc][e + 3], c, mv.w * 1.4426950408889634f);
                            }
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(kMaskEmpty + ms));
                    }
                    if (!ok) break;
                }
                // causal / length mask (frontier tiles only), row max of raw scores
                const bool masking = jt * BN + BN - 1 > lim_min;  // uniform over the CTA
                if (masking) {
                    const int cmax = lim - jt * BN;  // columns <= cmax are visible
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
                    ok = warp_wait(bar(kODone + t), (pv_own + j - 1) & 1);
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
                // P over the first 64 columns of this tile's S (read above)
                tc::st32(trow + col_s(t), *reinterpret_cast<const uint32_t(*)[32]>(pw));
                tc::st32(trow + col_s(t) + 32, *reinterpret_cast<const uint32_t(*)[32]>(pw + 32));
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kPFull + t));
            }
            if (!ok) break;
            const float lsum = lsum2.x + lsum2.y;
            // a split pair: this chunk's (m, l) of every row, o of rows with keys
            constexpr bool split = kSplit;
            const long long prow = kSplit ? orow_idx * p.nsplit + it.c : 0;
            if (split && row_valid) p.part_ml[prow] = make_float2(nkt > 0 ? mrow : neg_inf(), lsum);
            if (nkt > 0) {
                if (!warp_wait(bar(kODone + t), (pv_own + nkt - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
                if constexpr (split) {
                    // fp32 partial rows (512-byte aligned), 256-bit stores
#pragma unroll 1
                    for (int cc = 0; cc < 4; ++cc) {
                        float o[32];
                        tc::ld32(trow + col_o(t) + cc * 32, o);
                        tc::wait_ld();
                        if (row_valid) {
                            float* const po = p.part_o + prow * kD + cc * 32;
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                st_global_v8(po + 8 * q, *reinterpret_cast<const uint32_t(*)[8]>(o + 8 * q));
                        }
                    }
                } else {
                    // O/l as bf16: each warp's rows go out 16 at a time through
                    // its staging slice and one tiled store per 64-dim half
                    // (rows of one head, consecutive positions, all valid);
                    // other rows are stored directly
                    const uint32_t stage = base + kOffStage + (t * 4 + q4) * (kStageRows * 256);
                    uint16_t* const orow = static_cast<uint16_t*>(p.out) + orow_idx * kD;
#pragma unroll 1
                    for (int rd = 0; rd < 2; ++rd) {
                        const bool mine = (lane >> 4) == rd;
                        // (a ragged batch's short chunks gained nothing from it: measured)
                        const bool tiled = !kVarlen && !kMask && p.Lt % kStageRows == 0 &&
                                           __all_sync(0xffffffffu, !mine || row_valid);
                        if (tiled) {
                            if (lane == 0) tc::bulk_wait_read();  // the slice's last stores
                            __syncwarp();
                        }
                        const int rr = lane & 15;
#pragma unroll 1
                        for (int cc = 0; cc < 4; ++cc) {
                            float o[32];
                            tc::ld32(trow + col_o(t) + cc * 32, o);
                            tc::wait_ld();
                            if (!mine || !row_valid) continue;
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int e = q * 8;
                                const uint4 wv = make_uint4(pack_bf16x2(o[e + 0] * inv, o[e + 1] * inv),
                                                            pack_bf16x2(o[e + 2] * inv, o[e + 3] * inv),
                                                            pack_bf16x2(o[e + 4] * inv, o[e + 5] * inv),
                                                            pack_bf16x2(o[e + 6] * inv, o[e + 7] * inv));
                                if (tiled) {
                                    const int qq = cc * 4 + q;  // 16-byte chunk of the row
                                    const uint32_t a = stage + (qq >> 3) * (kStageRows * 128) + rr * 128 +
                                                       (((qq & 7) ^ (rr & 7)) << 4);
                                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                                                 "r"(wv.x), "r"(wv.y), "r"(wv.z), "r"(wv.w)
                                                 : "memory");
                                } else {
                                    *reinterpret_cast<uint4*>(orow + cc * 32 + e) = wv;
                                }
                            }
                        }
                        if (tiled) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            const int src = 16 * rd;  // the round's first row
                            {
                                const int row0 = static_cast<int>(
                                    __shfl_sync(0xffffffffu, static_cast<unsigned long long>(orow_idx), src));
                                if (lane == 0) {
                                    tc::tma_store_2d(&tm_o, stage, 0, row0);
                                    tc::tma_store_2d(&tm_o, stage + kStageRows * 128, 64, row0);
                                    tc::bulk_commit();
                                }
                            }
                        }
                    }
                }
                // O of this tile is read: the next item's first P.V may overwrite it
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kOFree + t));
            }
            if (!w.valid_seq && row_valid && !split) {
                uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow_idx * kD);
                for (int q = 0; q < kD / 8; ++q) orow[q] = make_uint4(0u, 0u, 0u, 0u);
            }
            sc += nkt;
            pvA += nkA;
            pvB += nkB;
            mask_ts += nkA + nkB;
        }
        if (!ok && lane == 0) give_up(p, abort_flag);
        if (lane == 0) tc::bulk_wait_all();  // the output stores have landed
    } else if (kMask && warp == 2) {
        // ====================== mask stager (warp 2, with a mask) ===================
        // Per key tile and query tile (A, then B), two half-tiles of 64 keys
        // into the three mask slots in turn: per 32-key column block with a
        // visible key, G boxes (one per head) of Lt rows.  (Prefetching the
        // next key tile's boxes into L2 as well, with TMA or per-thread
        // prefetches, made the masked prefill 7-60% slower: measured.)
        const uint64_t pol_m = l2_policy_evict_first();
        if (lane == 0) tc::prefetch_tensormap(&tm_m);
        int n = 0;                     // half-tiles staged
        int fills[2][kMaskSlots] = {};  // per query tile and slot
        bool ok = true;
        Item it;
        auto row_of = [&](const ItemWork& w, int t, int g) {
            return ((it.b * p.H_q) + it.kvh * p.G + g) * p.L + w.l0_t[t];
        };
        for (int k = 0; ok; ++k) {
            ok = take_item(k, it);
            if (!ok || !it.live) break;
            const ItemWork w = item_work<kSplit>(p, it);
            const int lim_t[2] = {tile_last_key(p, it, w.l0_t[0]), tile_last_key(p, it, w.l0_t[1])};
            for (int j = 0; ok && j < w.nkc; ++j) {
                for (int t = 0; t < 2 && ok; ++t) {
                    if (j >= w.nkc_t[t]) continue;
                    const int k0 = (w.j0 + j) * BN;
                    for (int hh = 0; hh < 2; ++hh) {
                        const int ms = n % kMaskSlots;
                        if (n >= kMaskSlots &&
                            !warp_wait(bar(kMaskEmpty + ms), ((n / kMaskSlots) - 1) & 1)) {
                            ok = false;
                            break;
                        }
                        if (aborted(abort_flag)) {
                            ok = false;
                            break;
                        }
                        int nb = 0;  // column blocks with a visible key
                        for (int cb = 0; cb < 2; ++cb) nb += (k0 + kMaskHalf * hh + 32 * cb <= lim_t[t]);
                        if (lane == 0) {
                            const uint32_t sb = base + mask_off(ms);
                            const uint32_t full = bar(kMaskFull + 3 * t + ms);
                            mbar_arrive_expect_tx(full, static_cast<uint32_t>(nb * BM * 128));
                            for (int cb = 0; cb < nb; ++cb)
                                for (int g = 0; g < p.G; ++g)
                                    tc::tma_load_2d(sb + cb * (BM * 128) + g * p.Lt * 128, &tm_m,
                                                    k0 + kMaskHalf * hh + 32 * cb, row_of(w, t, g),
                                                    full, pol_m);
                        }
                        __syncwarp();
                        ++fills[t][ms];
                        ++n;
                    }
                }
            }
        }
        if (!ok && lane == 0) give_up(p, abort_flag);
        // let the staged copies land before leaving
        for (int t = 0; t < 2; ++t)
            for (int ms = 0; ms < kMaskSlots; ++ms)
                if (fills[t][ms] > 0 && !mbar_wait(bar(kMaskFull + 3 * t + ms), (fills[t][ms] - 1) & 1))
                    give_up(p, abort_flag);
    } else if (kSplit && (warp == 2 || warp == 3)) {
        // ====================== remainder rows (warps 2, 3) =====================
        // S^T = K Q^T and O^T += V^T P^T with mma m16n8k16 (16 keys x 8 rows):
        // lane 4g + t holds keys g and g + 8 of rows 2t and 2t + 1, and O^T of
        // dims 16 i + g and 16 i + g + 8 of the same rows (rows past nrem are
        // zero).  P is rounded to bf16 and the row sums add the rounded weights.
        if (p.nrem > 0) {
            const int wr = warp - 2;          // keys 64 wr .. 64 wr + 63 of every tile
            const int g = lane >> 2, t4 = lane & 3;
            const int Lrem = p.L - p.rem_l0;
            const float c = p.scale_log2;
            int kt = 0;
            bool ok = true;
            Item it;
            for (int k = 0; ok; ++k) {
                ok = take_item(k, it);
                if (!ok || !it.live) break;
                const ItemWork w = item_work<true>(p, it);
                const bool rem = it.mp == p.nPairs - 1;
                uint32_t qf[8][2];
                float oacc[8][4];
                float m_r[2] = {neg_inf(), neg_inf()}, l_r[2] = {0.f, 0.f};
                int lim_r[2] = {-1, -1};  // last key each of rows 2t, 2t + 1 sees
                if (rem) {
                    const bool qok = g < p.nrem && w.valid_seq;
                    const int gq = g / Lrem, lq = p.rem_l0 + (g - gq * Lrem);
                    const uint16_t* const qrow =
                        static_cast<const uint16_t*>(p.q) +
                        ((static_cast<long long>(it.b) * p.H_q + it.kvh * p.G + gq) * p.L + lq) * kD;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        qf[ks][0] = qok ? __ldg(reinterpret_cast<const unsigned int*>(qrow + ks * 16 + 2 * t4)) : 0u;
                        qf[ks][1] = qok ? __ldg(reinterpret_cast<const unsigned int*>(qrow + ks * 16 + 8 + 2 * t4)) : 0u;
                    }
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int rr = 2 * t4 + e;
                        const int lr = p.rem_l0 + rr % Lrem;
                        if (rr < p.nrem && w.valid_seq)
                            lim_r[e] = min(p.causal ? lr + it.S - p.L : it.S - 1, it.S - 1);
                    }
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
                }
                for (int jj = 0; jj < w.nkc; ++jj) {
                    const int j = w.j0 + jj, gk = kt + jj, s = gk & 1;
                    // S^T as soon as K lands; K is released before P.V waits for V
                    ok = warp_wait(bar(kKFull + s), (gk >> 1) & 1);
                    if (!ok || aborted(abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t kb = base + kOffK + s * kTile, vb = base + kOffV + s * kTile;
                    const int kw0 = 64 * wr;  // first key of the warp in the tile
                    float sacc[4][4];
                    if (rem) {
                        // the warp's 64 keys as 4 groups of 16, interleaved so
                        // that 4 independent accumulation chains are in flight
#pragma unroll
                        for (int grp = 0; grp < 4; ++grp)
                            sacc[grp][0] = sacc[grp][1] = sacc[grp][2] = sacc[grp][3] = 0.f;
                        {
                            const int r0 = kw0 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                            for (int ks = 0; ks < 8; ++ks) {
                                const int cq = ks * 2 + (lane >> 4);
                                uint32_t a[4][4];
#pragma unroll
                                for (int grp = 0; grp < 4; ++grp) {
                                    const int r = r0 + 16 * grp;
                                    ldmatrix_x4(a[grp], kb + (cq >> 3) * kHalf + r * 128 + (((cq & 7) ^ (r & 7)) << 4));
                                }
#pragma unroll
                                for (int grp = 0; grp < 4; ++grp) mma_16816(sacc[grp], a[grp], qf[ks][0], qf[ks][1]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kKEmpty + s));
                    ok = warp_wait(bar(kVFull + s), (gk >> 1) & 1);
                    if (!ok || aborted(abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (rem) {
                        // scores in log2 units, masked past each row's last key;
                        // one max over the 64 keys per row
                        float mt0 = neg_inf(), mt1 = neg_inf();
#pragma unroll
                        for (int grp = 0; grp < 4; ++grp)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int key = j * BN + kw0 + 16 * grp + g + (e >> 1) * 8;
                                sacc[grp][e] = key <= lim_r[e & 1] ? sacc[grp][e] * c : neg_inf();
                                if (e & 1) mt1 = fmaxf(mt1, sacc[grp][e]);
                                else mt0 = fmaxf(mt0, sacc[grp][e]);
                            }
#pragma unroll
                        for (int o = 4; o < 32; o <<= 1) {
                            mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, o));
                            mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, o));
                        }
                        const bool gr0 = mt0 > m_r[0] + kLazyRescaleLog2;
                        const bool gr1 = mt1 > m_r[1] + kLazyRescaleLog2;
                        if (__any_sync(0xffffffffu, gr0 || gr1)) {
                            const float a0 = gr0 ? fast_exp2(m_r[0] - mt0) : 1.f;
                            const float a1 = gr1 ? fast_exp2(m_r[1] - mt1) : 1.f;
                            if (gr0) m_r[0] = mt0;
                            if (gr1) m_r[1] = mt1;
                            l_r[0] *= a0;
                            l_r[1] *= a1;
#pragma unroll
                            for (int mt = 0; mt < 8; ++mt) {
                                oacc[mt][0] *= a0;
                                oacc[mt][1] *= a1;
                                oacc[mt][2] *= a0;
                                oacc[mt][3] *= a1;
                            }
                        }
                        const float mu0 = m_r[0] == neg_inf() ? 0.f : m_r[0];
                        const float mu1 = m_r[1] == neg_inf() ? 0.f : m_r[1];
                        uint32_t pb[4][2];  // P^T fragments (B operand) per group
#pragma unroll
                        for (int grp = 0; grp < 4; ++grp) {
                            const uint32_t X0 = pack_bf16x2(fast_exp2(sacc[grp][0] - mu0), fast_exp2(sacc[grp][1] - mu1));
                            const uint32_t X1 = pack_bf16x2(fast_exp2(sacc[grp][2] - mu0), fast_exp2(sacc[grp][3] - mu1));
                            const float2 f0 = bf16x2_to_float2(X0), f1 = bf16x2_to_float2(X1);
                            l_r[0] += f0.x + f1.x;
                            l_r[1] += f0.y + f1.y;
                            pb[grp][0] = movmatrix_trans(X0);
                            pb[grp][1] = movmatrix_trans(X1);
                        }
                        // O^T += V^T P^T: consecutive products go to different dims
#pragma unroll
                        for (int grp = 0; grp < 4; ++grp) {
                            const int r = kw0 + 16 * grp + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
                            for (int mt = 0; mt < 8; ++mt) {
                                const int cq = mt * 2 + ((lane >> 3) & 1);
                                uint32_t a[4];
                                ldmatrix_x4_trans(a, vb + (cq >> 3) * kHalf + r * 128 + (((cq & 7) ^ (r & 7)) << 4));
                                mma_16816(oacc[mt], a, pb[grp][0], pb[grp][1]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kVEmpty + s));
                }
                if (!ok) break;
                kt += w.nkc;
                if (rem) {  // this warp's partial of the chunk: (m, l) per row, o^T
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) {
                        l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], o);
                        l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], o);
                    }
                    const int nslot = p.nsplit * 2, slot = it.c * 2 + wr;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int rr = 2 * t4 + e;
                        if (rr >= p.nrem) continue;
                        const long long pr =
                            (static_cast<long long>(it.b * p.H_kv + it.kvh) * p.nrem + rr) * nslot + slot;
                        if (g == 0) p.rem_ml[pr] = make_float2(l_r[e] > 0.f ? m_r[e] : neg_inf(), l_r[e]);
                        float* const po = p.rem_o + pr * kD;
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            po[16 * mt + g] = oacc[mt][e];
                            po[16 * mt + g + 8] = oacc[mt][2 + e];
                        }
                    }
                }
            }
            if (!ok && lane == 0) give_up(p, abort_flag);
        }
    } else {
        // warps 2 and 3 (other instances): readers of no item
    }

    // ---- tear-down: free TMEM once every role is done -----------------------
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// Merges the key chunks of split pairs: one warp per output row (b, h, l) of
// the [B, H_q, L, D] layout, four dims per lane.  Chunks that saw no key of a
// row (m = -inf) weigh nothing; a row with none (a sequence whose context
// breaks the contract) is written as zeros.
__global__ void __launch_bounds__(128) tile_combine_kernel(const PrefillParams p) {
    pdl_wait_primary();
    const long long rows = static_cast<long long>(p.B) * p.H_q * p.L;
    const long long row = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    int ns = p.nsplit;
    const float2* ml = p.part_ml + row * ns;
    const float* po = p.part_o + row * ns * kD;
    if (p.nrem > 0) {  // a remainder row: its partials per (chunk, warp)
        const int l = static_cast<int>(row % p.L);
        if (l >= p.rem_l0) {
            const long long bh = row / p.L;
            const int h = static_cast<int>(bh % p.H_q), b = static_cast<int>(bh / p.H_q);
            const int kvh = h / p.G, rr = (h - kvh * p.G) * (p.L - p.rem_l0) + (l - p.rem_l0);
            ns = 2 * p.nsplit;
            const long long pr = (static_cast<long long>(b * p.H_kv + kvh) * p.nrem + rr) * ns;
            ml = p.rem_ml + pr;
            po = p.rem_o + pr * kD;
        }
    }
    float den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int kFew = 8;
    if (ns <= kFew) {
        // few chunks: every load goes out before the first use
        float2 v[kFew];
        float4 o[kFew];
#pragma unroll
        for (int c = 0; c < kFew; ++c)
            if (c < ns) {
                v[c] = ml[c];
                o[c] = *reinterpret_cast<const float4*>(po + c * kD + 4 * lane);
            }
        float M = neg_inf();
#pragma unroll
        for (int c = 0; c < kFew; ++c)
            if (c < ns) M = fmaxf(M, v[c].x);
        if (M != neg_inf()) {
#pragma unroll
            for (int c = 0; c < kFew; ++c) {
                // (a chunk without keys wrote no o row: skipped, not weighted by 0)
                if (c >= ns || v[c].x == neg_inf()) continue;
                const float a = fast_exp2(v[c].x - M);
                den += a * v[c].y;
                acc.x += a * o[c].x;
                acc.y += a * o[c].y;
                acc.z += a * o[c].z;
                acc.w += a * o[c].w;
            }
        }
    } else {
        float M = neg_inf();
        for (int c = lane; c < ns; c += 32) M = fmaxf(M, ml[c].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        if (M != neg_inf()) {
            for (int c = 0; c < ns; ++c) {
                const float2 v = ml[c];
                if (v.x == neg_inf()) continue;
                const float a = fast_exp2(v.x - M);
                den += a * v.y;
                const float4 o = *reinterpret_cast<const float4*>(po + c * kD + 4 * lane);
                acc.x += a * o.x;
                acc.y += a * o.y;
                acc.z += a * o.z;
                acc.w += a * o.w;
            }
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + row * kD + 4 * lane) =
        make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
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

// fp32 mask map: rows x cols (cols a multiple of 4), boxes of 32 columns x
// box_rows rows, 128-byte swizzle; columns past cols read as zero.
bool make_map_mask(CUtensorMap* map, const float* ptr, long long rows, long long cols, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
    cuuint32_t box[2] = {32u, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box,
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

// Rows of the last query tile handled by warps 2 and 3 of the last full pair
// ([B, H_q, L, D] layout, no mask): G x its positions when the tile is alone
// in its pair and holds at most 8 rows, else 0.
int tile_remainder_rows(const pa_shape& sh) {
    if (!prefill_supported(sh)) return 0;
    const int G = sh.H_q / sh.H_kv, Lt = BM / G;
    const int nM = (sh.L + Lt - 1) / Lt;
    if (nM < 3 || nM % 2 == 0) return 0;
    const int rows = G * (sh.L - (nM - 1) * Lt);
    return rows <= 8 ? rows : 0;
}

int tile_nsplit(const pa_shape& sh, int sm_count) {
    if (!prefill_supported(sh) || sm_count < 1) return 1;
    const int G = sh.H_q / sh.H_kv, Lt = BM / G;
    const long long nM = (sh.L + Lt - 1) / Lt;
    const long long items = (tile_remainder_rows(sh) > 0 ? nM / 2 : (nM + 1) / 2) * sh.B * sh.H_kv;
    // One wave: as many chunks per pair as keep every item on an SM of its
    // own, of at least two key tiles each on the longest context.  Each item
    // a CTA takes after its first costs about three key-tile steps of
    // epilogue, query load and pipeline fill, which on the chunked tails
    // outweighed the balance that more, shorter chunks buy (measured: 2
    // chunks per pair 0.089 ms per call, 3: 0.116, 4: 0.106, 5: 0.096, 8: 0.107).
    if (items >= sm_count) return 1;
    const long long cap_tiles = (static_cast<long long>(sh.max_pages_per_seq) * sh.page_size + BN - 1) / BN;
    long long ns = sm_count / items;
    ns = std::min(ns, std::min(cap_tiles / 2, 16ll));
    return ns > 1 ? static_cast<int>(ns) : 1;
}

size_t tile_partial_bytes(const pa_shape& sh, int sm_count) {
    const long long ns = tile_nsplit(sh, sm_count);
    const int nrem = tile_remainder_rows(sh);
    if (ns <= 1 && nrem == 0) return 0;
    const size_t rows = static_cast<size_t>(sh.B) * sh.H_q * sh.L * ns;
    const size_t rrows = static_cast<size_t>(sh.B) * sh.H_kv * nrem * ns * 2;
    return align_up(rows * 8, 256) + rows * kD * 4 + align_up(rrows * 8, 256) + rrows * kD * 4;
}

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
    CUtensorMap tq, tk, tv, to, tm;
    const long long pool_rows = static_cast<long long>(sh.num_pages) * sh.H_kv * sh.page_size;
    const bool q_ok = c.cu_q ? make_map_tokens(&tq, c.q, sh.H_q, c.total_q, Lt)
                             : make_map(&tq, c.q, static_cast<long long>(sh.B) * sh.H_q * sh.L, Lt);
    // the output in boxes of 16 rows, for the epilogue's tiled stores (the
    // ragged batch's instance stores rows directly and never reads it)
    const bool o_ok = c.cu_q ? (to = tq, true)
                             : make_map(&to, c.out, static_cast<long long>(sh.B) * sh.H_q * sh.L, kStageRows);
    if (!q_ok || !o_ok || !make_map(&tk, c.kp, pool_rows, box_rows) ||
        !make_map(&tv, c.vp, pool_rows, box_rows))
        return PA_ERR_CUDA;
    // the explicit mask [B * H_q * L rows, mask_S columns] fp32, in boxes of
    // 32 columns x Lt rows (one head's rows of a query tile)
    tm = to;
    if (c.mask && !make_map_mask(&tm, c.mask, static_cast<long long>(sh.B) * sh.H_q * sh.L, c.mask_S, Lt))
        return PA_ERR_CUDA;

    static int attr_done[64] = {0};
    if (c.dev.device >= 0 && c.dev.device < 64 && !attr_done[c.dev.device]) {
        if (cudaFuncSetAttribute(prefill_tile_kernel<false, false, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(prefill_tile_kernel<false, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(prefill_tile_kernel<true, false, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(prefill_tile_kernel<false, true, false>,
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
    p.item_counter = reinterpret_cast<int*>(static_cast<uint8_t*>(c.ws) + kTileCounterOffset);
    p.nsplit = (c.cu_q || c.mask) ? 1 : tile_nsplit(sh, c.dev.sm_count);
    p.nrem = (c.cu_q || c.mask) ? 0 : tile_remainder_rows(sh);
    p.rem_l0 = 0;
    p.q = c.q;
    p.part_ml = nullptr;
    p.part_o = nullptr;
    p.rem_ml = nullptr;
    p.rem_o = nullptr;
    if (p.nrem > 0) {  // the last tile's rows go to warps 2 and 3 of the last full pair
        p.rem_l0 = (p.nM - 1) * Lt;
        p.nM -= 1;
        p.nPairs = p.nM / 2;
    }
    const bool split = p.nsplit > 1 || p.nrem > 0;  // partials and the merge kernel
    if (split) {
        uint8_t* const ws = static_cast<uint8_t*>(c.ws) + tile_partials_offset(sh, c.dev.sm_count);
        if (c.ws_bytes < tile_partials_offset(sh, c.dev.sm_count) + tile_partial_bytes(sh, c.dev.sm_count))
            return PA_ERR_WORKSPACE;
        const size_t rows = static_cast<size_t>(sh.B) * sh.H_q * sh.L * p.nsplit;
        const size_t rrows = static_cast<size_t>(sh.B) * sh.H_kv * p.nrem * p.nsplit * 2;
        size_t off = 0;
        p.part_ml = reinterpret_cast<float2*>(ws + off);
        off += align_up(rows * 8, 256);
        p.part_o = reinterpret_cast<float*>(ws + off);
        off += rows * kD * 4;
        p.rem_ml = reinterpret_cast<float2*>(ws + off);
        off += align_up(rrows * 8, 256);
        p.rem_o = reinterpret_cast<float*>(ws + off);
    }
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
    // persistent: one CTA per SM (or per item, when there are fewer)
    const long long items = pairs * sh.H_kv * p.nsplit;
    p.n_items = static_cast<int>(items);
    const unsigned grid = static_cast<unsigned>(std::min<long long>(items, c.dev.sm_count));
    if (c.ev_before && cudaEventRecord(c.ev_before, c.stream) != cudaSuccess) return PA_ERR_CUDA;
    if (c.cu_q)  // (a ragged batch takes no explicit mask)
        prefill_tile_kernel<false, true, false><<<grid, kThreads, kSmemBytes, c.stream>>>(tq, tk, tv, to, tm, p);
    else if (c.mask)
        prefill_tile_kernel<true, false, false><<<grid, kThreads, kSmemBytes, c.stream>>>(tq, tk, tv, to, tm, p);
    else if (split)
        prefill_tile_kernel<false, false, true><<<grid, kThreads, kSmemBytes, c.stream>>>(tq, tk, tv, to, tm, p);
    else
        prefill_tile_kernel<false, false, false><<<grid, kThreads, kSmemBytes, c.stream>>>(tq, tk, tv, to, tm, p);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (c.ev_after && cudaEventRecord(c.ev_after, c.stream) != cudaSuccess) return PA_ERR_CUDA;
    if (split) {  // merge the key chunks (may launch while the tiles finish)
        const long long rows = static_cast<long long>(sh.B) * sh.H_q * sh.L;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>((rows + 3) / 4));
        cfg.blockDim = dim3(128);
        cfg.stream = c.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, tile_combine_kernel, p) != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

}  // namespace pa
