// decode.cu -- schedule (a): short queries over a paged K/V pool on CUDA cores.
//
// What it computes is exact paged attention ("Week 3 Day 5: Paged
// FlashAttention", Tasks 1-2): every visible key s of sequence b is read
// from pages[block_table[b, s / page_size], kv_head, s % page_size, :] and
// folded into a per-row online softmax (running max m, running sum l,
// unnormalised accumulator o), in the recurrence of "Week 2 Day 5: Fused
// Decode Attention", Task 2, with exp2 and scale*log2(e) folded once into
// the query ("Week 3 Day 5", Task 2).
//
// How the work is laid out on GB300:
//   * A segment is (b, kv_head, chunk of <= RB query rows).  All G = H_q/H_kv
//     query heads and L positions of one kv head are rows of the same
//     segments, so each K/V byte is read from HBM once.
//   * The keys of all segments, counted in units of TK/7 keys, are cut into
//     about eight equal chunks per SM (stream-K with dynamic chunks): a
//     persistent grid of one CTA per SM starts on one chunk each and claims
//     the rest from an atomic counter, so neither ragged context lengths nor
//     SMs that stream at different speeds leave the grid unbalanced.  Each
//     chunk is cut into tiles of up to TK keys.  A chunk that holds a whole
//     segment writes its normalised output; a segment split across chunks
//     leaves one fp32 partial (m, l, o[D]) per piece, merged by
//     decode_combine_kernel (the split-combine of "Week 2 Day 5", Task 2,
//     across CTAs instead of SIMD groups).
//   * One producer warp resolves page ids through the block table and issues
//     1-D bulk (TMA) copies of the page-contiguous K and V rows of each tile
//     into a 3-stage shared-memory ring (mbarrier completion by bytes).  A
//     tile that crosses a page boundary is simply copied as several pieces.
//   * Seven consumer warps each take TK/7 keys of a stage (seven consumers
//     plus the producer make eight warps, two per SM sub-partition, so each
//     thread may hold up to 255 registers).  P lanes share one
//     key: each lane holds 128/P dims of the query rows in registers (fp32,
//     pre-scaled), forms partial dot products with packed f32x2 FMAs and
//     reduces them with warp shuffles.  State stays in registers; the
//     running max is only moved when a tile raises it by more than 2^8, so
//     the accumulators are rescaled rarely (the result is unchanged: m only
//     needs to bound the exponents).
//   * Warps merge their states through shared memory at the end of each
//     segment piece.  All intra-CTA waits are bounded mbarrier waits.
#include <cuda_bf16.h>

#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

constexpr int kD = kHeadDim;
constexpr float kLazyRescaleLog2 = 8.0f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

struct DecodeParams {
    const void* q;
    const void* kp;
    const void* vp;
    const int32_t* bt;
    const int32_t* ctx;
    void* out;
    float2* part_ml;  // [slots][RB] (m, l) per piece and row
    float* part_o;    // [slots][RB][D]
    int* prefix;      // [B] exclusive unit prefix; [B] = total units; [B+1] = units per chunk
    uint32_t* flag;
    int* chunk_counter;  // next dynamic chunk (fixed workspace offset, 0 between calls)
    int* done_counter;   // CTAs finished (the last one resets both counters)
    int B, H_q, H_kv, L, G, num_pages, ps, max_npg, nchunk, causal;
    long long max_S;
    float scale_log2;
};

template <typename T, int RB_, int P_, int TK_, int NCW_, int NST_>
struct Cfg {
    using Elem = T;
    static constexpr int RB = RB_;    // query rows per segment
    static constexpr int P = P_;      // lanes sharing one key
    static constexpr int TK = TK_;    // keys per stage
    static constexpr int NCW = NCW_;  // consumer warps
    static constexpr int NST = NST_;  // pipeline stages
    static constexpr int ES = sizeof(T);
    static constexpr int ROW = kD * ES;
    static constexpr int HDR = 128;
    static constexpr int QBYTES = RB * ROW;
    static constexpr int KBYTES = TK * ROW;
    static constexpr int STAGE = HDR + QBYTES + 2 * KBYTES;
    static constexpr int MSTRIDE = kD + 2;  // floats per (warp, row) merge record
    static constexpr int MERGE = (NCW * RB * MSTRIDE * 4 + 127) / 128 * 128;
    static constexpr int NBARS = 2 * NST + 2;
    static constexpr int SMEM = NST * STAGE + MERGE + NBARS * 8;
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int KPW = TK / NCW;  // keys per warp per stage
    // Keys per unit of the even split over CTAs; tiles start on unit
    // boundaries and hold at most NCW units.
    static constexpr int GRAN = KPW;
    static constexpr int KPI = 32 / P;    // keys per warp instruction
    static constexpr int IT = KPW / KPI;
    static constexpr int DPL = kD / P;    // dims held per lane
    static constexpr int CH = 16 / ES;    // elements per 16-byte chunk
    static constexpr int NCH = DPL / CH;  // chunks per lane per row
    static_assert(KPW % KPI == 0, "keys per warp must fill whole instructions");
    static_assert(DPL % CH == 0 && DPL % 2 == 0, "lane dims must be whole chunks");
    static_assert(STAGE % 128 == 0, "stage alignment");
    static_assert(TK <= 128, "at most 128 page pieces per tile (4 per producer lane)");
    static_assert(THREADS % 128 == 0, "whole warps per SM sub-partition");
};

struct StageHdr {
    int seg_id, b, kvh, chunk, key0, nvalid, S, flags, slot;
};
enum : int { kStart = 1, kEnd = 2, kFinal = 4, kLast = 8 };

// Chunks of work per CTA on average (the first is static, the rest are
// claimed dynamically).
constexpr int kChunksPerCta = 8;

// Counts this CTA as finished; the last CTA of the grid resets the chunk
// counter and itself, so the next call starts from zero.  Every CTA calls it
// once, after its last claim on the chunk counter.
__device__ __forceinline__ void finish_chunk_counters(const DecodeParams& p, int grid) {
    __threadfence();
    if (atomicAdd(p.done_counter, 1) == grid - 1) {
        atomicExch(p.chunk_counter, 0);
        atomicExch(p.done_counter, 0);
        __threadfence();
    }
}

// The context length the kernels use for sequence b: 0 (no work, rows
// written as zeros) when it breaks the contract.
__device__ __forceinline__ int checked_len(const DecodeParams& p, int b, bool report) {
    const int S = __ldg(p.ctx + b);
    const bool bad = S < 1 || static_cast<long long>(S) > p.max_S || (p.causal && S < p.L);
    if (bad) {
        if (report) atomicOr(p.flag, PA_FLAG_BAD_CONTEXT);
        return 0;
    }
    return S;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Inclusive block scan of one int per thread; *total gets the block sum.
template <int NT>
__device__ int block_incl_scan(int v, int* sw, int* total) {
    static_assert(NT % 32 == 0 && NT / 32 <= 32, "block size");
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sw[w] = x;
    __syncthreads();
    if (w == 0) {
        int t = lane < NT / 32 ? sw[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < NT / 32) sw[lane] = t;
    }
    __syncthreads();
    const int r = x + (w > 0 ? sw[w - 1] : 0);
    *total = sw[NT / 32 - 1];
    __syncthreads();
    return r;
}

// One lane's DPL dims of a row: chunks li, li+P, li+2P, ... of 16 bytes.
template <class C>
__device__ __forceinline__ void load_row(const uint8_t* row, int li, float2 (&v)[C::DPL / 2]) {
#pragma unroll
    for (int j = 0; j < C::NCH; ++j) {
        const uint4 u = *reinterpret_cast<const uint4*>(row + (li + j * C::P) * 16);
        if constexpr (sizeof(typename C::Elem) == 2) {
            v[j * 4 + 0] = bf16x2_to_float2(u.x);
            v[j * 4 + 1] = bf16x2_to_float2(u.y);
            v[j * 4 + 2] = bf16x2_to_float2(u.z);
            v[j * 4 + 3] = bf16x2_to_float2(u.w);
        } else {
            v[j * 2 + 0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
            v[j * 2 + 1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
        }
    }
}

// Dim index of lane-element e (0 <= e < DPL).
template <class C>
__device__ __forceinline__ int lane_dim(int li, int e) {
    return (li + (e / C::CH) * C::P) * C::CH + e % C::CH;
}

template <typename T>
__device__ __forceinline__ void store_elem(T* base, long long idx, float v);
template <>
__device__ __forceinline__ void store_elem<__nv_bfloat16>(__nv_bfloat16* base, long long idx,
                                                          float v) {
    reinterpret_cast<uint16_t*>(base)[idx] = float_to_bf16_bits(v);
}
template <>
__device__ __forceinline__ void store_elem<float>(float* base, long long idx, float v) {
    base[idx] = v;
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1) decode_split_kernel(const DecodeParams p) {
    using T = typename C::Elem;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* const stage0 = smem;
    float* const merge = reinterpret_cast<float*>(smem + C::NST * C::STAGE);
    uint64_t* const bars = reinterpret_cast<uint64_t*>(smem + C::NST * C::STAGE + C::MERGE);
    __shared__ int s_scan[32];
    __shared__ int s_start_b, s_start_pref;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8 * C::NST;
    const uint32_t mfull = full0 + 16 * C::NST, mdone = mfull + 8;

    // Rows of a stage the producer does not write must still hold finite
    // values (their scores are masked, their weights are exactly 0).
    for (int i = tid; i < C::NST * C::STAGE / 16; i += C::THREADS)
        reinterpret_cast<uint4*>(stage0)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, C::NCW);
        }
        mbar_init(mfull, C::NCW);
        mbar_init(mdone, C::NCW);
        s_abort = 0;
        s_start_b = -1;
        s_start_pref = 0;
        fence_mbar_init();
    }
    fence_proxy_async_smem();

    // ---- split of the batch's keys into chunks --------------------------------
    // Work is counted in units of C::GRAN keys per segment and cut into about
    // kChunksPerCta equal chunks per CTA.  CTA c starts with chunk c and then
    // claims further chunks from a counter, so SMs that stream faster take
    // more of them.
    const int segs_per_b = p.H_kv * p.nchunk;
    int mine = 0;
    for (int b = tid; b < p.B; b += C::THREADS)
        mine += segs_per_b * ((checked_len(p, b, blockIdx.x == 0) + C::GRAN - 1) / C::GRAN);
    int total;
    block_incl_scan<C::THREADS>(mine, s_scan, &total);
    const int grid = static_cast<int>(gridDim.x);
    const int cu = max(1, (total + grid * kChunksPerCta - 1) / (grid * kChunksPerCta));
    const int nchunks = (total + cu - 1) / cu;
    const int u0 = static_cast<int>(blockIdx.x) * cu;
    int carry = 0;
    for (int base = 0; base < p.B; base += C::THREADS) {
        const int b = base + tid;
        const int v = b < p.B ? segs_per_b * ((checked_len(p, b, false) + C::GRAN - 1) / C::GRAN) : 0;
        int tot;
        const int incl = block_incl_scan<C::THREADS>(v, s_scan, &tot);
        const int excl = carry + incl - v;
        if (b < p.B) {
            if (blockIdx.x == 0) p.prefix[b] = excl;
            if (v > 0 && excl <= u0 && u0 < excl + v) {
                s_start_b = b;
                s_start_pref = excl;
            }
        }
        carry += tot;
    }
    if (blockIdx.x == 0 && tid == 0) {
        p.prefix[p.B] = total;
        p.prefix[p.B + 1] = cu;
    }
    __syncthreads();
    pdl_launch_dependents();
    if (static_cast<int>(blockIdx.x) >= nchunks) {
        if (tid == 0) finish_chunk_counters(p, grid);
        return;
    }

    if (warp == C::NCW) {
        // =========================== producer warp ===========================
        const uint64_t pol = l2_policy_evict_first();
        const uint8_t* const kp = static_cast<const uint8_t*>(p.kp);
        const uint8_t* const vp = static_cast<const uint8_t*>(p.vp);
        const uint8_t* const qp = static_cast<const uint8_t*>(p.q);
        int b = s_start_b, bpref = s_start_pref;
        int S = checked_len(p, b, false);
        int ng = (S + C::GRAN - 1) / C::GRAN;
        int units_b = segs_per_b * ng;
        int issued = 0, i = 0;
        int chunk = static_cast<int>(blockIdx.x);
        int next = __shfl_sync(0xffffffffu, lane == 0 ? atomicAdd(p.chunk_counter, 1) : 0, 0) + grid;
        bool stop = false;
        while (!stop) {
            const int cu0 = chunk * cu, cu1 = min(cu0 + cu, total);
            const bool last_chunk = next >= nchunks;
            for (int u = cu0; u < cu1; ++i) {
                while (u >= bpref + units_b) {
                    bpref += units_b;
                    ++b;
                    S = checked_len(p, b, false);
                    ng = (S + C::GRAN - 1) / C::GRAN;
                    units_b = segs_per_b * ng;
                }
                const int loc = u - bpref;
                const int sib = loc / ng;
                const int g = loc - sib * ng;
                const int kvh = sib / p.nchunk, chunk_r = sib - kvh * p.nchunk;
                const int seg_u0 = bpref + sib * ng, seg_u1 = seg_u0 + ng;  // segment's units
                const int piece_u1 = min(cu1, seg_u1);
                const int stage = i % C::NST;
                const uint32_t fb = full0 + 8 * stage, eb = empty0 + 8 * stage;
                if (i >= C::NST &&
                    !__all_sync(0xffffffffu, mbar_wait(eb, ((i / C::NST) - 1) & 1))) {
                    if (lane == 0) atomicOr(p.flag, PA_FLAG_TIMEOUT);
                    s_abort = 1;
                    stop = true;
                    break;
                }
                if (__any_sync(0xffffffffu, s_abort != 0)) {
                    stop = true;
                    break;
                }
                uint8_t* const st = stage0 + stage * C::STAGE;
                const int key0 = g * C::GRAN;
                const int piece_key1 = min(S, (piece_u1 - seg_u0) * C::GRAN);
                const int nvalid = min(C::TK, piece_key1 - key0);
                const int u_next = u + (nvalid + C::GRAN - 1) / C::GRAN;
                const int lp0 = key0 / p.ps;
                const int nseg = (key0 + nvalid - 1) / p.ps - lp0 + 1;
                int pp[4];
                uint32_t bytes = 0;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const int sidx = lane + 32 * w;
                    pp[w] = -1;
                    if (sidx < nseg) {
                        const int lp = lp0 + sidx;
                        const int v = __ldg(p.bt + static_cast<long long>(b) * p.max_npg + lp);
                        const int klo = max(key0, lp * p.ps);
                        const int khi = min(key0 + nvalid, (lp + 1) * p.ps);
                        if (v >= 0 && v < p.num_pages) {
                            pp[w] = v;
                            bytes += 2u * static_cast<uint32_t>(khi - klo) * C::ROW;
                        } else {
                            atomicOr(p.flag, PA_FLAG_BAD_PAGE);
                        }
                    }
                }
                const bool start = (u == cu0) || (g == 0);
                const int row0 = chunk_r * C::RB;
                const int nrows = min(C::RB, p.G * p.L - row0);
                if (lane == 0 && start) bytes += static_cast<uint32_t>(nrows) * C::ROW;
                bytes = static_cast<uint32_t>(warp_sum(static_cast<int>(bytes)));
                if (lane == 0) {
                    StageHdr* h = reinterpret_cast<StageHdr*>(st);
                    h->seg_id = (b * p.H_kv + kvh) * p.nchunk + chunk_r;
                    h->b = b;
                    h->kvh = kvh;
                    h->chunk = chunk_r;
                    h->key0 = key0;
                    h->nvalid = nvalid;
                    h->S = S;
                    h->slot = h->seg_id + chunk;
                    const bool end = u_next >= piece_u1;
                    h->flags = (start ? kStart : 0) | (end ? kEnd : 0) |
                               ((seg_u0 >= cu0 && seg_u1 <= cu1) ? kFinal : 0) |
                               ((end && piece_u1 == cu1 && last_chunk) ? kLast : 0);
                    mbar_arrive_expect_tx(fb, bytes);
                }
                __syncwarp();
                const uint32_t kdst = smem_u32(st) + C::HDR + C::QBYTES;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    if (pp[w] < 0) continue;
                    const int lp = lp0 + lane + 32 * w;
                    const int klo = max(key0, lp * p.ps);
                    const int khi = min(key0 + nvalid, (lp + 1) * p.ps);
                    const long long row =
                        (static_cast<long long>(pp[w]) * p.H_kv + kvh) * p.ps + (klo - lp * p.ps);
                    const uint32_t nb = static_cast<uint32_t>(khi - klo) * C::ROW;
                    const uint32_t off = static_cast<uint32_t>(klo - key0) * C::ROW;
                    bulk_g2s(kdst + off, kp + row * C::ROW, nb, fb, pol);
                    bulk_g2s(kdst + C::KBYTES + off, vp + row * C::ROW, nb, fb, pol);
                }
                if (lane == 0 && start) {
                    const long long qrow =
                        (static_cast<long long>(b) * p.H_q + static_cast<long long>(kvh) * p.G) * p.L +
                        row0;
                    bulk_g2s(smem_u32(st) + C::HDR, qp + qrow * C::ROW,
                             static_cast<uint32_t>(nrows) * C::ROW, fb, pol);
                }
                issued = i + 1;
                u = u_next;
            }
            if (stop || last_chunk) break;
            chunk = next;
            next = __shfl_sync(0xffffffffu, lane == 0 ? atomicAdd(p.chunk_counter, 1) : 0, 0) + grid;
        }
        // Never leave with copies in flight into this CTA's shared memory.
        for (int k = max(0, issued - C::NST); k < issued; ++k)
            if (!mbar_wait(full0 + 8 * (k % C::NST), (k / C::NST) & 1))
                atomicOr(p.flag, PA_FLAG_TIMEOUT);
        if (lane == 0) finish_chunk_counters(p, grid);
        return;
    }

    // ============================ consumer warps ============================
    const int grp = lane / C::P, li = lane % C::P;
    float2 q2[C::RB][C::DPL / 2];
    float2 o2[C::RB][C::DPL / 2];
    float mrow[C::RB], lsum[C::RB];
    int lrow[C::RB];
    int lmin = 0;
    int nend = 0;
    T* const out = static_cast<T*>(p.out);
#pragma unroll
    for (int r = 0; r < C::RB; ++r) {
        mrow[r] = neg_inf();
        lsum[r] = 0.f;
        lrow[r] = 0;
#pragma unroll
        for (int e = 0; e < C::DPL / 2; ++e) {
            q2[r][e] = make_float2(0.f, 0.f);
            o2[r][e] = make_float2(0.f, 0.f);
        }
    }

    for (int i = 0;; ++i) {
        const int stage = i % C::NST;
        if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * stage, (i / C::NST) & 1))) {
            if (lane == 0) atomicOr(p.flag, PA_FLAG_TIMEOUT);
            s_abort = 1;
            break;
        }
        if (__any_sync(0xffffffffu, s_abort != 0)) break;
        const uint8_t* const st = stage0 + stage * C::STAGE;
        const StageHdr h = *reinterpret_cast<const StageHdr*>(st);

        if (h.flags & kStart) {
            const int rows = p.G * p.L - h.chunk * C::RB;
            lmin = INT_MAX;
#pragma unroll
            for (int r = 0; r < C::RB; ++r) {
                load_row<C>(st + C::HDR + r * C::ROW, li, q2[r]);
#pragma unroll
                for (int e = 0; e < C::DPL / 2; ++e) {
                    q2[r][e].x *= p.scale_log2;
                    q2[r][e].y *= p.scale_log2;
                    o2[r][e] = make_float2(0.f, 0.f);
                }
                mrow[r] = neg_inf();
                lsum[r] = 0.f;
                lrow[r] = r < rows ? (h.chunk * C::RB + r) % p.L : p.L - 1;
                lmin = min(lmin, lrow[r]);
            }
        }

        const int kw0 = warp * C::KPW;
        if (h.nvalid > kw0) {
            const uint8_t* const Ks = st + C::HDR + C::QBYTES;
            const uint8_t* const Vs = Ks + C::KBYTES;
            float s[C::IT][C::RB];
#pragma unroll
            for (int it = 0; it < C::IT; ++it) {
                const int kl = kw0 + it * C::KPI + grp;
                float2 k2[C::DPL / 2];
                load_row<C>(Ks + kl * C::ROW, li, k2);
#pragma unroll
                for (int r = 0; r < C::RB; ++r) {
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < C::DPL / 2; ++e) acc = __ffma2_rn(q2[r][e], k2[e], acc);
                    float d = acc.x + acc.y;
#pragma unroll
                    for (int o = 1; o < C::P; o <<= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                    s[it][r] = d;
                }
            }
            // Score mask (the separate "second mask" of a masked load): keys
            // past the context or past a row's causal frontier get -inf.
            const int last_key = h.key0 + kw0 + C::KPW - 1;
            const bool tail = h.nvalid < kw0 + C::KPW;
            if (tail || (p.causal && last_key > lmin + h.S - p.L)) {
#pragma unroll
                for (int it = 0; it < C::IT; ++it) {
                    const int kl = kw0 + it * C::KPI + grp;
                    const int kg = h.key0 + kl;
#pragma unroll
                    for (int r = 0; r < C::RB; ++r) {
                        const bool vis = kl < h.nvalid && (!p.causal || kg <= lrow[r] + h.S - p.L);
                        if (!vis) s[it][r] = neg_inf();
                    }
                }
            }
            float mt[C::RB];
            bool resc = false;
#pragma unroll
            for (int r = 0; r < C::RB; ++r) {
                float x = s[0][r];
#pragma unroll
                for (int it = 1; it < C::IT; ++it) x = fmaxf(x, s[it][r]);
#pragma unroll
                for (int o = C::P; o < 32; o <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
                mt[r] = x;
                resc |= x > mrow[r] + kLazyRescaleLog2;
            }
            if (resc) {
#pragma unroll
                for (int r = 0; r < C::RB; ++r) {
                    const float mn = fmaxf(mrow[r], mt[r]);
                    const float a = (mn == neg_inf()) ? 1.f : fast_exp2(mrow[r] - mn);
                    lsum[r] *= a;
#pragma unroll
                    for (int e = 0; e < C::DPL / 2; ++e) {
                        o2[r][e].x *= a;
                        o2[r][e].y *= a;
                    }
                    mrow[r] = mn;
                }
            }
            float mu[C::RB];
#pragma unroll
            for (int r = 0; r < C::RB; ++r) mu[r] = (mrow[r] == neg_inf()) ? 0.f : mrow[r];
#pragma unroll
            for (int it = 0; it < C::IT; ++it) {
                const int kl = kw0 + it * C::KPI + grp;
                float2 v2[C::DPL / 2];
                load_row<C>(Vs + kl * C::ROW, li, v2);
#pragma unroll
                for (int r = 0; r < C::RB; ++r) {
                    const float pr = fast_exp2(s[it][r] - mu[r]);
                    lsum[r] += pr;
                    const float2 pp2 = make_float2(pr, pr);
#pragma unroll
                    for (int e = 0; e < C::DPL / 2; ++e) o2[r][e] = __ffma2_rn(pp2, v2[e], o2[r][e]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);

        if (h.flags & kEnd) {
            // groups of P lanes saw different keys: sum them (same m per warp)
#pragma unroll
            for (int r = 0; r < C::RB; ++r) {
#pragma unroll
                for (int o = C::P; o < 32; o <<= 1) {
                    lsum[r] += __shfl_xor_sync(0xffffffffu, lsum[r], o);
#pragma unroll
                    for (int e = 0; e < C::DPL / 2; ++e) {
                        o2[r][e].x += __shfl_xor_sync(0xffffffffu, o2[r][e].x, o);
                        o2[r][e].y += __shfl_xor_sync(0xffffffffu, o2[r][e].y, o);
                    }
                }
            }
            float* const mw = merge + warp * C::RB * C::MSTRIDE;
            if (lane < C::P) {
#pragma unroll
                for (int r = 0; r < C::RB; ++r) {
#pragma unroll
                    for (int e = 0; e < C::DPL / 2; ++e) {
                        mw[r * C::MSTRIDE + 2 + lane_dim<C>(li, 2 * e)] = o2[r][e].x;
                        mw[r * C::MSTRIDE + 2 + lane_dim<C>(li, 2 * e + 1)] = o2[r][e].y;
                    }
                }
            }
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < C::RB; ++r) {
                    mw[r * C::MSTRIDE] = mrow[r];
                    mw[r * C::MSTRIDE + 1] = lsum[r];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(mfull);
            if (!__all_sync(0xffffffffu, mbar_wait(mfull, nend & 1))) {
                if (lane == 0) atomicOr(p.flag, PA_FLAG_TIMEOUT);
                s_abort = 1;
                break;
            }
            const int rows_valid = min(C::RB, p.G * p.L - h.chunk * C::RB);
            const long long base_row =
                (static_cast<long long>(h.b) * p.H_q + static_cast<long long>(h.kvh) * p.G) * p.L +
                static_cast<long long>(h.chunk) * C::RB;
            const long long slot = h.slot;
            for (int idx = tid; idx < C::RB * kD; idx += C::NCW * 32) {
                const int r = idx / kD, d = idx - r * kD;
                if (r >= rows_valid) continue;
                float M = neg_inf();
#pragma unroll
                for (int w = 0; w < C::NCW; ++w) M = fmaxf(M, merge[(w * C::RB + r) * C::MSTRIDE]);
                float den = 0.f, acc = 0.f;
                if (M != neg_inf()) {
#pragma unroll
                    for (int w = 0; w < C::NCW; ++w) {
                        const float* rec = merge + (w * C::RB + r) * C::MSTRIDE;
                        const float a = fast_exp2(rec[0] - M);
                        den += a * rec[1];
                        acc += a * rec[2 + d];
                    }
                }
                if (h.flags & kFinal) {
                    store_elem<T>(out, (base_row + r) * kD + d, den > 0.f ? acc / den : 0.f);
                } else {
                    p.part_o[(slot * C::RB + r) * kD + d] = acc;
                    if (d == 0) p.part_ml[slot * C::RB + r] = make_float2(M, den);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(mdone);
            if (!__all_sync(0xffffffffu, mbar_wait(mdone, nend & 1))) {
                if (lane == 0) atomicOr(p.flag, PA_FLAG_TIMEOUT);
                s_abort = 1;
                break;
            }
            ++nend;
        }
        if (h.flags & kLast) break;
    }
}

// Four output dims of one row, stored together.
template <typename T>
__device__ __forceinline__ void store4(T* base, long long idx, float4 v);
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* base, long long idx, float4 v) {
    *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(base) + idx) =
        make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}
template <>
__device__ __forceinline__ void store4<float>(float* base, long long idx, float4 v) {
    *reinterpret_cast<float4*>(base + idx) = v;
}

// Merges the pieces of every segment that was split across CTAs (one CTA per
// segment, one warp per row, four dims per lane; the pieces' (m, l) are read
// by the lanes in parallel), and writes zeros for sequences whose context
// length broke the contract.
template <class C>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p) {
    using T = typename C::Elem;
    pdl_wait_primary();
    const int seg = blockIdx.x;
    const int segs_per_b = p.H_kv * p.nchunk;
    const int b = seg / segs_per_b, sib = seg - b * segs_per_b;
    const int kvh = sib / p.nchunk, chunk = sib - kvh * p.nchunk;
    const int S = checked_len(p, b, false);
    const int ng = (S + C::GRAN - 1) / C::GRAN;
    const int rows_valid = min(C::RB, p.G * p.L - chunk * C::RB);
    const long long base_row =
        (static_cast<long long>(b) * p.H_q + static_cast<long long>(kvh) * p.G) * p.L +
        static_cast<long long>(chunk) * C::RB;
    T* const out = static_cast<T*>(p.out);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d0 = lane * 4;
    if (ng == 0) {
        for (int r = warp; r < rows_valid; r += 4)
            store4<T>(out, (base_row + r) * kD + d0, make_float4(0.f, 0.f, 0.f, 0.f));
        return;
    }
    const int per = p.prefix[p.B + 1];
    const int first = p.prefix[b] + sib * ng;
    const int c0 = first / per, c1 = (first + ng - 1) / per;
    if (c0 == c1) return;  // the segment lay in one CTA, which wrote it
    const int np = c1 - c0 + 1;
    const long long slot0 = static_cast<long long>(seg) + c0;
    for (int r = warp; r < rows_valid; r += 4) {
        float M = neg_inf();
        for (int i = lane; i < np; i += 32) M = fmaxf(M, p.part_ml[(slot0 + i) * C::RB + r].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float den = 0.f;
        if (M != neg_inf()) {
            for (int base = 0; base < np; base += 32) {
                const int i = base + lane;
                float a = 0.f;
                if (i < np) {
                    const float2 ml = p.part_ml[(slot0 + i) * C::RB + r];
                    a = fast_exp2(ml.x - M);
                    den += a * ml.y;
                }
                const int n = min(32, np - base);
#pragma unroll 4
                for (int j = 0; j < n; ++j) {
                    const float aj = __shfl_sync(0xffffffffu, a, j);
                    const float4 o = *reinterpret_cast<const float4*>(
                        p.part_o + ((slot0 + base + j) * C::RB + r) * kD + d0);
                    acc.x += aj * o.x;
                    acc.y += aj * o.y;
                    acc.z += aj * o.z;
                    acc.w += aj * o.w;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        store4<T>(out, (base_row + r) * kD + d0,
                  make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct WsLayout {
    size_t prefix_off, ml_off, o_off, total;
    long long nseg, slots;
};

WsLayout ws_layout(const pa_shape& sh, int grid, int RB) {
    const long long G = sh.H_q / sh.H_kv;
    const long long nchunk = (G * sh.L + RB - 1) / RB;
    WsLayout w;
    w.nseg = static_cast<long long>(sh.B) * sh.H_kv * nchunk;
    w.slots = w.nseg + static_cast<long long>(grid) * kChunksPerCta;
    size_t off = kFlagBytes;
    w.prefix_off = off;
    off = align_up(off + 4 * (static_cast<size_t>(sh.B) + 2), 256);
    w.ml_off = off;
    off = align_up(off + 8 * static_cast<size_t>(w.slots) * RB, 256);
    w.o_off = off;
    off += 4 * static_cast<size_t>(w.slots) * RB * kD;
    w.total = off;
    return w;
}

template <class C>
pa_status launch_cfg(const Call& c) {
    const pa_shape& sh = c.sh;
    const int grid = decode_grid(sh, c.dev.sm_count);
    const WsLayout w = ws_layout(sh, grid, C::RB);
    if (c.ws_bytes < w.total) return PA_ERR_WORKSPACE;
    // Bound on the flattened unit count: every index stays inside int.
    const long long max_units = w.nseg * ((static_cast<long long>(sh.max_pages_per_seq) *
                                               sh.page_size + C::GRAN - 1) / C::GRAN);
    if (max_units >= INT_MAX / 2) return PA_ERR_UNSUPPORTED;

    static int attr_done[64] = {0};
    if (c.dev.device >= 0 && c.dev.device < 64 && !attr_done[c.dev.device]) {
        if (cudaFuncSetAttribute(decode_split_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM) != cudaSuccess)
            return PA_ERR_CUDA;
        attr_done[c.dev.device] = 1;
    }
    uint8_t* ws = static_cast<uint8_t*>(c.ws);
    DecodeParams p;
    p.q = c.q;
    p.kp = c.kp;
    p.vp = c.vp;
    p.bt = c.bt;
    p.ctx = c.ctx;
    p.out = c.out;
    p.part_ml = reinterpret_cast<float2*>(ws + w.ml_off);
    p.part_o = reinterpret_cast<float*>(ws + w.o_off);
    p.prefix = reinterpret_cast<int*>(ws + w.prefix_off);
    p.flag = reinterpret_cast<uint32_t*>(ws);
    p.chunk_counter = reinterpret_cast<int*>(ws + kChunkCounterOffset);
    p.done_counter = reinterpret_cast<int*>(ws + kDoneCounterOffset);
    p.B = sh.B;
    p.H_q = sh.H_q;
    p.H_kv = sh.H_kv;
    p.L = sh.L;
    p.G = sh.H_q / sh.H_kv;
    p.num_pages = sh.num_pages;
    p.ps = sh.page_size;
    p.max_npg = sh.max_pages_per_seq;
    p.nchunk = static_cast<int>((static_cast<long long>(p.G) * sh.L + C::RB - 1) / C::RB);
    p.causal = c.causal ? 1 : 0;
    p.max_S = static_cast<long long>(sh.max_pages_per_seq) * sh.page_size;
    p.scale_log2 = c.scale * 1.4426950408889634f;

    if (c.ev_before && cudaEventRecord(c.ev_before, c.stream) != cudaSuccess) return PA_ERR_CUDA;
    decode_split_kernel<C><<<grid, C::THREADS, C::SMEM, c.stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (c.ev_after && cudaEventRecord(c.ev_after, c.stream) != cudaSuccess) return PA_ERR_CUDA;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(w.nseg));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_combine_kernel<C>, p) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

}  // namespace

int decode_rows_per_chunk(const pa_shape& sh) {
    const long long R = static_cast<long long>(sh.H_q / sh.H_kv) * sh.L;
    if (R <= 1) return 1;
    if (R <= 2) return 2;
    if (R <= 4) return 4;
    return 8;
}

int decode_grid(const pa_shape& /*sh*/, int sm_count) { return sm_count > 0 ? sm_count : 1; }

size_t decode_workspace_bytes(const pa_shape& sh, int sm_count) {
    return ws_layout(sh, decode_grid(sh, sm_count), decode_rows_per_chunk(sh)).total;
}

pa_status decode_launch(const Call& c) {
    const int RB = decode_rows_per_chunk(c.sh);
    using bf = __nv_bfloat16;
    if (c.sh.dtype == PA_BF16) {
        switch (RB) {
            case 1: return launch_cfg<Cfg<bf, 1, 8, 112, 7, 3>>(c);
            case 2: return launch_cfg<Cfg<bf, 2, 8, 112, 7, 3>>(c);
            case 4: return launch_cfg<Cfg<bf, 4, 8, 112, 7, 3>>(c);
            default: return launch_cfg<Cfg<bf, 8, 16, 56, 7, 3>>(c);
        }
    }
    switch (RB) {
        case 1: return launch_cfg<Cfg<float, 1, 8, 56, 7, 3>>(c);
        case 2: return launch_cfg<Cfg<float, 2, 8, 56, 7, 3>>(c);
        case 4: return launch_cfg<Cfg<float, 4, 8, 56, 7, 3>>(c);
        default: return launch_cfg<Cfg<float, 8, 16, 28, 7, 3>>(c);
    }
}

}  // namespace pa
