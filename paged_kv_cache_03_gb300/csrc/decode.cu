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
//     about four equal chunks per SM (stream-K with dynamic chunks): a
//     persistent grid of one CTA per SM starts on one chunk each and claims
//     the rest from an atomic counter, so neither ragged context lengths nor
//     SMs that stream at different speeds leave the grid unbalanced.  Each
//     chunk is cut into tiles of up to TK keys.  A chunk that holds a whole
//     segment writes its normalised output; a segment split across chunks
//     leaves one fp32 partial (m, l, o[D]) per piece, merged by
//     decode_combine_kernel (the split-combine of "Week 2 Day 5", Task 2,
//     across CTAs instead of SIMD groups).
//   * One producer warp resolves page ids through the block table and fills
//     a 3-stage shared-memory ring (mbarrier completion by bytes), in one of
//     two forms:
//       - bf16 on pages of a multiple of 64 slots, up to 4 query rows per
//         segment: 128-key tiles that start on 128-key boundaries, landed by
//         2-D TMA boxes with the 128-byte swizzle (one box per operand half
//         when a page holds the whole tile; a segment's last, partial tile
//         in 16-row boxes).  Eight consumer warps take 16 keys each and run
//         S^T = K Q^T and O^T += V^T P^T on the warp-level tensor cores
//         (mma m16n8k16 bf16, fragments by ldmatrix from the swizzled tile,
//         P rounded to bf16 with the row sums adding the rounded weights).
//       - otherwise: 1-D bulk copies of the page-contiguous K and V rows (a
//         tile that crosses a page boundary is several pieces), and seven
//         consumer warps on CUDA cores, TK/7 keys each.  P lanes share one
//         key: each lane holds 128/P dims of the query rows in registers
//         (fp32, pre-scaled), forms partial dot products with packed f32x2
//         FMAs and reduces them with warp shuffles.
//     Few large copies per tile matter: a measured producer spent about 65
//     cycles of issue per TMA request, so 28 requests a tile (16-row boxes)
//     made the single producer warp the bottleneck.
//   * State stays in registers; the running max is only moved when a tile
//     raises it by more than 2^8, so the accumulators are rescaled rarely
//     (the result is unchanged: m only needs to bound the exponents).
//   * Warps merge their states through shared memory at the end of each
//     segment piece.  All intra-CTA waits are bounded mbarrier waits.
#include <cuda_bf16.h>

#include <climits>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

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
    int tk_pages, tk_slots;  // a full tile of TK keys spans TK / ps pages + TK % ps slots
    // tensor-core consumers: TMA box heights in keys, for a full tile (a divisor
    // of the page size and of GRAN) and for a segment's last, partial tile
    int boxr, boxr_tail;
    const float* mask;       // optional additive mask [B * H_q, L, mask_S], or null
    long long mask_S;
    // ragged batch: query rows packed by token [total_q, H_q, D], sequence b
    // owns tokens cu_q[b] .. cu_q[b + 1] - 1; null for the [B, H_q, L, D] layout
    const int32_t* cu_q;
    int total_q;
    int route_mixed;  // 1: sequences with more than L query positions belong to the tiles
};

// MMA_: the consumers run Q.K^T and P.V on the warp-level tensor cores
// (mma m16n8k16, bf16) over K/V tiles that TMA boxes land 128-byte swizzled;
// otherwise they run them on CUDA cores over rows copied as they lie.
template <typename T, int RB_, int P_, int TK_, int NCW_, int NST_, int MINB_ = 1, int GRAN_ = 0,
          bool MMA_ = false>
struct Cfg {
    using Elem = T;
    static constexpr int RB = RB_;    // query rows per segment
    static constexpr int P = P_;      // lanes sharing one key (CUDA-core consumers)
    static constexpr int TK = TK_;    // keys per stage
    static constexpr int NCW = NCW_;  // consumer warps
    static constexpr int NST = NST_;  // pipeline stages
    static constexpr int MINB = MINB_;  // CTAs resident per SM
    static constexpr bool MMA = MMA_;
    static constexpr int ES = sizeof(T);
    static constexpr int ROW = kD * ES;
    static constexpr int HDR = 128;
    static constexpr int QBYTES = RB * ROW;
    static constexpr int KBYTES = TK * ROW;
    // Stage layout.  CUDA-core consumers: header, query rows, K rows, V rows
    // (256-byte rows as they lie in the pool).  Tensor-core consumers: K and
    // V each as two 64-dim halves of TK rows x 128 bytes (128-byte swizzle,
    // every half 1024-byte aligned), then the query rows and the header.
    static constexpr int KHALF = TK * 128;
    static constexpr int OFF_K = MMA ? 0 : HDR + QBYTES;
    static constexpr int OFF_V = MMA ? 2 * KHALF : HDR + QBYTES + KBYTES;
    static constexpr int OFF_Q = MMA ? 4 * KHALF : HDR;
    static constexpr int OFF_HDR = MMA ? 4 * KHALF + QBYTES : 0;
    static constexpr int STAGE =
        MMA ? (4 * KHALF + QBYTES + HDR + 1023) / 1024 * 1024 : HDR + QBYTES + 2 * KBYTES;
    // merge record per (warp, row): o[128] then m, l (16-byte aligned rows)
    static constexpr int MSTRIDE = kD + 4;
    static constexpr int MERGE = (NCW * RB * MSTRIDE * 4 + 127) / 128 * 128;
    // per-warp softmax weights of one stage, [KPW keys][RB rows]
    static constexpr int PBUF = MMA ? 0 : (NCW * (TK / NCW) * RB * 4 + 127) / 128 * 128;
    static constexpr int NBARS = 2 * NST + 2;
    // (+1024: the tensor-core layout aligns its base to 1024 bytes)
    static constexpr int SMEM = NST * STAGE + MERGE + PBUF + NBARS * 8 + (MMA ? 1024 : 0);
    static constexpr int THREADS = (NCW + 1) * 32;
    static constexpr int KPW = TK / NCW;  // keys per warp per stage
    // Keys per unit of the split over CTAs (a power of two dividing TK);
    // tiles start on unit boundaries.
    static constexpr int GRAN = GRAN_ > 0 ? GRAN_ : KPW;
    static_assert(TK % GRAN == 0, "tiles are whole units");
    static constexpr int KPI = 32 / P;    // keys per warp instruction
    static constexpr int IT = KPW / KPI;
    static constexpr int DPL = kD / P;    // dims held per lane
    static constexpr int CH = 16 / ES;    // elements per 16-byte chunk
    static constexpr int NCH = DPL / CH;  // chunks per lane per row
    static_assert(KPW % KPI == 0, "keys per warp must fill whole instructions");
    static_assert(DPL % CH == 0 && DPL % 2 == 0, "lane dims must be whole chunks");
    static_assert(STAGE % 128 == 0, "stage alignment");
    static constexpr int PIECE_ITERS = (TK + 31) / 32;  // page pieces per producer lane (ps = 1)
    static_assert(MMA || (THREADS * MINB) % 128 == 0, "whole warps per SM sub-partition");
    static_assert(!MMA || (ES == 2 && KPW == 16 && RB <= 8 && KHALF % 1024 == 0 &&
                           GRAN % 16 == 0),
                  "tensor-core consumers: bf16, 16 keys per warp, up to 8 rows");
};

struct alignas(16) StageHdr {
    int seg_id, b, kvh, chunk, key0, nvalid, S, flags, slot, Lb, q0, pad2;
};
enum : int { kStart = 1, kEnd = 2, kFinal = 4, kLast = 8 };

// Chunks of work per CTA on average (the first is static, the rest are
// claimed dynamically).
constexpr int kChunksPerCta = 4;

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

// The work of sequence b in this launch.  Lb: its query positions (p.L in
// the [B, H_q, L, D] layout); q0: its first token (ragged batch).  nch = 0:
// the sequence is not this launch's (no new queries, or more than p.L of
// them in a mixed batch, which the tile schedule takes), or its offsets are
// broken (flagged; nothing of it is written).  S = 0 with nch > 0: its context
// length breaks the contract (flagged; its rows are written as zeros).
struct SeqWork {
    int S, nch, Lb, q0;
};

// From the raw values S_raw = context_lens[b], q0 = cu_q[b], q1 = cu_q[b + 1].
template <int RB, bool kVar>
__device__ __forceinline__ SeqWork seq_work_raw(const DecodeParams& p, int S_raw, int q0, int q1,
                                                bool report) {
    SeqWork w;
    w.Lb = p.L;
    w.q0 = 0;
    if constexpr (kVar) {
        w.q0 = q0;
        w.Lb = q1 - w.q0;
        const bool broken =
            w.q0 < 0 || w.Lb < 0 || q1 > p.total_q || (!p.route_mixed && w.Lb > p.L);
        if (broken || w.Lb == 0 || w.Lb > p.L) {
            if (broken && report) atomicOr(p.flag, PA_FLAG_BAD_CONTEXT);
            w.S = 0;
            w.nch = 0;
            return w;
        }
    }
    w.nch = kVar ? (p.G * w.Lb + RB - 1) / RB : p.nchunk;
    const int S = S_raw;
    const bool bad = S < 1 || static_cast<long long>(S) > p.max_S || (p.causal && S < w.Lb);
    if (bad && report) atomicOr(p.flag, PA_FLAG_BAD_CONTEXT);
    w.S = bad ? 0 : S;
    return w;
}

template <int RB, bool kVar>
__device__ __forceinline__ SeqWork seq_work(const DecodeParams& p, int b, bool report) {
    const int q0 = kVar ? __ldg(p.cu_q + b) : 0;
    const int q1 = kVar ? __ldg(p.cu_q + b + 1) : 0;
    return seq_work_raw<RB, kVar>(p, __ldg(p.ctx + b), q0, q1, report);
}

// Row index (in units of D elements) of row rr = g * Lb + l of the (b, kv
// head) block in the query / output layout.
template <bool kVar>
__device__ __forceinline__ long long out_row(const DecodeParams& p, int b, int kvh, int Lb, int q0,
                                             int rr) {
    if constexpr (kVar) {
        const int g = rr / Lb, l = rr - g * Lb;
        return static_cast<long long>(q0 + l) * p.H_q + static_cast<long long>(kvh) * p.G + g;
    }
    return (static_cast<long long>(b) * p.H_q + static_cast<long long>(kvh) * p.G) * p.L + rr;
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



// The producer's position in the flattened work list, advanced tile by tile
// without divisions.  Page ids of the current sequence are held in two
// 32-entry register windows (lane i: pages wb + i and wb + 32 + i), the
// second one loaded while the first is in use, and the first window of the
// next sequence is requested as soon as a sequence is entered, so block-table
// lookups stay off the path from a freed stage to its next copy.
template <class C>
struct Walker {
    int chunk, next, cu0, cu1;  // current chunk, the one claimed after it, its units
    int u;                      // first unit of the next tile
    int b, bpref, S, ng;        // sequence, its first unit, length, units per segment
    int nch, Lb, q0;            // its row chunks, query positions, first token
    int sib, g;                 // segment within the sequence, unit within the segment
    int kvh, chunk_r;           // kv head and row chunk of the segment
    int key0, lp, slot;         // first key of the next tile, its page and slot
    int S_ahead;                // context length of sequence b + 1 (requested early)
    int qn, qn_ahead;           // cu_q[b + 1], cu_q[b + 2] (ragged batch, requested early)
    int wb, win0, win1;         // page-id windows of sequence b
    int nb_win;                 // pages 0..31 of sequence b + 1
};

// Block-table entry (b, lp), or -1 past the row.  The page windows may fetch
// entries past a sequence's last page; those values are never used.
__device__ __forceinline__ int bt_entry(const DecodeParams& p, int b, int lp) {
    return lp < p.max_npg ? __ldg(p.bt + static_cast<long long>(b) * p.max_npg + lp) : -1;
}

template <class C>
__device__ __forceinline__ void load_windows(const DecodeParams& p, int lane, Walker<C>& w) {
    w.win0 = bt_entry(p, w.b, w.wb + lane);
    w.win1 = bt_entry(p, w.b, w.wb + 32 + lane);
}

// Position the walker at unit w.u (a chunk start); sequences at or after w.b.
// Enters sequence w.b: its length, units per segment and row chunks.
template <class C>
__device__ __forceinline__ void walker_set(const DecodeParams& p, Walker<C>& w, const SeqWork& sw) {
    w.S = sw.S;
    w.nch = sw.nch;
    w.Lb = sw.Lb;
    w.q0 = sw.q0;
    w.ng = sw.nch > 0 ? (sw.S + C::GRAN - 1) / C::GRAN : 0;
}

// Requests the raw metadata of sequence w.b + 1 for the next walker_set.
template <class C, bool kVar>
__device__ __forceinline__ void walker_look_ahead(const DecodeParams& p, Walker<C>& w) {
    w.S_ahead = w.b + 1 < p.B ? __ldg(p.ctx + w.b + 1) : 0;
    if constexpr (kVar) w.qn_ahead = w.b + 1 < p.B ? __ldg(p.cu_q + w.b + 2) : 0;
}

template <class C, bool kVar>
__device__ void walker_seek(const DecodeParams& p, int lane, Walker<C>& w) {
    const int segs_plain = p.H_kv * p.nchunk;
    while (w.u >= w.bpref + (kVar ? p.H_kv * w.nch : segs_plain) * w.ng) {
        w.bpref += (kVar ? p.H_kv * w.nch : segs_plain) * w.ng;
        ++w.b;
        walker_set<C>(p, w, seq_work<C::RB, kVar>(p, w.b, false));
    }
    if constexpr (kVar) w.qn = __ldg(p.cu_q + w.b + 1);
    walker_look_ahead<C, kVar>(p, w);
    const int loc = w.u - w.bpref;
    w.sib = loc / w.ng;
    w.g = loc - w.sib * w.ng;
    const int nch = kVar ? w.nch : p.nchunk;
    w.kvh = w.sib / nch;
    w.chunk_r = w.sib - w.kvh * nch;
    w.key0 = w.g * C::GRAN;
    w.lp = w.key0 / p.ps;
    w.slot = w.key0 - w.lp * p.ps;
    w.wb = w.lp;
    load_windows(p, lane, w);
    w.nb_win = w.b + 1 < p.B ? bt_entry(p, w.b + 1, lane) : -1;
}

// Page id of page index `lpi` of sequence w.b (all lanes call it together;
// lanes whose piece is not `active` get -1 without touching memory).
template <class C>
__device__ __forceinline__ int page_id(const DecodeParams& p, const Walker<C>& w, int lpi,
                                       bool active) {
    const int rel = lpi - w.wb;
    const int a = __shfl_sync(0xffffffffu, w.win0, rel & 31);
    const int c = __shfl_sync(0xffffffffu, w.win1, rel & 31);
    if (!active) return -1;
    if (rel >= 0 && rel < 32) return a;
    if (rel >= 32 && rel < 64) return c;
    return bt_entry(p, w.b, lpi);  // outside both windows (tiny pages): direct
}

// Row owned by in-group lane li after transpose_reduce<RB, P>: each
// splitting step keeps the upper half of the remaining rows in lanes whose
// step bit is set.
template <int RB, int P>
__device__ __forceinline__ int row_of_lane(int li) {
    int rho = 0, rc = RB;
#pragma unroll
    for (int step = P / 2; step >= 1; step >>= 1) {
        if (rc > 1) {
            if (li & step) rho += rc / 2;
            rc /= 2;
        }
    }
    return rho;
}

// Sums v[r] over the P lanes of a group for every row r and leaves the total
// of row row_of_lane(li) in this lane.  While more than one row is left, a
// step exchanges half of them (the half the partner keeps) instead of all,
// so RB rows over P lanes cost RB - 1 + log2(P / RB) shuffles, not
// RB * log2(P).
template <int RB, int P>
__device__ __forceinline__ float transpose_reduce(float (&v)[RB], int li) {
    static_assert(RB <= P, "one lane per row at least");
    int rc = RB;
#pragma unroll
    for (int step = P / 2; step >= 1; step >>= 1) {
        if (rc > 1) {
            const bool up = (li & step) != 0;
            const int half = rc / 2;
#pragma unroll
            for (int i = 0; i < RB / 2; ++i) {
                if (i < half) {
                    const float send = up ? v[i] : v[i + half];
                    const float keep = up ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, step);
                }
            }
            rc = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], step);
        }
    }
    return v[0];
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

// The end of a segment piece, once this warp has written its record (o[D],
// m, l per row) into the merge buffer: after every consumer warp has, warp r
// merges row r (and r + NCW, ...) over the warps' records, four dims per
// lane, and writes the normalised output (a piece that is the whole segment)
// or an fp32 partial for the combine kernel.  Returns false if a wait timed
// out.
template <class C, bool kVar>
__device__ __forceinline__ bool merge_piece(const DecodeParams& p, const StageHdr& h, int hLb,
                                            const float* merge, int warp, int lane,
                                            uint32_t mfull, uint32_t mdone, int nend) {
    using T = typename C::Elem;
    if (lane == 0) mbar_arrive(mfull);
    if (!__all_sync(0xffffffffu, mbar_wait(mfull, nend & 1))) return false;
    const int rows_valid = min(C::RB, p.G * hLb - h.chunk * C::RB);
    const long long slot = h.slot;
    T* const out = static_cast<T*>(p.out);
    for (int r = warp; r < rows_valid; r += C::NCW) {
        float M = neg_inf();
#pragma unroll
        for (int wq = 0; wq < C::NCW; ++wq) M = fmaxf(M, merge[(wq * C::RB + r) * C::MSTRIDE + kD]);
        float den = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != neg_inf()) {
#pragma unroll
            for (int wq = 0; wq < C::NCW; ++wq) {
                const float* rec = merge + (wq * C::RB + r) * C::MSTRIDE;
                const float a = fast_exp2(rec[kD] - M);
                den += a * rec[kD + 1];
                const float4 ov = *reinterpret_cast<const float4*>(rec + 4 * lane);
                acc.x += a * ov.x;
                acc.y += a * ov.y;
                acc.z += a * ov.z;
                acc.w += a * ov.w;
            }
        }
        if (h.flags & kFinal) {
            const float inv = den > 0.f ? 1.f / den : 0.f;
            store4<T>(out, out_row<kVar>(p, h.b, h.kvh, hLb, h.q0, h.chunk * C::RB + r) * kD + 4 * lane,
                      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
        } else {
            *reinterpret_cast<float4*>(p.part_o + (slot * C::RB + r) * kD + 4 * lane) = acc;
            if (lane == 0) p.part_ml[slot * C::RB + r] = make_float2(M, den);
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(mdone);
    return __all_sync(0xffffffffu, mbar_wait(mdone, nend & 1));
}

// F: 0 plain, 1 with an explicit mask, 2 a ragged batch.  Separate
// instantiations, so the plain kernel carries none of the others' code.
template <class C, int F>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_kt,
                        const __grid_constant__ CUtensorMap tm_vt, const DecodeParams p) {
    using T = typename C::Elem;
    constexpr bool kMask = F == 1, kVar = F == 2;
    static_assert(!(C::MMA && kMask), "the tensor-core consumers take no explicit mask");
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // the tensor-core layout's swizzled halves need a 1024-byte aligned base
    uint8_t* const smem =
        C::MMA ? smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u) : smem_raw;
    uint8_t* const stage0 = smem;
    float* const merge = reinterpret_cast<float*>(smem + C::NST * C::STAGE);
    float* const pbuf_all = reinterpret_cast<float*>(smem + C::NST * C::STAGE + C::MERGE);
    uint64_t* const bars =
        reinterpret_cast<uint64_t*>(smem + C::NST * C::STAGE + C::MERGE + C::PBUF);
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
    // units of sequence b: its segments (kv heads x row chunks) x key units
    const int segs_per_b = p.H_kv * p.nchunk;  // (the [B, H_q, L, D] layout)
    auto units_of = [&](int b, bool report) {
        const SeqWork sw = seq_work<C::RB, kVar>(p, b, report);
        return p.H_kv * sw.nch * ((sw.S + C::GRAN - 1) / C::GRAN);
    };
    int mine = 0;
    for (int b = tid; b < p.B; b += C::THREADS) mine += units_of(b, blockIdx.x == 0);
    int total;
    block_incl_scan<C::THREADS>(mine, s_scan, &total);
    const int grid = static_cast<int>(gridDim.x);
    const int cu = max(1, (total + grid * kChunksPerCta - 1) / (grid * kChunksPerCta));
    const int nchunks = (total + cu - 1) / cu;
    const int u0 = static_cast<int>(blockIdx.x) * cu;
    int carry = 0;
    for (int base = 0; base < p.B; base += C::THREADS) {
        const int b = base + tid;
        const int v = b < p.B ? units_of(b, false) : 0;
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
    // Launched beside the tile kernel of a mixed ragged batch (as its
    // programmatic dependent), this grid must not finish before that one:
    // every exit waits for it, so stream order still covers both kernels.
    // (Without a preceding programmatic launch the wait returns at once.)
    if (static_cast<int>(blockIdx.x) >= nchunks) {
        if (tid == 0) finish_chunk_counters(p, grid);
        pdl_wait_primary();
        return;
    }

    if (warp == C::NCW) {
        // =========================== producer warp ===========================
        const uint64_t pol = l2_policy_evict_first();
        const uint8_t* const kp = static_cast<const uint8_t*>(p.kp);
        const uint8_t* const vp = static_cast<const uint8_t*>(p.vp);
        const uint8_t* const qp = static_cast<const uint8_t*>(p.q);
        constexpr int kGranShift = __builtin_ctz(C::GRAN);
        static_assert((C::GRAN & (C::GRAN - 1)) == 0, "unit size must be a power of two");
        Walker<C> w;
        w.chunk = static_cast<int>(blockIdx.x);
        w.next = __shfl_sync(0xffffffffu, lane == 0 ? atomicAdd(p.chunk_counter, 1) : 0, 0) + grid;
        w.cu0 = w.chunk * cu;
        w.cu1 = min(w.cu0 + cu, total);
        w.u = w.cu0;
        w.b = s_start_b;
        w.bpref = s_start_pref;
        walker_set<C>(p, w, seq_work<C::RB, kVar>(p, w.b, false));
        walker_seek<C, kVar>(p, lane, w);
        int issued = 0;
        for (int i = 0;; ++i) {
            // ---- this tile: keys [key0, key0 + nvalid) of segment (b, sib) ----
            const int seg_u0 = w.bpref + w.sib * w.ng, seg_u1 = seg_u0 + w.ng;
            const int piece_u1 = min(w.cu1, seg_u1);
            const int piece_key1 = min(w.S, (piece_u1 - seg_u0) << kGranShift);
            const int nvalid = min(C::TK, piece_key1 - w.key0);
            const int units = (nvalid + C::GRAN - 1) >> kGranShift;
            const bool last_chunk = w.next >= nchunks;
            const bool start = (w.u == w.cu0) || (w.g == 0);
            const bool end = w.u + units >= piece_u1;
            const int flags = (start ? kStart : 0) | (end ? kEnd : 0) |
                              ((seg_u0 >= w.cu0 && seg_u1 <= w.cu1) ? kFinal : 0) |
                              ((end && piece_u1 == w.cu1 && last_chunk) ? kLast : 0);
            // page pieces: piece j covers page lp + j (lane j + 32 k handles it);
            // a tile spans at most TK / ps + 2 pages, one lane each unless ps < 4
            const int row0 = w.chunk_r * C::RB;
            const int nrows = min(C::RB, p.G * (kVar ? w.Lb : p.L) - row0);
            int pid[C::PIECE_ITERS], klo[C::PIECE_ITERS], kn[C::PIECE_ITERS];
            bool any_bad = false;
            uint32_t bytes;
            int box_row = -1;  // tensor-core layout: pool row of this lane's box
            const bool full_tile = nvalid == C::TK;
            const int bh = full_tile ? p.boxr : p.boxr_tail;  // box height of this tile
            if constexpr (C::MMA) {
                // Boxes of bh keys, lane i copying box i (keys key0 + i * bh ...):
                // a full tile in boxes of p.boxr keys (one box when a page holds
                // the whole tile), a segment's last, partial tile in boxes of
                // p.boxr_tail keys.  Box heights divide the page size and every
                // tile start, so no box crosses a page.  The last box may run past
                // the context into unused page slots (< boxr_tail rows); the
                // consumers mask those keys and zero those V rows.
                const int nb = (nvalid + bh - 1) / bh;
                const bool act = lane < nb;
                const int off = w.slot + lane * bh;  // from the start of page w.lp
                const int lpo = off / p.ps;
                const int id = page_id<C>(p, w, w.lp + lpo, act);
                if (act) {
                    if (id >= 0 && id < p.num_pages)
                        box_row = (id * p.H_kv + w.kvh) * p.ps + (off - lpo * p.ps);
                    else
                        any_bad = true;
                }
                const int good = __popc(__ballot_sync(0xffffffffu, box_row >= 0));
                bytes = static_cast<uint32_t>(good) * 4u * 128u * static_cast<uint32_t>(bh) +
                        (start ? static_cast<uint32_t>(nrows) * C::ROW : 0u);
                if (any_bad) atomicOr(p.flag, PA_FLAG_BAD_PAGE);
            }
            if constexpr (!C::MMA) {
#pragma unroll
            for (int k = 0; k < C::PIECE_ITERS; ++k) {
                pid[k] = -1;
                klo[k] = 0;
                kn[k] = 0;
                if (k > 0 && p.ps >= 4) continue;  // uniform: whole warp skips
                const int j = lane + 32 * k;
                const int lo = j == 0 ? w.key0 : w.key0 - w.slot + j * p.ps;
                const int hi = min(w.key0 + nvalid, w.key0 - w.slot + (j + 1) * p.ps);
                const bool active = lo < hi;
                const int id = page_id<C>(p, w, w.lp + j, active);
                klo[k] = lo;
                kn[k] = hi - lo;
                if (active) {
                    if (id >= 0 && id < p.num_pages) {
                        pid[k] = id;
                    } else {
                        any_bad = true;
                    }
                }
            }
            }
            // bytes the stage will receive: all K/V rows of the tile (plus the
            // query rows at a piece start), minus pieces with a bad page id
            if constexpr (!C::MMA) bytes = 2u * static_cast<uint32_t>(nvalid) * C::ROW +
                                           (start ? static_cast<uint32_t>(nrows) * C::ROW : 0u);
            if (!C::MMA && __ballot_sync(0xffffffffu, any_bad)) {
                uint32_t miss = 0;
#pragma unroll
                for (int k = 0; k < C::PIECE_ITERS; ++k)
                    if (kn[k] > 0 && pid[k] < 0) miss += 2u * static_cast<uint32_t>(kn[k]) * C::ROW;
                bytes -= static_cast<uint32_t>(warp_sum(static_cast<int>(miss)));
                if (any_bad) atomicOr(p.flag, PA_FLAG_BAD_PAGE);
            }

            // the explicit mask's rows of this tile go to L2 now, NST stages
            // before the consumers read them: [key0, key0 + nvalid) widened to
            // whole 16-byte words, inside the row (mask_S % 4 == 0, >= S)
            if (kMask && p.mask && lane < nrows && nvalid > 0) {
                const int rg = row0 + lane, gq = rg / w.Lb, lq = rg - gq * w.Lb;
                const int lo = w.key0 & ~3, hi = (w.key0 + nvalid + 3) & ~3;
                bulk_prefetch_l2(p.mask + ((static_cast<long long>(w.b) * p.H_q +
                                            w.kvh * p.G + gq) * w.Lb + lq) * p.mask_S + lo,
                                 static_cast<uint32_t>(hi - lo) * 4u);
            }

            const int stage = i % C::NST;
            const uint32_t fb = full0 + 8 * stage, eb = empty0 + 8 * stage;
            if (i >= C::NST &&
                !__all_sync(0xffffffffu, mbar_wait(eb, ((i / C::NST) - 1) & 1))) {
                if (lane == 0) atomicOr(p.flag, PA_FLAG_TIMEOUT);
                s_abort = 1;
                break;
            }
            if ((i & 7) == 0 && __any_sync(0xffffffffu, s_abort != 0)) break;
            uint8_t* const st = stage0 + stage * C::STAGE;
            if (lane == 0) {
                const int seg_id = (w.b * p.H_kv + w.kvh) * p.nchunk + w.chunk_r;
                uint4* h = reinterpret_cast<uint4*>(st + C::OFF_HDR);
                h[0] = make_uint4(seg_id, w.b, w.kvh, w.chunk_r);
                h[1] = make_uint4(w.key0, nvalid, w.S, flags);
                h[2] = make_uint4(seg_id + w.chunk, w.Lb, w.q0, 0);
                mbar_arrive_expect_tx(fb, bytes);
            }
            __syncwarp();
            const uint32_t kdst = smem_u32(st) + C::OFF_K;
            if constexpr (C::MMA) {
                if (box_row >= 0) {
                    const uint32_t kd = kdst + static_cast<uint32_t>(lane * bh) * 128u;
                    const uint32_t vd = smem_u32(st) + C::OFF_V +
                                        static_cast<uint32_t>(lane * bh) * 128u;
                    const CUtensorMap* mk = full_tile ? &tm_k : &tm_kt;
                    const CUtensorMap* mv = full_tile ? &tm_v : &tm_vt;
                    tc::tma_load_2d(kd, mk, 0, box_row, fb, pol);
                    tc::tma_load_2d(kd + C::KHALF, mk, 64, box_row, fb, pol);
                    tc::tma_load_2d(vd, mv, 0, box_row, fb, pol);
                    tc::tma_load_2d(vd + C::KHALF, mv, 64, box_row, fb, pol);
                }
            }
            if constexpr (!C::MMA) {
#pragma unroll
            for (int k = 0; k < C::PIECE_ITERS; ++k) {
                if (pid[k] < 0) continue;
                const int j = lane + 32 * k;
                const long long row = (static_cast<long long>(pid[k]) * p.H_kv + w.kvh) * p.ps +
                                      (j == 0 ? w.slot : 0);
                const uint32_t nb = static_cast<uint32_t>(kn[k]) * C::ROW;
                const uint32_t off = static_cast<uint32_t>(klo[k] - w.key0) * C::ROW;
                bulk_g2s(kdst + off, kp + row * C::ROW, nb, fb, pol);
                bulk_g2s(kdst + C::KBYTES + off, vp + row * C::ROW, nb, fb, pol);
            }
            }
            if (start) {
                if constexpr (!kVar) {  // the segment's rows are contiguous
                    if (lane == 0)
                        bulk_g2s(smem_u32(st) + C::OFF_Q,
                                 qp + out_row<false>(p, w.b, w.kvh, p.L, 0, row0) * C::ROW,
                                 static_cast<uint32_t>(nrows) * C::ROW, fb, pol);
                } else if (lane < nrows) {  // one token-major row per lane
                    bulk_g2s(smem_u32(st) + C::OFF_Q + lane * C::ROW,
                             qp + out_row<true>(p, w.b, w.kvh, w.Lb, w.q0, row0 + lane) * C::ROW,
                             C::ROW, fb, pol);
                }
            }
            issued = i + 1;

            // ---- advance to the next tile ----
            w.u += units;
            if (w.u >= w.cu1) {
                if (last_chunk) break;
                w.chunk = w.next;
                w.next = __shfl_sync(0xffffffffu, lane == 0 ? atomicAdd(p.chunk_counter, 1) : 0,
                                     0) + grid;
                w.cu0 = w.chunk * cu;
                w.cu1 = min(w.cu0 + cu, total);
                w.u = w.cu0;
                walker_seek<C, kVar>(p, lane, w);
            } else if (w.u >= seg_u1) {
                // next segment: same sequence (next row chunk / kv head) or the next one
                w.g = 0;
                w.key0 = 0;
                w.lp = 0;
                w.slot = 0;
                ++w.sib;
                if (++w.chunk_r == (kVar ? w.nch : p.nchunk)) {
                    w.chunk_r = 0;
                    ++w.kvh;
                }
                if (w.sib == (kVar ? p.H_kv * w.nch : segs_per_b)) {
                    // next sequence with work (sequences with no keys are skipped)
                    do {
                        w.bpref += (kVar ? p.H_kv * w.nch : segs_per_b) * w.ng;
                        ++w.b;
                        walker_set<C>(p, w, seq_work_raw<C::RB, kVar>(p, w.S_ahead, w.qn,
                                                                       w.qn_ahead, false));
                        w.qn = w.qn_ahead;
                        walker_look_ahead<C, kVar>(p, w);
                        w.win0 = w.nb_win;
                        w.nb_win = w.b + 1 < p.B ? bt_entry(p, w.b + 1, lane) : -1;
                    } while (w.ng == 0);
                    w.sib = 0;
                    w.kvh = 0;
                    w.chunk_r = 0;
                    w.wb = 0;
                    w.win1 = bt_entry(p, w.b, 32 + lane);
                } else if (w.wb != 0) {
                    w.wb = 0;
                    load_windows(p, lane, w);
                }
            } else {
                // a full tile (nvalid == TK) inside the segment
                w.g += units;
                w.key0 += nvalid;
                w.lp += p.tk_pages;
                w.slot += p.tk_slots;
                if (w.slot >= p.ps) {
                    w.slot -= p.ps;
                    ++w.lp;
                }
                if (w.lp >= w.wb + 32) {  // slide the windows by 32 pages
                    w.wb += 32;
                    w.win0 = w.win1;
                    w.win1 = bt_entry(p, w.b, w.wb + 32 + lane);
                }
            }
        }
        // Never leave with copies in flight into this CTA's shared memory.
        for (int k = max(0, issued - C::NST); k < issued; ++k)
            if (!mbar_wait(full0 + 8 * (k % C::NST), (k / C::NST) & 1))
                atomicOr(p.flag, PA_FLAG_TIMEOUT);
        if (lane == 0) finish_chunk_counters(p, grid);
        pdl_wait_primary();
        return;
    }

    // ============================ consumer warps ============================
    if constexpr (C::MMA) {
        // Tensor-core consumers.  Warp w takes keys kw0 .. kw0 + 15 of each
        // stage and computes S^T = K Q^T (m16n8k16: 16 keys x 8 query rows,
        // rows past RB are zero) and O^T += V^T P^T (16 dims x 8 rows per
        // instruction, 8 of them for D = 128).  Lane 4g + t holds the scores
        // of keys g and g + 8 for rows 2t and 2t + 1, and O^T of dims
        // 16 i + g and 16 i + g + 8 for the same two rows.  P is rounded to
        // bf16 for the product, and the row sums add the rounded weights.
        const int g = lane >> 2, t4 = lane & 3;
        const int kw0 = warp * C::KPW;
        uint32_t qf[8][2];   // Q^T B fragments of the 8 k-steps (16 dims each)
        float oacc[8][4];    // O^T accumulators
        float m_r[2] = {neg_inf(), neg_inf()}, l_r[2] = {0.f, 0.f};
        int lpos[2] = {0, 0};  // query positions of rows 2t, 2t + 1
        int lmin = 0;
        int nend = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            qf[i][0] = qf[i][1] = 0u;
            oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
        }
        for (int i = 0;; ++i) {
            const int stage = i % C::NST;
            if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * stage, (i / C::NST) & 1))) {
                if (lane == 0) atomicOr(p.flag, PA_FLAG_TIMEOUT);
                s_abort = 1;
                break;
            }
            if ((i & 7) == 0 && __any_sync(0xffffffffu, s_abort != 0)) break;
            uint8_t* const st = stage0 + stage * C::STAGE;
            const StageHdr h = *reinterpret_cast<const StageHdr*>(st + C::OFF_HDR);
            const int hLb = kVar ? h.Lb : p.L;

            if (h.flags & kStart) {
                const int rows = p.G * hLb - h.chunk * C::RB;
                const bool qrow_ok = g < C::RB && g < rows;
                const uint8_t* const qrow = st + C::OFF_Q + g * C::ROW;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    qf[ks][0] = qrow_ok ? *reinterpret_cast<const uint32_t*>(qrow + (ks * 16 + 2 * t4) * 2) : 0u;
                    qf[ks][1] = qrow_ok ? *reinterpret_cast<const uint32_t*>(qrow + (ks * 16 + 8 + 2 * t4) * 2) : 0u;
                }
#pragma unroll
                for (int mt = 0; mt < 8; ++mt)
                    oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
                m_r[0] = m_r[1] = neg_inf();
                l_r[0] = l_r[1] = 0.f;
                lmin = INT_MAX;
#pragma unroll
                for (int r = 0; r < C::RB; ++r)
                    lmin = min(lmin, r < rows ? (h.chunk * C::RB + r) % hLb : hLb - 1);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = 2 * t4 + e;
                    lpos[e] = (r < C::RB && r < rows) ? (h.chunk * C::RB + r) % hLb : hLb - 1;
                }
            }

            if (h.nvalid > kw0) {
                // The last box of a context may bring unused page slots past it
                // (any contents): their scores are masked below, and their V
                // rows are zeroed here, since a weight of 0 times NaN is NaN.
                {
                    const int zlo = h.nvalid;
                    const int zhi =
                        min(kw0 + C::KPW, (h.nvalid + p.boxr_tail - 1) / p.boxr_tail * p.boxr_tail);
                    if (zlo < zhi) {  // uniform over the warp
                        for (int idx = lane; idx < (zhi - zlo) * 16; idx += 32) {
                            const int r = zlo + (idx >> 4), c = idx & 15;
                            *reinterpret_cast<uint4*>(st + C::OFF_V + (c >> 3) * C::KHALF + r * 128 +
                                                      (((c & 7) ^ (r & 7)) << 4)) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();  // before the stage's next TMA fill
                        __syncwarp();
                    }
                }
                // S^T = K Q^T over the 8 k-steps of 16 dims
                float sacc[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    const int r = kw0 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const uint32_t rb = smem_u32(st) + C::OFF_K + r * 128;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int c = ks * 2 + (lane >> 4);
                        uint32_t a[4];
                        ldmatrix_x4(a, rb + (c >> 3) * C::KHALF + (((c & 7) ^ (r & 7)) << 4));
                        mma_16816(sacc, a, qf[ks][0], qf[ks][1]);
                    }
                }
                // log2-unit scores; keys past the context or a row's causal
                // frontier get -inf
                const float c = p.scale_log2;
                float x[4] = {sacc[0] * c, sacc[1] * c, sacc[2] * c, sacc[3] * c};
                const int last_key = h.key0 + kw0 + C::KPW - 1;
                if (h.nvalid < kw0 + C::KPW || (p.causal && last_key > lmin + h.S - hLb)) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int kl = kw0 + g + (e >> 1) * 8;
                        const bool vis = kl < h.nvalid &&
                                         (!p.causal || h.key0 + kl <= lpos[e & 1] + h.S - hLb);
                        if (!vis) x[e] = neg_inf();
                    }
                }
                float mt0 = fmaxf(x[0], x[2]), mt1 = fmaxf(x[1], x[3]);
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, o));
                    mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, o));
                }
                const bool gr0 = mt0 > m_r[0] + kLazyRescaleLog2;
                const bool gr1 = mt1 > m_r[1] + kLazyRescaleLog2;
                if (__any_sync(0xffffffffu, gr0 || gr1)) {
                    // rows whose max grew by more than 2^8 move it and rescale
                    const float a0 = gr0 ? fast_exp2(m_r[0] - mt0) : 1.f;  // 2^-inf = 0
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
                // P^T as bf16: (key g, rows 2t, 2t+1) and (key g + 8, ...), each
                // an 8 x 8 block in C layout, transposed into B fragments
                const uint32_t X0 = pack_bf16x2(fast_exp2(x[0] - mu0), fast_exp2(x[1] - mu1));
                const uint32_t X1 = pack_bf16x2(fast_exp2(x[2] - mu0), fast_exp2(x[3] - mu1));
                {
                    const float2 f0 = bf16x2_to_float2(X0), f1 = bf16x2_to_float2(X1);
                    l_r[0] += f0.x + f1.x;
                    l_r[1] += f0.y + f1.y;
                }
                const uint32_t pb0 = movmatrix_trans(X0), pb1 = movmatrix_trans(X1);
                // O^T += V^T P^T, 16 dims per instruction
                {
                    const int r = kw0 + (lane & 7) + (lane >> 4) * 8;
                    const uint32_t rb = smem_u32(st) + C::OFF_V + r * 128;
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        const int cc = mt * 2 + ((lane >> 3) & 1);
                        uint32_t a[4];
                        ldmatrix_x4_trans(a, rb + (cc >> 3) * C::KHALF + (((cc & 7) ^ (r & 7)) << 4));
                        mma_16816(oacc[mt], a, pb0, pb1);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * stage);

            if (h.flags & kEnd) {
                // this warp's record: o[D], m, l of every row of the piece
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], o);
                    l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], o);
                }
                float* const mw = merge + warp * C::RB * C::MSTRIDE;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = 2 * t4 + e;
                    if (r < C::RB) {
#pragma unroll
                        for (int mt = 0; mt < 8; ++mt) {
                            mw[r * C::MSTRIDE + 16 * mt + g] = oacc[mt][e];
                            mw[r * C::MSTRIDE + 16 * mt + g + 8] = oacc[mt][2 + e];
                        }
                        if (g == 0) {
                            mw[r * C::MSTRIDE + kD] = m_r[e];
                            mw[r * C::MSTRIDE + kD + 1] = l_r[e];
                        }
                    }
                }
                __syncwarp();
                if (!merge_piece<C, kVar>(p, h, hLb, merge, warp, lane, mfull, mdone, nend)) {
                    if (lane == 0) atomicOr(p.flag, PA_FLAG_TIMEOUT);
                    s_abort = 1;
                    break;
                }
                ++nend;
            }
            if (h.flags & kLast) break;
        }
    } else {
    // Q.K^T: P lanes share one key (each holds DPL dims of every query row in
    // registers); after the transposed reduction each lane owns the score of
    // row `rho` of its group's key, so exp2 and the running sum run once per
    // (key, row).  P.V: lane i owns output dims 4i..4i+3 of every row and
    // walks the warp's keys, reading the weights from a per-warp buffer, so
    // the accumulator is 4 floats per row and never needs a cross-lane sum.
    const int grp = lane / C::P, li = lane % C::P;
    const int rho = row_of_lane<C::RB, C::P>(li);
    constexpr int SPREAD = C::P / C::RB;  // lanes of a group that own the same row
    float* const pbuf = pbuf_all + warp * C::KPW * C::RB;
    float2 q2[C::RB][C::DPL / 2];
    float2 o4[C::RB][2];                      // dims 4*lane .. 4*lane+3 of each row
    float m_mine = neg_inf(), l_mine = 0.f;  // running max / sum of row rho
    int lrow_mine = 0;
    int lmin = 0;
    int nend = 0;
#pragma unroll
    for (int r = 0; r < C::RB; ++r) {
#pragma unroll
        for (int e = 0; e < C::DPL / 2; ++e) q2[r][e] = make_float2(0.f, 0.f);
        o4[r][0] = o4[r][1] = make_float2(0.f, 0.f);
    }

    for (int i = 0;; ++i) {
        const int stage = i % C::NST;
        if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * stage, (i / C::NST) & 1))) {
            if (lane == 0) atomicOr(p.flag, PA_FLAG_TIMEOUT);
            s_abort = 1;
            break;
        }
        if ((i & 7) == 0 && __any_sync(0xffffffffu, s_abort != 0)) break;
        const uint8_t* const st = stage0 + stage * C::STAGE;
        const StageHdr h = *reinterpret_cast<const StageHdr*>(st + C::OFF_HDR);
        const int hLb = kVar ? h.Lb : p.L;  // the segment's query positions

        if (h.flags & kStart) {
            const int rows = p.G * hLb - h.chunk * C::RB;
            lmin = INT_MAX;
#pragma unroll
            for (int r = 0; r < C::RB; ++r) {
                load_row<C>(st + C::OFF_Q + r * C::ROW, li, q2[r]);
#pragma unroll
                for (int e = 0; e < C::DPL / 2; ++e) {
                    q2[r][e].x *= p.scale_log2;
                    q2[r][e].y *= p.scale_log2;
                }
                o4[r][0] = o4[r][1] = make_float2(0.f, 0.f);
                lmin = min(lmin, r < rows ? (h.chunk * C::RB + r) % hLb : hLb - 1);
            }
            lrow_mine = rho < rows ? (h.chunk * C::RB + rho) % hLb : hLb - 1;
            m_mine = neg_inf();
            l_mine = 0.f;
        }

        const int kw0 = warp * C::KPW;
        if (h.nvalid > kw0) {
            const uint8_t* const Ks = st + C::OFF_K;
            const uint8_t* const Vs = st + C::OFF_V;
            // An explicit additive mask joins the score of (key, row) in log2
            // units before the max; its loads go out before the dot products.
            float mv[C::IT];
            // (p.mask is never null in this instance; with the run-time test the
            // compiler emits code 9% faster than with kMask alone, measured)
            if (kMask && p.mask) {
                const int rg = h.chunk * C::RB + rho;  // row of the (b, kv head) block
                const bool rok = rg < p.G * hLb;
                const int gq = rg / hLb, lq = rg - gq * hLb;
                const float* mrow = p.mask + ((static_cast<long long>(h.b) * p.H_q +
                                               h.kvh * p.G + gq) * hLb + lq) * p.mask_S +
                                    h.key0;
#pragma unroll
                for (int it = 0; it < C::IT; ++it) {
                    const int kl = kw0 + it * C::KPI + grp;
                    mv[it] = rok && kl < h.nvalid ? __ldcs(mrow + kl) : 0.f;
                }
            }
            float sc[C::IT];  // score of (this group's key of iteration it, row rho)
#pragma unroll
            for (int it = 0; it < C::IT; ++it) {
                const int kl = kw0 + it * C::KPI + grp;
                float2 k2[C::DPL / 2];
                load_row<C>(Ks + kl * C::ROW, li, k2);
                float d[C::RB];
#pragma unroll
                for (int r = 0; r < C::RB; ++r) {
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < C::DPL / 2; ++e) acc = __ffma2_rn(q2[r][e], k2[e], acc);
                    d[r] = acc.x + acc.y;
                }
                sc[it] = transpose_reduce<C::RB, C::P>(d, li);
            }
            if (kMask && p.mask) {
#pragma unroll
                for (int it = 0; it < C::IT; ++it) sc[it] += mv[it] * 1.4426950408889634f;
            }
            // Score mask (the separate "second mask" of a masked load): keys
            // past the context or past a row's causal frontier get -inf.
            const int last_key = h.key0 + kw0 + C::KPW - 1;
            const bool tail = h.nvalid < kw0 + C::KPW;
            if (tail || (p.causal && last_key > lmin + h.S - hLb)) {
#pragma unroll
                for (int it = 0; it < C::IT; ++it) {
                    const int kl = kw0 + it * C::KPI + grp;
                    const int kg = h.key0 + kl;
                    const bool vis =
                        kl < h.nvalid && (!p.causal || kg <= lrow_mine + h.S - hLb);
                    if (!vis) sc[it] = neg_inf();
                }
            }
            float mt = sc[0];
#pragma unroll
            for (int it = 1; it < C::IT; ++it) mt = fmaxf(mt, sc[it]);
#pragma unroll
            for (int o = C::P; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
            const bool grow = mt > m_mine + kLazyRescaleLog2;
            if (__any_sync(0xffffffffu, grow)) {
                // rows whose max grew by more than 2^8 move it and rescale
                const float a = grow ? fast_exp2(m_mine - mt) : 1.f;  // 2^-inf = 0 at the start
                if (grow) m_mine = mt;
                l_mine *= a;
#pragma unroll
                for (int r = 0; r < C::RB; ++r) {
                    const float ar = __shfl_sync(0xffffffffu, a, r * SPREAD);
                    o4[r][0].x *= ar;
                    o4[r][0].y *= ar;
                    o4[r][1].x *= ar;
                    o4[r][1].y *= ar;
                }
            }
            const float mu = (m_mine == neg_inf()) ? 0.f : m_mine;
#pragma unroll
            for (int it = 0; it < C::IT; ++it) {
                const float pm = fast_exp2(sc[it] - mu);
                l_mine += pm;
                if (li % SPREAD == 0) pbuf[(it * C::KPI + grp) * C::RB + rho] = pm;
            }
            __syncwarp();
#pragma unroll 4
            for (int k = 0; k < C::KPW; ++k) {
                const int kl = kw0 + k;  // this warp's keys in order
                float pw[C::RB];
#pragma unroll
                for (int r = 0; r < C::RB; ++r) pw[r] = pbuf[k * C::RB + r];
                float2 v0, v1;
                if constexpr (sizeof(T) == 2) {
                    const uint2 u = *reinterpret_cast<const uint2*>(Vs + kl * C::ROW + lane * 8);
                    v0 = bf16x2_to_float2(u.x);
                    v1 = bf16x2_to_float2(u.y);
                } else {
                    const float4 f = *reinterpret_cast<const float4*>(Vs + kl * C::ROW + lane * 16);
                    v0 = make_float2(f.x, f.y);
                    v1 = make_float2(f.z, f.w);
                }
#pragma unroll
                for (int r = 0; r < C::RB; ++r) {
                    const float2 pp2 = make_float2(pw[r], pw[r]);
                    o4[r][0] = __ffma2_rn(pp2, v0, o4[r][0]);
                    o4[r][1] = __ffma2_rn(pp2, v1, o4[r][1]);
                }
            }
            __syncwarp();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);

        if (h.flags & kEnd) {
            // this warp's record: its dims of every row, and (m, l) per row
#pragma unroll
            for (int o = C::P; o < 32; o <<= 1) l_mine += __shfl_xor_sync(0xffffffffu, l_mine, o);
            float* const mw = merge + warp * C::RB * C::MSTRIDE;
#pragma unroll
            for (int r = 0; r < C::RB; ++r)
                *reinterpret_cast<float4*>(mw + r * C::MSTRIDE + 4 * lane) =
                    make_float4(o4[r][0].x, o4[r][0].y, o4[r][1].x, o4[r][1].y);
            if (lane < C::P && li % SPREAD == 0) {
                mw[rho * C::MSTRIDE + kD] = m_mine;
                mw[rho * C::MSTRIDE + kD + 1] = l_mine;
            }
            __syncwarp();
            if (!merge_piece<C, kVar>(p, h, hLb, merge, warp, lane, mfull, mdone, nend)) {
                if (lane == 0) atomicOr(p.flag, PA_FLAG_TIMEOUT);
                s_abort = 1;
                break;
            }
            ++nend;
        }
        if (h.flags & kLast) break;
    }
    }
    pdl_wait_primary();
}

// Merges the pieces of every segment that was split across CTAs (one CTA per
// segment, one warp per row, four dims per lane; the pieces' (m, l) are read
// by the lanes in parallel), and writes zeros for sequences whose context
// length broke the contract.
template <class C, bool kVar>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p) {
    using T = typename C::Elem;
    pdl_wait_primary();
    // segment ids number (b, kv head, row chunk) with p.nchunk chunks per kv
    // head; sequence b has sw.nch <= p.nchunk of them
    const int seg = blockIdx.x;
    const int b = seg / (p.H_kv * p.nchunk), kc = seg - b * (p.H_kv * p.nchunk);
    const int kvh = kc / p.nchunk, chunk = kc - kvh * p.nchunk;
    const SeqWork sw = seq_work<C::RB, kVar>(p, b, false);
    if (chunk >= sw.nch) return;  // not this launch's rows
    const int ng = (sw.S + C::GRAN - 1) / C::GRAN;
    const int rows_valid = min(C::RB, p.G * sw.Lb - chunk * C::RB);
    T* const out = static_cast<T*>(p.out);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int d0 = lane * 4;
    auto orow = [&](int r) { return out_row<kVar>(p, b, kvh, sw.Lb, sw.q0, chunk * C::RB + r); };
    if (ng == 0) {
        for (int r = warp; r < rows_valid; r += 4)
            store4<T>(out, orow(r) * kD + d0, make_float4(0.f, 0.f, 0.f, 0.f));
        return;
    }
    const int sib = kvh * sw.nch + chunk;  // the walker's segment order within b
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
        store4<T>(out, orow(r) * kD + d0,
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

struct PoolMaps {
    CUtensorMap k, v, kt, vt;  // full tiles, partial tiles
};

template <class C, int F>
pa_status launch_split_combine(const Call& c, const DecodeParams& p, int grid, long long nseg,
                               const PoolMaps& m) {
    static int attr_done[64] = {0};
    if (c.dev.device >= 0 && c.dev.device < 64 && !attr_done[c.dev.device]) {
        if (cudaFuncSetAttribute(decode_split_kernel<C, F>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::SMEM) != cudaSuccess)
            return PA_ERR_CUDA;
        attr_done[c.dev.device] = 1;
    }
    if (c.ev_before && cudaEventRecord(c.ev_before, c.stream) != cudaSuccess) return PA_ERR_CUDA;
    if (c.overlap_prev) {  // may start while the preceding tile kernel runs
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(C::THREADS);
        cfg.dynamicSmemBytes = C::SMEM;
        cfg.stream = c.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, decode_split_kernel<C, F>, m.k, m.v, m.kt, m.vt, p) !=
            cudaSuccess)
            return PA_ERR_CUDA;
    } else {
        decode_split_kernel<C, F><<<grid, C::THREADS, C::SMEM, c.stream>>>(m.k, m.v, m.kt, m.vt, p);
        if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    }
    if (c.ev_after && cudaEventRecord(c.ev_after, c.stream) != cudaSuccess) return PA_ERR_CUDA;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nseg));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = c.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_combine_kernel<C, F == 2>, p) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

template <class C>
pa_status launch_cfg(const Call& c) {
    const pa_shape& sh = c.sh;
    const int grid = c.dev.sm_count * C::MINB;
    // the workspace is sized for the largest grid any configuration uses
    const WsLayout w = ws_layout(sh, decode_grid(sh, c.dev.sm_count), C::RB);
    if (c.ws_bytes < w.total) return PA_ERR_WORKSPACE;
    // Bound on the flattened unit count: every index stays inside int.
    const long long max_units = w.nseg * ((static_cast<long long>(sh.max_pages_per_seq) *
                                               sh.page_size + C::GRAN - 1) / C::GRAN);
    if (max_units >= INT_MAX / 2) return PA_ERR_UNSUPPORTED;

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
    p.mask = c.mask;
    p.mask_S = c.mask_S;
    p.cu_q = c.cu_q;
    p.total_q = c.total_q;
    p.route_mixed = c.route_mixed;
    p.tk_pages = C::TK / sh.page_size;
    p.tk_slots = C::TK % sh.page_size;
    // tensor-core consumers: K and V land through 2-D maps over the pools,
    // boxes of gcd(page_size, GRAN) rows for full tiles and of 16 (or 8) rows
    // for a segment's last tile
    {
        int a = sh.page_size, b = C::GRAN;
        while (b) {
            const int t = a % b;
            a = b;
            b = t;
        }
        p.boxr = a;
    }
    p.boxr_tail = sh.page_size % 16 == 0 ? 16 : 8;
    PoolMaps m;
    memset(&m, 0, sizeof m);
    if constexpr (C::MMA) {
        const long long pool_rows = static_cast<long long>(sh.num_pages) * sh.H_kv * sh.page_size;
        if (!make_map(&m.k, c.kp, pool_rows, p.boxr) || !make_map(&m.v, c.vp, pool_rows, p.boxr) ||
            !make_map(&m.kt, c.kp, pool_rows, p.boxr_tail) ||
            !make_map(&m.vt, c.vp, pool_rows, p.boxr_tail))
            return PA_ERR_CUDA;
        if (c.cu_q) return launch_split_combine<C, 2>(c, p, grid, w.nseg, m);
        return launch_split_combine<C, 0>(c, p, grid, w.nseg, m);
    } else {
        if (c.cu_q) return launch_split_combine<C, 2>(c, p, grid, w.nseg, m);
        if (c.mask) return launch_split_combine<C, 1>(c, p, grid, w.nseg, m);
        return launch_split_combine<C, 0>(c, p, grid, w.nseg, m);
    }
}

// The tensor-core consumers (128-key tiles that start on 128-key boundaries,
// up to 4 query rows per segment) take bf16 without an explicit mask on pages
// of a multiple of 64 slots: a full tile is then one or two TMA boxes per
// operand half.  Smaller pages would need up to 16 boxes a tile, and the
// producer's issue cost would bind; those keep the CUDA-core consumers and 1-D
// bulk copies.
bool decode_mma_ok(const Call& c) {
    return c.sh.dtype == PA_BF16 && !c.mask && c.sh.page_size % 64 == 0 &&
           decode_rows_per_chunk(c.sh) <= 4;
}

}  // namespace

int decode_rows_per_chunk(const pa_shape& sh) {
    const long long R = static_cast<long long>(sh.H_q / sh.H_kv) * sh.L;
    if (R <= 1) return 1;
    if (R <= 2) return 2;
    if (R <= 4) return 4;
    return 8;
}

// Largest persistent grid of any decode configuration (one CTA per SM).
int decode_grid(const pa_shape& /*sh*/, int sm_count) { return sm_count > 0 ? sm_count : 1; }

size_t decode_workspace_bytes(const pa_shape& sh, int sm_count) {
    return ws_layout(sh, decode_grid(sh, sm_count), decode_rows_per_chunk(sh)).total;
}

size_t varlen_plan_offset(const pa_shape& sh, int sm_count) {
    const size_t d = decode_workspace_bytes(sh, sm_count);
    return align_up(d > kFlagBytes ? d : kFlagBytes, 256);
}

size_t tile_partials_offset(const pa_shape& sh, int sm_count) {
    return align_up(varlen_plan_offset(sh, sm_count) + 4 * (static_cast<size_t>(sh.B) + 2), 256);
}

size_t workspace_bytes_total(const pa_shape& sh, int sm_count) {
    return tile_partials_offset(sh, sm_count) + tile_partial_bytes(sh, sm_count);
}

pa_status decode_launch(const Call& c) {
    const int RB = decode_rows_per_chunk(c.sh);
    using bf = __nv_bfloat16;
    if (decode_mma_ok(c)) {
        switch (RB) {
            case 1: return launch_cfg<Cfg<bf, 1, 8, 128, 8, 3, 1, 128, true>>(c);
            case 2: return launch_cfg<Cfg<bf, 2, 8, 128, 8, 3, 1, 128, true>>(c);
            default: return launch_cfg<Cfg<bf, 4, 8, 128, 8, 3, 1, 128, true>>(c);
        }
    }
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
