// append.cu -- the new tokens' K/V rows stored in their pages.
//
// The L new tokens of sequence b are the last L logical positions of its
// context, s = context_lens[b] - L + t, and go through the same translation
// as every read of the page walk ("Week 3 Day 5: Paged FlashAttention",
// Task 1; pages and block tables are its prerequisite):
//   pages[block_table[b, s / page_size], kv_head, s % page_size, :]
//       = new[b, kv_head, t, :]
// The copy is exact.  One 16-byte chunk per thread: the reads of the new rows
// are fully coalesced, every destination row is one contiguous 256-byte
// (bf16) or 512-byte (fp32) segment.  Sequences whose context length breaks
// the contract set PA_FLAG_BAD_CONTEXT and are skipped; a token whose page id
// is out of range sets PA_FLAG_BAD_PAGE and is skipped.
#include "internal.h"

namespace pa {
namespace {

struct AppendParams {
    const uint4* k_new;
    const uint4* v_new;
    uint4* kp;
    uint4* vp;
    const int32_t* bt;
    const int32_t* ctx;
    uint32_t* flag;
    int rows;  // B * H_kv * L new rows (host-checked: rows * chunks per row < 2^31)
    int H_kv, L, ps, max_npg, num_pages;
    long long max_S;
};

// LPR lanes (16-byte chunks) per row: 16 for bf16, 32 for fp32.  Each thread
// copies its chunk of rows row, row + R, row + 2R, ... with R rows per grid
// sweep; the index arithmetic is 32-bit except the pool offset.
template <int LPR>
__global__ void __launch_bounds__(256) append_kv_kernel(const AppendParams p) {
    const int c = static_cast<int>(threadIdx.x) & (LPR - 1);
    const int rows_per_sweep = static_cast<int>(gridDim.x * blockDim.x) / LPR;
    for (int row = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) / LPR); row < p.rows;
         row += rows_per_sweep) {
        const int bk = row / p.L;  // (b, kvh) of the row, t its new token
        const int t = row - bk * p.L;
        const int b = bk / p.H_kv;
        const int kvh = bk - b * p.H_kv;
        const int S = __ldg(p.ctx + b);
        if (S < p.L || static_cast<long long>(S) > p.max_S) {
            if (kvh == 0 && t == 0 && c == 0) atomicOr(p.flag, PA_FLAG_BAD_CONTEXT);
            continue;
        }
        const int s = S - p.L + t;
        const int lp = s / p.ps, slot = s - lp * p.ps;
        const int pp = __ldg(p.bt + static_cast<long long>(b) * p.max_npg + lp);
        if (pp < 0 || pp >= p.num_pages) {
            if (c == 0) atomicOr(p.flag, PA_FLAG_BAD_PAGE);
            continue;
        }
        const int src = row * LPR + c;
        const long long dst = ((static_cast<long long>(pp) * p.H_kv + kvh) * p.ps + slot) * LPR + c;
        const uint4 kv = __ldcs(p.k_new + src);
        const uint4 vv = __ldcs(p.v_new + src);
        p.kp[dst] = kv;
        p.vp[dst] = vv;
    }
}

}  // namespace

pa_status append_launch(const pa_shape& sh, const void* k_new, const void* v_new, void* kp,
                        void* vp, const int32_t* bt, const int32_t* ctx, uint32_t* flag,
                        int sm_count, cudaStream_t stream) {
    AppendParams p;
    p.k_new = static_cast<const uint4*>(k_new);
    p.v_new = static_cast<const uint4*>(v_new);
    p.kp = static_cast<uint4*>(kp);
    p.vp = static_cast<uint4*>(vp);
    p.bt = bt;
    p.ctx = ctx;
    p.flag = flag;
    p.rows = sh.B * sh.H_kv * sh.L;
    p.H_kv = sh.H_kv;
    p.L = sh.L;
    p.ps = sh.page_size;
    p.max_npg = sh.max_pages_per_seq;
    p.num_pages = sh.num_pages;
    p.max_S = static_cast<long long>(sh.max_pages_per_seq) * sh.page_size;
    const int lpr = sh.dtype == PA_BF16 ? 16 : 32;
    // enough 256-thread blocks to cover the rows once, at most 8 per SM
    const long long blocks = (static_cast<long long>(p.rows) * lpr + 255) / 256;
    const long long cap = 8ll * (sm_count > 0 ? sm_count : 1);
    const unsigned grid = static_cast<unsigned>(blocks < cap ? blocks : cap);
    if (lpr == 16)
        append_kv_kernel<16><<<grid, 256, 0, stream>>>(p);
    else
        append_kv_kernel<32><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
