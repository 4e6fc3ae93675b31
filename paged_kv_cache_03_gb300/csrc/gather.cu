// gather.cu -- debug gather of the page translation of "Week 3 Day 5: Paged
// FlashAttention", Task 1: dense[b, kvh, s, :] = pages[block_table[b, s /
// page_size], kvh, s % page_size, :] for s < context_lens[b], zero after.
// Pure data movement (16-byte chunks), so it is compared bitwise.
#include "internal.h"

namespace pa {
namespace {

__global__ void gather_kernel(const uint4* kp, const uint4* vp, const int32_t* bt,
                              const int32_t* ctx, int H_kv, int ps, int max_npg, int num_pages,
                              int max_S, int cpr, uint4* kd, uint4* vd, uint32_t* flag) {
    const int b = blockIdx.z, kvh = blockIdx.y;
    int S = ctx[b];
    const long long cap = static_cast<long long>(max_npg) * ps;
    if (S < 0 || S > cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(flag, PA_FLAG_BAD_CONTEXT);
        S = S < 0 ? 0 : static_cast<int>(cap);
    }
    if (S > max_S) S = max_S;
    const long long n = static_cast<long long>(max_S) * cpr;
    const long long dbase = (static_cast<long long>(b) * H_kv + kvh) * n;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int s = static_cast<int>(i / cpr);
        const int c = static_cast<int>(i - static_cast<long long>(s) * cpr);
        uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
        if (s < S) {
            const int pp = bt[static_cast<long long>(b) * max_npg + s / ps];
            if (pp >= 0 && pp < num_pages) {
                const long long row = (static_cast<long long>(pp) * H_kv + kvh) * ps + s % ps;
                kv = kp[row * cpr + c];
                vv = vp[row * cpr + c];
            } else if (c == 0) {
                atomicOr(flag, PA_FLAG_BAD_PAGE);
            }
        }
        kd[dbase + i] = kv;
        vd[dbase + i] = vv;
    }
}

}  // namespace

pa_status gather_launch(const pa_shape& sh, const void* kp, const void* vp, const int32_t* bt,
                        const int32_t* ctx, int max_S, void* kd, void* vd, uint32_t* flag,
                        cudaStream_t stream) {
    if (sh.B > 65535 || sh.H_kv > 65535) return PA_ERR_UNSUPPORTED;
    const int es = sh.dtype == PA_BF16 ? 2 : 4;
    const int cpr = sh.D * es / 16;
    const long long n = static_cast<long long>(max_S) * cpr;
    const int threads = 256;
    long long blocks = (n + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    dim3 grid(static_cast<unsigned>(blocks), sh.H_kv, sh.B);
    gather_kernel<<<grid, threads, 0, stream>>>(
        static_cast<const uint4*>(kp), static_cast<const uint4*>(vp), bt, ctx, sh.H_kv,
        sh.page_size, sh.max_pages_per_seq, sh.num_pages, max_S, cpr, static_cast<uint4*>(kd),
        static_cast<uint4*>(vd), flag);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
