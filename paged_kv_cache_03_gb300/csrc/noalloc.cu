// noalloc.cu -- the decode schedule with its scratch in a fixed, library-owned
// device array, for callers that cannot allocate device memory.
//
// Who needs this: a serving process that has handed all free HBM to its K/V
// page pool and caching allocator cannot get a fresh workspace from
// cudaMalloc (the call fails, or would have to bypass the allocator that owns
// the memory), and cudaMalloc/cudaFree may synchronise the whole device,
// which a latency-bound decode loop cannot afford.  Such callers pass only
// inputs and outputs; the scratch lives here.
//
// The array is a file-scope __device__ variable, so every GPU on which the
// library is used holds kNoAllocScratchBytes for the life of the process.
// Host code cannot use the array's name as a device address; the first call
// on each device looks the address up with cudaGetSymbolAddress (with that
// device current) and caches it.  That first call may load the module, so it
// should happen before any stream capture.
//
// All calls share the one array and it keeps the last call's contents.  Each
// call clears the 4-byte error flag at its start; everything else in the
// scratch is written before it is read.  Two calls whose kernels overlap on
// the GPU (different streams, no ordering between them) race on the scratch.
#include <mutex>

#include "internal.h"

namespace pa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {};

pa_status scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    if (dev >= 64) return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return PA_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_paged_attention_decode_noalloc(
    const pa_shape* shape, const void* query, const void* key_pages, const void* value_pages,
    const int32_t* block_table, const int32_t* context_lens, float scale, int causal, void* out,
    uint32_t* device_flag_out, void* cuda_stream) {
    if (!shape) return PA_ERR_INVALID_ARG;
    void* scratch = nullptr;
    pa_status st = pa::scratch_for_current_device(&scratch);
    if (st != PA_OK) return st;
    const size_t need = pa_workspace_bytes(shape);
    if (need == 0) return PA_ERR_INVALID_ARG;
    if (need > pa::kNoAllocScratchBytes) return PA_ERR_WORKSPACE;  // beyond the fixed maximum
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    if (cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    st = pa_paged_attention_sched(shape, query, key_pages, value_pages, block_table, context_lens,
                                  scale, causal, out, scratch, pa::kNoAllocScratchBytes,
                                  cuda_stream, PA_SCHED_DECODE);
    if (st != PA_OK) return st;
    if (device_flag_out &&
        cudaMemcpyAsync(device_flag_out, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                        s) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}
