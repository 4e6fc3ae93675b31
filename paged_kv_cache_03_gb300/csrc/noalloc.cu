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
// Host code cannot use the array's name as a device address: each call looks
// the address up with cudaGetSymbolAddress, with the calling thread's device
// current.  The lookup is cheap once the library's device code is loaded on
// that device, and it stays right if the context is destroyed and created
// again (cudaDeviceReset).  The first call on a device may load that code, so
// it should happen before any stream capture.
//
// Every argument is checked before anything is enqueued: a rejected call
// touches neither the array nor device_flag_out.  All calls share the one
// array and it keeps the last call's contents.  Each accepted call clears the
// 4-byte error flag at its start; everything else in the scratch is written
// before it is read.  Two calls whose kernels overlap on the GPU (different
// streams, no ordering between them) race on the scratch.
#include "internal.h"

namespace pa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

}  // namespace
}  // namespace pa

extern "C" pa_status pa_paged_attention_decode_noalloc(
    const pa_shape* shape, const void* query, const void* key_pages, const void* value_pages,
    const int32_t* block_table, const int32_t* context_lens, float scale, int causal, void* out,
    uint32_t* device_flag_out, void* cuda_stream) {
    // the same host-side checks as the regular entry points, first
    pa_status st = pa::check_call_args(shape, query, key_pages, value_pages, block_table,
                                       context_lens, scale, out);
    if (st != PA_OK) return st;
    if (device_flag_out && reinterpret_cast<uintptr_t>(device_flag_out) % 4 != 0)
        return PA_ERR_INVALID_ARG;
    pa::DeviceInfo dev;
    st = pa::current_device_info(&dev);
    if (st != PA_OK) return st;
    if (dev.cc_major != 10 || dev.cc_minor != 3) return PA_ERR_UNSUPPORTED;
    const size_t need = pa::decode_workspace_bytes(*shape, dev.sm_count);  // the page walk's
    if (need > pa::kNoAllocScratchBytes) return PA_ERR_WORKSPACE;  // beyond the fixed maximum
    void* scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, pa::g_noalloc_scratch) != cudaSuccess || !scratch) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
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
