// selftest.cu -- exercises the give-up path of the kernels' bounded on-chip
// waits without a fault: one warp waits, with mbar_wait_for (the wait every
// kernel uses), on an mbarrier phase that nothing ever completes.  The wait
// runs out after the given time, the kernel records PA_FLAG_TIMEOUT in the
// flag word and returns normally, so the context stays usable.
#include "internal.h"
#include "ptx.cuh"

namespace pa {
namespace {

__global__ void wait_timeout_probe_kernel(uint32_t* flag, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);  // one arrival would complete phase 0; none comes
        fence_mbar_init();
    }
    __syncwarp();
    const bool ok = mbar_wait_for(b, 0, limit_ns);
    if (!ok && threadIdx.x == 0) atomicOr(flag, PA_FLAG_TIMEOUT);
}

}  // namespace

pa_status wait_timeout_launch(uint32_t* flag, unsigned long long limit_ns, cudaStream_t stream) {
    wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(flag, limit_ns);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
