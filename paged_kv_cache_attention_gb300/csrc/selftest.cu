// selftest.cu -- a check that the bounded pipeline waits give up by themselves
// on this device.  Every wait of the library's kernels on a pipeline barrier
// is bounded: when the phase does not complete within the limit the wait
// ORs PKV_DEVERR_TIMEOUT into the caller's error word and returns, the kernel
// leaves, and the context stays usable.  This call runs one such wait on a
// barrier nothing arrives on, so that a caller (or a test) can see that path
// end to end without breaking any real pipeline.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(int32_t *dev_error) {
    __shared__ alignas(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncwarp();
    // phase 0 never completes: the wait must give up after its limit
    warp_wait_bounded(b, 0, dev_error);
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_selftest_bounded_wait(int32_t *dev_error, void *stream) {
    if (!dev_error) return PKV_ERR_INVALID_ARG;
    pkv::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_error);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
