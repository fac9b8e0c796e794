// selftest.cu -- failure detection of the library's bounded waits, exercised
// without faulting the GPU: one CTA waits on an mbarrier that nothing ever
// arrives on.  The wait gives up after its clock budget (about 2 s), writes
// NVFP4_ERR_TIMEOUT to the status word and the kernel returns normally, so
// the context stays usable.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {
namespace {

using namespace tc;

__global__ void bounded_wait_kernel(int32_t* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_abort;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        s_abort = 0;
        mbar_fence_init();
    }
    __syncthreads();
    warp_wait(smem_u32(&bar), 0, &s_abort, status);  // phase 0 never completes
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_selftest_bounded_wait(int32_t* d_status, cudaStream_t stream) {
    if (!d_status) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(d_status)) return NVFP4_ERR_ALIGN;
    NVFP4_LAUNCH("selftest_bounded_wait", stream, bounded_wait_kernel<<<1, 32, 0, stream>>>(d_status));
    return last_launch_status();
}
