// quant_noalloc.cu -- nvfp4_quantize_weights for callers that cannot
// allocate device memory.
//
// nvfp4_quantize_weights needs a small scratch buffer (one fp32 running max
// per tensor) that the caller normally passes as `ws`.  Some callers have no
// way to provide it: code that must not call cudaMalloc because another
// component owns all device memory (a fixed pool sized ahead of time), a
// plain-C loader linked against this library without any allocator of its
// own, or a hot loop that must not call cudaMalloc because it can implicitly
// synchronise the whole device.  For them this entry point keeps its
// scratch in a fixed array in the library's own device memory
// (kNoAllocMaxTensors floats, 16 KB on every GPU that loads the library,
// held until the process exits) and allocates nothing at any call.
//
// The array's host-side name is not a device address: its device address is
// looked up with cudaGetSymbolAddress on every call, with the caller's
// device current (a host-side query that allocates nothing), so a call made
// after cudaDeviceReset or under another context of the device still gets
// the array of the context it runs in.  The first call of a process on a
// device may load the library's device code (lazy module loading), so make
// it before any stream capture.  Every call on a device shares the one
// array, so calls that may overlap on the GPU (two streams, two host
// threads) race and must be ordered by the caller.
#include "common.cuh"
#include "internal.cuh"

namespace nvfp4 {

namespace {

constexpr int kNoAllocMaxTensors = 4096;

static __device__ __align__(256) float g_noalloc_amax[kNoAllocMaxTensors];

// Device address of g_noalloc_amax in the current context (nullptr on error).
float* noalloc_scratch() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_amax) != cudaSuccess) return nullptr;
    return static_cast<float*>(p);
}

}  // namespace

}  // namespace nvfp4

using namespace nvfp4;

extern "C" int nvfp4_quantize_weights_noalloc_max_batch(void) { return kNoAllocMaxTensors; }

extern "C" nvfp4_status nvfp4_quantize_weights_noalloc(const uint16_t* w, int batch, int N, int K, uint8_t* codes,
                                                       uint8_t* scales, float* weight_scale_2,
                                                       cudaStream_t stream) {
    if (batch > kNoAllocMaxTensors) return NVFP4_ERR_SHAPE;  // beyond the built-in scratch
    const nvfp4_status st = check_weight_recipe(w, batch, N, K, codes, scales, weight_scale_2);
    if (st != NVFP4_OK || (size_t)batch * N * K == 0) return st;
    float* amax = noalloc_scratch();
    if (!amax) return NVFP4_ERR_CUDA;
    return launch_weight_recipe(w, batch, N, K, amax, codes, scales, weight_scale_2, stream);
}
