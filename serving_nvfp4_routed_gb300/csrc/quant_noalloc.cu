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
// looked up once per device with cudaGetSymbolAddress, on the first call
// made while that device is current, and cached.  Every call on a device
// shares the one array, so calls that may overlap on the GPU (two streams,
// two host threads) race and must be ordered by the caller.
#include <mutex>

#include "common.cuh"
#include "internal.cuh"

namespace nvfp4 {

namespace {

constexpr int kNoAllocMaxTensors = 4096;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_amax[kNoAllocMaxTensors];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_amax on the current device (nullptr on error).
float* noalloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_amax) != cudaSuccess) return nullptr;
        g_noalloc_ptr[dev] = static_cast<float*>(p);
    }
    return g_noalloc_ptr[dev];
}

}  // namespace

}  // namespace nvfp4

using namespace nvfp4;

extern "C" int nvfp4_quantize_weights_noalloc_max_batch(void) { return kNoAllocMaxTensors; }

extern "C" nvfp4_status nvfp4_quantize_weights_noalloc(const uint16_t* w, int batch, int N, int K, uint8_t* codes,
                                                       uint8_t* scales, float* weight_scale_2,
                                                       cudaStream_t stream) {
    if (batch < 0 || N < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
    if (K % 16 != 0) return NVFP4_ERR_SHAPE;
    if (batch > kNoAllocMaxTensors) return NVFP4_ERR_SHAPE;  // beyond the built-in scratch
    if ((size_t)batch * N * K == 0) return NVFP4_OK;
    if (!w || !codes || !scales || !weight_scale_2) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(codes) || !aligned16(scales) || !aligned16(weight_scale_2))
        return NVFP4_ERR_ALIGN;
    float* amax = noalloc_scratch();
    if (!amax) return NVFP4_ERR_CUDA;
    // the running maxima start from zero on every call (the array keeps the
    // previous call's values)
    launch_zero(amax, sizeof(float) * batch, stream);
    const size_t n_per = (size_t)N * K;
    const int gx = (int)std::max<size_t>(
        1, std::min<size_t>((n_per / 8 + 255) / 256, (size_t)num_sms() * 8 / std::max(1, batch) + 1));
    NVFP4_LAUNCH("tensor_amax", stream,
                 tensor_amax_kernel<<<dim3(gx, batch), 256, 0, stream>>>(w, n_per, amax));
    const size_t total = n_per / 8 * batch;
    const int grid = (int)std::min<size_t>((total + 255) / 256, (size_t)num_sms() * 16);
    NVFP4_LAUNCH("quantize_weights", stream,
                 quantize_weights_kernel<<<grid, 256, 0, stream>>>(w, n_per, batch, amax, codes, scales,
                                                                   weight_scale_2));
    return last_launch_status();
}
