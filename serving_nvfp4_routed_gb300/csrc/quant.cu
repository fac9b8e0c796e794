// quant.cu -- NVFP4 quantisation on the GPU: the ModelOpt weight recipe
// (global amax pass, then block scales and codes) and static-scale
// activation quantisation.
//
// Format: TensorFold issue #308, "GLM-5.3-Flash on CUDA: read
// nvidia/GLM-5.3-Flash-NVFP4 (ModelOpt NVFP4) as stored, W4A16", section "The
// checkpoint" (e2m1 codes, e4m3 scale per 16 inputs, fp32 weight_scale_2,
// static input_scale); recipe: section "What the branch does" (experts
// packed by ModelOpt's recipe at load, one projection at a time).
//
// Each thread owns whole 16-value blocks (two 16-byte loads of bf16).
// The scale arithmetic is IEEE fp32 round-to-nearest in the recipe's order:
//   sf = (bam / 6) / gs;  s = e4m3_rn_sat(sf);  q = e2m1_rn_sat(v / (S * gs))
// so that codes and scales are bit-identical to the format's definition.
#include "common.cuh"
#include "internal.cuh"

namespace nvfp4 {

__global__ void zero_words_kernel(uint32_t* p, size_t n) {
    grid_dep_wait();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        p[i] = 0u;
}

void launch_zero(void* p, size_t bytes, cudaStream_t s) {
    size_t n = bytes / 4;
    if (n == 0) return;
    int grid = (int)std::min<size_t>((n + 255) / 256, (size_t)num_sms() * 8);
    NVFP4_LAUNCH("zero_words", s, launch_pdl(zero_words_kernel, dim3(grid), dim3(256), 0, s, reinterpret_cast<uint32_t*>(p), n));
}

// Per-tensor max |w| over `batch` tensors of n_per elements each.
__global__ void tensor_amax_kernel(const uint16_t* __restrict__ w, size_t n_per, float* __restrict__ amax) {
    const int b = blockIdx.y;
    const uint4* src = reinterpret_cast<const uint4*>(w + (size_t)b * n_per);
    const size_t n8 = n_per / 8;
    float m = 0.0f;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
        uint4 u = __ldg(src + i);
        uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m = fmaxf(m, fabsf(bf16_bits_to_f32(ww[j] & 0xFFFFu)));
            m = fmaxf(m, fabsf(bf16_bits_to_f32(ww[j] >> 16)));
        }
    }
    m = warp_max(m);
    __shared__ float red[32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.0f;
        v = warp_max(v);
        if (threadIdx.x == 0) atomic_max_nonneg(amax + b, v);
    }
}

// Scale byte of a 16-block with amax bam under the tensor scale gs, and the
// block's divisor S * gs (0 when the block quantises to zero codes).
__device__ __forceinline__ uint32_t block_scale(float bam, float gs, float& denom) {
    denom = 0.0f;
    if (!(gs > 0.0f)) return 0u;
    const uint32_t sbyte = f32_to_e4m3(__fdiv_rn(__fdiv_rn(bam, 6.0f), gs));
    const float S = e4m3_to_f32(sbyte);
    if (S != 0.0f) denom = __fmul_rn(S, gs);
    return sbyte;
}

// The e2m1 codes of 8 values of a block with divisor denom (packed, element 0
// in the low nibble): code(fl(v / denom)).
__device__ __forceinline__ uint32_t quant8(const float v[8], float denom) {
    if (denom == 0.0f) return 0u;
    const float r = __frcp_rn(denom);
    float q[8];
    bool near = false;  // a product near a significand 1, 1.25, 1.5 or 1.75: divide there
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        q[i] = __fmul_rn(v[i], r);
        near |= e2m1_quotient_near(q[i]);
    }
    if (near) {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = e2m1_quotient(v[i], denom, r);
    }
    return f32x8_to_e2m1x8(q);
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 u, float v[8], float& amax) {
    const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
    amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[2 * j] = bf16_bits_to_f32(ww[j] & 0xFFFFu);
        v[2 * j + 1] = bf16_bits_to_f32(ww[j] >> 16);
        amax = fmaxf(amax, fmaxf(fabsf(v[2 * j]), fabsf(v[2 * j + 1])));
    }
}

__device__ __forceinline__ void load_bf16x8(const uint16_t* p, float v[8], float& amax) {
    unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(p)), v, amax);
}

// Tensor blockIdx.y: one thread per 16-value block (two 16-byte loads), the
// blocks grid-strided over blockIdx.x; the tensor scale gs is taken once
// per thread.
__global__ void quantize_weights_kernel(const uint16_t* __restrict__ w, size_t n_per,
                                        const float* __restrict__ amax, uint8_t* __restrict__ codes,
                                        uint8_t* __restrict__ scales, float* __restrict__ ws2_out) {
    const int b = blockIdx.y;
    const float gs = __fdiv_rn(amax[b], 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) ws2_out[b] = gs;
    const size_t nblk = n_per / 16;
    const uint16_t* wb = w + (size_t)b * n_per;
    uint8_t* cb = codes + (size_t)b * (n_per / 2);
    uint8_t* sb = scales + (size_t)b * nblk;
    for (size_t k = blockIdx.x * (size_t)blockDim.x + threadIdx.x; k < nblk; k += (size_t)gridDim.x * blockDim.x) {
        float v0[8], v1[8], m0, m1;
        load_bf16x8(wb + k * 16, v0, m0);
        load_bf16x8(wb + k * 16 + 8, v1, m1);
        float denom;
        const uint32_t sbyte = block_scale(fmaxf(m0, m1), gs, denom);
        const uint32_t c0 = quant8(v0, denom), c1 = quant8(v1, denom);
        *reinterpret_cast<uint2*>(cb + k * 8) = make_uint2(c0, c1);
        sb[k] = (uint8_t)sbyte;
    }
}

// Output row r quantises source row src(r) with the input scale of the
// expert whose row range holds r.  A warp takes a unit of `spu` segments of
// one row, a segment being 32 16-value blocks (one per lane: 32-byte loads,
// 8-byte code and 1-byte scale stores); units are grid-strided.  A few rows
// (a decode batch) take one segment per unit so that every SM gets work;
// many rows take whole rows.  The expert offsets are cached in shared
// memory for the row's lookup.
constexpr int kQaWarps = 8;
constexpr int kQaMaxE = 1024;

__global__ void __launch_bounds__(kQaWarps * 32) quantize_act_kernel(
    const uint16_t* __restrict__ x, int M, int K, const int32_t* __restrict__ row_to_slot, int top_k,
    const float* __restrict__ input_scale, const int32_t* __restrict__ offsets, int E, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, int spu) {
    __shared__ int s_off[kQaMaxE + 1];
    grid_dep_wait();
    const bool cached = offsets && E <= kQaMaxE;
    if (cached)
        for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = offsets[i];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = K / 16;
    const int nseg = (nb + 31) / 32;
    const unsigned useg = (unsigned)((nseg + spu - 1) / spu);  // units per row
    const unsigned units = (unsigned)M * useg;
    for (unsigned u = blockIdx.x * kQaWarps + warp; u < units; u += gridDim.x * kQaWarps) {
        const int r = (int)(u / useg);
        const int seg0 = (int)(u % useg) * spu;
        const int src = row_to_slot ? row_to_slot[r] / top_k : r;
        float gs;
        if (offsets) {
            int lo = 0, hi = E;  // find e with offsets[e] <= r < offsets[e+1]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if ((cached ? s_off[mid] : offsets[mid]) <= r) lo = mid; else hi = mid;
            }
            gs = input_scale[lo];
        } else {
            gs = input_scale[0];
        }
        const uint16_t* xr = x + (size_t)src * K;
        const int b1 = min(nb, (seg0 + spu) * 32);
        for (int b = seg0 * 32 + lane; b < b1; b += 32) {
            float v0[8], v1[8], m0, m1;
            load_bf16x8(xr + (size_t)b * 16, v0, m0);
            load_bf16x8(xr + (size_t)b * 16 + 8, v1, m1);
            float denom;
            const uint32_t s0 = block_scale(fmaxf(m0, m1), gs, denom);
            const uint32_t c0 = quant8(v0, denom), c1 = quant8(v1, denom);
            *reinterpret_cast<uint2*>(codes + (size_t)r * (K / 2) + (size_t)b * 8) = make_uint2(c0, c1);
            scales[(size_t)r * nb + b] = (uint8_t)s0;
        }
    }
    grid_dep_launch();
}

void launch_quantize_act(const uint16_t* x, int M, int K, const int32_t* row_to_slot, int top_k,
                         const float* input_scale, const int32_t* offsets, int E, uint8_t* codes,
                         uint8_t* scales, cudaStream_t s) {
    if ((size_t)M * K == 0) return;
    const int cap = num_sms() * 8;  // CTAs
    const int nseg = (K / 16 + 31) / 32;
    // one segment per unit while the rows alone would leave warps idle
    const int spu = (long long)M < (long long)cap * kQaWarps ? 1 : nseg;
    const long long units = (long long)M * ((nseg + spu - 1) / spu);
    const int grid = (int)std::min<long long>((units + kQaWarps - 1) / kQaWarps, cap);
    NVFP4_LAUNCH("quantize_act", s,
                 launch_pdl(quantize_act_kernel, dim3(grid), dim3(kQaWarps * 32), 0, s, x, M, K, row_to_slot,
                            top_k, input_scale, offsets, E, codes, scales, spu));
}

nvfp4_status check_weight_recipe(const uint16_t* w, int batch, int N, int K, const uint8_t* codes,
                                 const uint8_t* scales, const float* weight_scale_2) {
    if (batch < 0 || N < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
    if (K % 16 != 0 || batch > kMaxRecipeBatch) return NVFP4_ERR_SHAPE;
    if ((size_t)batch * N * K == 0) return NVFP4_OK;
    if (!w || !codes || !scales || !weight_scale_2) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(codes) || !aligned16(scales) || !aligned16(weight_scale_2))
        return NVFP4_ERR_ALIGN;
    return NVFP4_OK;
}

nvfp4_status launch_weight_recipe(const uint16_t* w, int batch, int N, int K, float* amax, uint8_t* codes,
                                  uint8_t* scales, float* weight_scale_2, cudaStream_t stream) {
    // the running maxima start from zero on every call
    launch_zero(amax, sizeof(float) * batch, stream);
    const size_t n_per = (size_t)N * K;
    const int gx = (int)std::max<size_t>(
        1, std::min<size_t>((n_per / 8 + 255) / 256, (size_t)num_sms() * 8 / std::max(1, batch) + 1));
    NVFP4_LAUNCH("tensor_amax", stream,
                 tensor_amax_kernel<<<dim3(gx, batch), 256, 0, stream>>>(w, n_per, amax));
    const int qx = (int)std::max<size_t>(
        1, std::min<size_t>((n_per / 16 + 255) / 256, (size_t)num_sms() * 16 / std::max(1, batch) + 1));
    NVFP4_LAUNCH("quantize_weights", stream,
                 quantize_weights_kernel<<<dim3(qx, batch), 256, 0, stream>>>(w, n_per, amax, codes, scales,
                                                                              weight_scale_2));
    return last_launch_status();
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" size_t nvfp4_quantize_weights_workspace_size(int batch, int N, int K) {
    (void)N;
    (void)K;
    return align_up((size_t)(batch > 0 ? batch : 0) * sizeof(float), 256);
}

extern "C" nvfp4_status nvfp4_quantize_weights(const uint16_t* w, int batch, int N, int K, uint8_t* codes,
                                               uint8_t* scales, float* weight_scale_2, void* ws,
                                               size_t ws_bytes, cudaStream_t stream) {
    const nvfp4_status st = check_weight_recipe(w, batch, N, K, codes, scales, weight_scale_2);
    if (st != NVFP4_OK || (size_t)batch * N * K == 0) return st;
    if (!ws) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(ws)) return NVFP4_ERR_ALIGN;
    if (ws_bytes < nvfp4_quantize_weights_workspace_size(batch, N, K)) return NVFP4_ERR_WORKSPACE;
    return launch_weight_recipe(w, batch, N, K, static_cast<float*>(ws), codes, scales, weight_scale_2, stream);
}

extern "C" nvfp4_status nvfp4_quantize_act(const uint16_t* x, int M, int K, const int32_t* row_to_slot,
                                           int top_k, const float* input_scale,
                                           const int32_t* expert_offsets, int E, uint8_t* codes,
                                           uint8_t* scales, cudaStream_t stream) {
    if (M < 0 || K < 0) return NVFP4_ERR_INVALID_ARG;
    if (K % 16 != 0) return NVFP4_ERR_SHAPE;
    if (M == 0 || K == 0) return NVFP4_OK;
    if (!x || !input_scale || !codes || !scales) return NVFP4_ERR_INVALID_ARG;
    if (row_to_slot && top_k < 1) return NVFP4_ERR_INVALID_ARG;
    if (expert_offsets && (E < 1 || E > 1024)) return NVFP4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(input_scale) ||
        (row_to_slot && !aligned16(row_to_slot)) || (expert_offsets && !aligned16(expert_offsets)))
        return NVFP4_ERR_ALIGN;
    launch_quantize_act(x, M, K, row_to_slot, top_k, input_scale, expert_offsets, E, codes, scales, stream);
    return last_launch_status();
}
