// moe_gemv.cu -- decode-shaped grouped NVFP4 expert GEMM.
//
// TensorFold issue #308 "GLM-5.3-Flash on CUDA: read nvidia/GLM-5.3-Flash-NVFP4
// (ModelOpt NVFP4) as stored, W4A16", "What the branch does": the routed
// experts run through one grouped kernel over bf16 rows, with weight_scale_2
// as the per-expert multiplier; FP4 x FP4 (W4A4) is the checkpoint's own
// math.  "Questions", item 4: decode and prompt shapes get different kernels.
//
// With few tokens per expert the layer is a stream of 4.5-bit weights
// (codes + e4m3 scales) from HBM; every weight is read once and used by the
// handful of rows routed to its expert.  Design:
//   * work item = (expert, 16 output features, up to 8 routed rows); work
//     items are taken from an atomic counter so that CTAs stay busy;
//   * the CTA's NW warps split K; each warp reduces its K range with
//     mma.sync m16n8k16 (f32 accumulate) and the partial sums meet in shared
//     memory;
//   * K is permuted inside each CK-wide chunk so that lane quad c of a
//     warp owns the contiguous physical range [c*CK/4, (c+1)*CK/4): every
//     lane loads its weights with 16-byte loads straight into the mma
//     A-fragment positions, and the B operand uses the same permutation
//     (a dot product does not depend on the order of its terms);
//   * dequantisation in registers: cvt e2m1x2 -> f16x2 (exact), times the
//     block scale e4m3 -> f16 (exact: every e2m1*e4m3 product has at most 6
//     significant bits and lies in [2^-10, 2688]);
//   * bf16 activations enter the f16 MMA after a per-row power-of-two scale
//     2^-s that puts the row's max |x| in [2^14, 2^15): exact for every
//     element within 2^28 of the row max, the rest rounded on a grid of
//     2^-39 * row max; 2^s is applied to the fp32 accumulator;
//   * W4A4 activations are NVFP4 rows, dequantised to f16 like the weights
//     (exact), and the static input_scale multiplies the accumulator;
//   * epilogues: SwiGLU to bf16 h (with a running per-row max |h| for the
//     down projection's row scale), SwiGLU + NVFP4 requantisation of h with
//     the down input_scale (W4A4), or the weighted top-k combine into an fp32
//     accumulator with red.add (down projection).
#include "common.cuh"
#include "internal.cuh"

namespace nvfp4 {

namespace {

template <int CK>
struct Chunk {
    static constexpr int TS = CK / 4;   // physical K per lane
    static constexpr int CB = CK / 8;   // code bytes per lane per row
    static constexpr int SB = CK / 64;  // scale bytes per lane per row
    static constexpr int KS = CK / 16;  // mma k-steps per chunk
    static constexpr int CW = CB / 4;   // code words per lane per row
};

template <int CK>
__device__ __forceinline__ void load_codes(const uint8_t* p, uint32_t* w) {
    if constexpr (CK == 256) {
        uint4 u0 = __ldg(reinterpret_cast<const uint4*>(p));
        uint4 u1 = __ldg(reinterpret_cast<const uint4*>(p) + 1);
        w[0] = u0.x; w[1] = u0.y; w[2] = u0.z; w[3] = u0.w;
        w[4] = u1.x; w[5] = u1.y; w[6] = u1.z; w[7] = u1.w;
    } else {
        uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        w[0] = u.x; w[1] = u.y;
    }
}

template <int CK>
__device__ __forceinline__ uint32_t load_scales(const uint8_t* p) {
    if constexpr (CK == 256) return __ldg(reinterpret_cast<const uint32_t*>(p));
    else return __ldg(p);
}

// Dequantised f16x2 words for k-steps jj and jj+1 (jj even) from one code
// word of a lane: out[0] = phys 4jj..4jj+1, out[1] = 4jj+2..4jj+3,
// out[2], out[3] the same for jj+1.  Both steps lie in 16-block jj/4.
__device__ __forceinline__ void deq_word(uint32_t word, uint32_t sw, int jj, uint32_t out[4]) {
    uint32_t f[4];
    e2m1x8_to_f16x8(word, f);
    const int blk = jj >> 2;
    const uint32_t s2 = e4m3x2_to_f16x2((sw >> (16 * (blk >> 1))) & 0xFFFFu);
    const uint32_t S = f16x2_bcast(s2, blk & 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = hmul2_u32(f[i], S);
}

__device__ __forceinline__ uint32_t bf16x2_scaled_to_f16x2(uint32_t u, float sc) {
    return f32x2_to_f16x2(bf16_bits_to_f32(u & 0xFFFFu) * sc, bf16_bits_to_f32(u >> 16) * sc);
}

// e2m1 codes of two values as one byte (lo in the low nibble), sign kept.
__device__ __forceinline__ uint32_t e2m1x2_byte(float lo, float hi) {
    uint32_t r;
    asm("{\n.reg .b8 b;\ncvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\nmov.b32 %0, {b, b, b, b};\n}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return (r & 0xFFu) | ((__float_as_uint(lo) >> 31) << 3) | ((__float_as_uint(hi) >> 31) << 7);
}

template <int CK, int BMODE, int OUTMODE, int NPROJ, int NW>
__global__ void __launch_bounds__(NW * 32) gemv_kernel(const GemvArgs a) {
    using C = Chunk<CK>;
    __shared__ float s_red[NW][NPROJ * 4][32];
    __shared__ int s_work;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int n_active = *a.n_active;
    const int total_tiles = a.tile_start[n_active];
    const int n_slabs = a.N / 16;
    const int total = total_tiles * n_slabs;
    const int nchunks = a.K / CK;
    const size_t K2 = (size_t)a.K / 2, K16 = (size_t)a.K / 16;

    for (;;) {
        if (threadIdx.x == 0) s_work = atomicAdd(a.work_counter, 1);
        __syncthreads();
        const int w = s_work;
        __syncthreads();
        if (w >= total) break;
        const int slab = w % n_slabs, tile = w / n_slabs;
        int lo = 0, hi = n_active;  // largest ai with tile_start[ai] <= tile
        while (hi - lo > 1) {
            int mid = (lo + hi) >> 1;
            if (a.tile_start[mid] <= tile) lo = mid; else hi = mid;
        }
        const int e = a.active[lo];
        const int row0 = a.offsets[e] + (tile - a.tile_start[lo]) * kGemvTokTile;
        const int nrows = min(kGemvTokTile, a.offsets[e + 1] - row0);
        const int n0 = slab * 16;

        // this lane's B row (token column g of the n-tile)
        const bool bvalid = g < nrows;
        const int r_b = row0 + (bvalid ? g : 0);
        int brow = r_b;
        float bscale = 1.0f;
        if constexpr (BMODE == B_BF16) {
            if (a.b_by_token) brow = a.row_to_slot ? a.row_to_slot[r_b] / a.top_k : r_b;
            bscale = exp2i(-row_exponent(a.b_amax[brow]));
        }

        float acc[NPROJ][4];
#pragma unroll
        for (int p = 0; p < NPROJ; ++p)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[p][i] = 0.0f;

        for (int ch = warp; ch < nchunks; ch += NW) {
            const size_t kb = (size_t)ch * CK + (size_t)c * C::TS;
            uint32_t acw[NPROJ][2][C::CW];
            uint32_t asw[NPROJ][2];
#pragma unroll
            for (int p = 0; p < NPROJ; ++p)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const size_t row = (size_t)e * a.N + n0 + g + 8 * hf;
                    load_codes<CK>(a.a_codes[p] + row * K2 + kb / 2, acw[p][hf]);
                    asw[p][hf] = load_scales<CK>(a.a_scales[p] + row * K16 + kb / 16);
                }
            uint32_t bw[C::TS / 2];  // B_BF16: bf16x2 words; B_NVFP4: code words then scale word
            uint32_t bsw = 0;
            if constexpr (BMODE == B_BF16) {
                if (bvalid) {
                    const uint4* src = reinterpret_cast<const uint4*>(a.b_bf16 + (size_t)brow * a.K + kb);
#pragma unroll
                    for (int i = 0; i < C::TS / 8; ++i) {
                        uint4 u = __ldg(src + i);
                        bw[4 * i] = u.x; bw[4 * i + 1] = u.y; bw[4 * i + 2] = u.z; bw[4 * i + 3] = u.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < C::TS / 2; ++i) bw[i] = 0u;
                }
            } else {
                if (bvalid) {
                    load_codes<CK>(a.b_codes + (size_t)r_b * K2 + kb / 2, bw);
                    bsw = load_scales<CK>(a.b_scales + (size_t)r_b * K16 + kb / 16);
                } else {
#pragma unroll
                    for (int i = 0; i < C::CW; ++i) bw[i] = 0u;
                }
            }
#pragma unroll
            for (int jj = 0; jj < C::KS; jj += 2) {
                uint32_t bq[4];  // B words for steps jj (bq[0], bq[1]) and jj+1 (bq[2], bq[3])
                if constexpr (BMODE == B_BF16) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) bq[i] = bf16x2_scaled_to_f16x2(bw[2 * jj + i], bscale);
                } else {
                    deq_word(bw[jj >> 1], bsw, jj, bq);
                }
#pragma unroll
                for (int p = 0; p < NPROJ; ++p) {
                    uint32_t r0[4], r1[4];
                    deq_word(acw[p][0][jj >> 1], asw[p][0], jj, r0);
                    deq_word(acw[p][1][jj >> 1], asw[p][1], jj, r1);
                    const uint32_t af0[4] = {r0[0], r1[0], r0[1], r1[1]};
                    const uint32_t af1[4] = {r0[2], r1[2], r0[3], r1[3]};
                    const uint32_t b0[2] = {bq[0], bq[1]};
                    const uint32_t b1[2] = {bq[2], bq[3]};
                    mma_16816(acc[p], af0, b0);
                    mma_16816(acc[p], af1, b1);
                }
            }
        }

        // cross-warp reduction of the partial sums
#pragma unroll
        for (int p = 0; p < NPROJ; ++p)
#pragma unroll
            for (int i = 0; i < 4; ++i) s_red[warp][p * 4 + i][lane] = acc[p][i];
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int p = 0; p < NPROJ; ++p)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float s = 0.0f;
#pragma unroll
                    for (int w2 = 0; w2 < NW; ++w2) s += s_red[w2][p * 4 + i][lane];
                    acc[p][i] = s;
                }

            // epilogue: column cc of this lane is permuted row row0 + 2c + cc
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int col = 2 * c + cc;
                const bool valid = col < nrows;
                const int r = row0 + (valid ? col : 0);
                float rs;  // scale taking the accumulator to x W^T (without ws2)
                if constexpr (BMODE == B_BF16) {
                    int br = r;
                    if (a.b_by_token) br = a.row_to_slot ? a.row_to_slot[r] / a.top_k : r;
                    rs = exp2i(row_exponent(a.b_amax[br]));
                } else {
                    rs = a.b_gs[e];
                }
                if constexpr (OUTMODE == OUT_H || OUTMODE == OUT_HQ) {
                    const float wg = a.a_ws2[0][e], wu = a.a_ws2[1][e];
                    float hv[2];
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const float G = round_bf16(__fmul_rn(__fmul_rn(acc[0][2 * hf + cc], rs), wg));
                        const float U = round_bf16(__fmul_rn(__fmul_rn(acc[NPROJ - 1][2 * hf + cc], rs), wu));
                        const float sg = G / (1.0f + expf(-G));
                        hv[hf] = round_bf16(sg * U);
                    }
                    if constexpr (OUTMODE == OUT_H) {
                        if (valid) {
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf)
                                a.h_out[(size_t)r * a.N + n0 + g + 8 * hf] =
                                    f32_to_bf16_bits(hv[hf]);
                        }
                        if (a.h_amax) {
                            float m = valid ? fmaxf(fabsf(hv[0]), fabsf(hv[1])) : 0.0f;
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                            if (valid && g == 0) atomic_max_nonneg(a.h_amax + r, m);
                        }
                    } else {
                        // NVFP4 requantisation of h: this 16-feature slab is one block
                        const float gs2 = a.hq_gs[e];
                        float m = fmaxf(fabsf(hv[0]), fabsf(hv[1]));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                        uint32_t sbyte = 0, q[2] = {0u, 0u};
                        if (gs2 > 0.0f) {
                            const float sf = __fdiv_rn(__fdiv_rn(m, 6.0f), gs2);
                            sbyte = f32_to_e4m3(sf);
                            const float S = e4m3_to_f32(sbyte);
                            if (S != 0.0f) {
                                const float den = __fmul_rn(S, gs2);
                                const uint32_t byte = e2m1x2_byte(__fdiv_rn(hv[0], den), __fdiv_rn(hv[1], den));
                                q[0] = byte & 0xFu;
                                q[1] = byte >> 4;
                            }
                        }
                        const uint32_t p0 = __shfl_down_sync(0xffffffffu, q[0], 4);
                        const uint32_t p1 = __shfl_down_sync(0xffffffffu, q[1], 4);
                        if (valid && (g & 1) == 0) {
                            uint8_t* dst = a.hq_out + (size_t)r * (a.N / 2) + n0 / 2;
                            dst[g / 2] = (uint8_t)(q[0] | (p0 << 4));
                            dst[g / 2 + 4] = (uint8_t)(q[1] | (p1 << 4));
                        }
                        if (valid && g == 0) a.hs_out[(size_t)r * (a.N / 16) + n0 / 16] = (uint8_t)sbyte;
                    }
                } else if constexpr (OUTMODE == OUT_COMBINE) {
                    if (valid) {
                        const int slot = a.row_to_slot[r];
                        const int t = slot / a.top_k;
                        const float wt = a.topk_w[slot];
                        const float ws = a.a_ws2[0][e];
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const float y = __fmul_rn(__fmul_rn(acc[0][2 * hf + cc], rs), ws);
                            atomicAdd(a.acc_out + (size_t)t * a.N + n0 + g + 8 * hf, wt * y);
                        }
                    }
                } else {  // OUT_BF16
                    if (valid) {
                        const float ws = a.a_ws2[0][e];
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf)
                            a.y_out[(size_t)r * a.N + n0 + g + 8 * hf] =
                                f32_to_bf16_bits(__fmul_rn(__fmul_rn(acc[0][2 * hf + cc], rs), ws));
                    }
                }
            }
        }
        __syncthreads();
    }
}

constexpr int kNW = 8;

template <int CK, int BMODE, int OUTMODE, int NPROJ>
void launch_t(const GemvArgs& a, int max_work, cudaStream_t s, const char* name) {
    auto kern = gemv_kernel<CK, BMODE, OUTMODE, NPROJ, kNW>;
    static int per_sm = 0;
    if (per_sm == 0) {
        int v = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kNW * 32, 0);
        per_sm = v > 0 ? v : 1;
    }
    int grid = std::max(1, std::min(max_work, per_sm * num_sms()));
    NVFP4_LAUNCH(name, s, kern<<<grid, kNW * 32, 0, s>>>(a));
}

template <int CK>
void launch_ck(int bmode, int outmode, const GemvArgs& a, int max_work, cudaStream_t s) {
    const bool two = a.nproj == 2;
    if (bmode == B_BF16) {
        if (outmode == OUT_H && two) return launch_t<CK, B_BF16, OUT_H, 2>(a, max_work, s, "gemv_gateup_w4a16");
        if (outmode == OUT_COMBINE) return launch_t<CK, B_BF16, OUT_COMBINE, 1>(a, max_work, s, "gemv_down_w4a16");
        if (outmode == OUT_BF16) return launch_t<CK, B_BF16, OUT_BF16, 1>(a, max_work, s, "gemv_linear_w4a16");
    } else {
        if (outmode == OUT_HQ && two) return launch_t<CK, B_NVFP4, OUT_HQ, 2>(a, max_work, s, "gemv_gateup_w4a4");
        if (outmode == OUT_COMBINE) return launch_t<CK, B_NVFP4, OUT_COMBINE, 1>(a, max_work, s, "gemv_down_w4a4");
    }
}

}  // namespace

void launch_gemv(int bmode, int outmode, const GemvArgs& a, int max_work, cudaStream_t s) {
    if (a.K % 256 == 0) launch_ck<256>(bmode, outmode, a, max_work, s);
    else launch_ck<64>(bmode, outmode, a, max_work, s);
}

// ---------------------------------------------------------------------------
// small helper kernels of the MoE call
// ---------------------------------------------------------------------------
__global__ void moe_prep_kernel(const uint16_t* __restrict__ x, int T, int d, float* __restrict__ x_amax,
                                float* __restrict__ acc, int k, float* __restrict__ h_amax, int* counters,
                                int n_counters) {
    const int t = blockIdx.x;
    if (t == 0 && threadIdx.x < n_counters) counters[threadIdx.x] = 0;
    float4* a4 = reinterpret_cast<float4*>(acc + (size_t)t * d);
    for (int i = threadIdx.x; i < d / 4; i += blockDim.x) a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (h_amax && threadIdx.x < k) h_amax[(size_t)t * k + threadIdx.x] = 0.0f;
    if (x_amax) {
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
        float m = 0.0f;
        for (int i = threadIdx.x; i < d / 8; i += blockDim.x) {
            uint4 u = __ldg(src + i);
            uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_f32(ww[j] & 0xFFFFu)), fabsf(bf16_bits_to_f32(ww[j] >> 16))));
        }
        m = warp_max(m);
        __shared__ float red[32];
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x < 32) {
            float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
            v = warp_max(v);
            if (threadIdx.x == 0) x_amax[t] = v;
        }
    }
}

void launch_moe_prep(const uint16_t* x, int T, int d, float* x_amax, float* acc, int k, float* h_amax,
                     int* counters, int n_counters, cudaStream_t s) {
    NVFP4_LAUNCH("moe_prep", s,
                 moe_prep_kernel<<<std::max(T, 1), 256, 0, s>>>(x, T, d, x_amax, acc, k, h_amax, counters,
                                                                n_counters));
}

__global__ void finalize_kernel(const float* __restrict__ acc, size_t n4, uint16_t* __restrict__ out) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        float4 v = reinterpret_cast<const float4*>(acc)[i];
        uint2 o;
        o.x = (uint32_t)f32_to_bf16_bits(v.x) | ((uint32_t)f32_to_bf16_bits(v.y) << 16);
        o.y = (uint32_t)f32_to_bf16_bits(v.z) | ((uint32_t)f32_to_bf16_bits(v.w) << 16);
        reinterpret_cast<uint2*>(out)[i] = o;
    }
}

void launch_finalize(const float* acc, size_t n, uint16_t* out, cudaStream_t s) {
    size_t n4 = n / 4;
    if (n4 == 0) return;
    int grid = (int)std::min<size_t>((n4 + 255) / 256, (size_t)num_sms() * 8);
    NVFP4_LAUNCH("finalize", s, finalize_kernel<<<grid, 256, 0, s>>>(acc, n4, out));
}

}  // namespace nvfp4
