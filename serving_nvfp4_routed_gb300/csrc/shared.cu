// shared.cu -- the BF16 shared-expert MLP after the weighted combine:
//   G = bf16(x Wg^T)   U = bf16(x Wu^T)   h = bf16(silu(G) * U)
//   out = bf16(out + h Wd^T)          (out holds the routed layer's result)
//
// TensorFold issue #308, "The checkpoint": the shared experts stay BF16 next
// to the NVFP4 routed experts; "What the branch does": the shared expert runs
// as a BF16 MLP.  It runs on every token, so it is two dense GEMMs.
//
// Both GEMMs: one CTA per (128 tokens, NT output columns) tile, NT = 256,
// or 64 when the 256-wide tiles would leave most SMs idle (a decode batch:
// the weights are then spread over 4x as many CTAs);
// tcgen05.mma kind::f16 with bf16 A (rows) and bf16 B (weight rows) exactly
// as stored, both moved by TMA (128-byte swizzle, k-stages of 64, a ring of
// 4), M=128, N=NT, an fp32 accumulator in tensor memory.  Gate/up tile:
// B rows 0..NT/2-1 = Wg rows f0.., NT/2..NT-1 = Wu rows f0.., so a token's gate
// and up values for a feature share one TMEM lane and the SwiGLU is local
// to the thread.  Warp 0 runs the MMA loop (one elected lane issues), warp
// 1's lane 0 the TMA ring, warps 4-7 the epilogue (one token per lane).
// mbarrier waits are bounded and report NVFP4_ERR_TIMEOUT.
#include "common.cuh"
#include "internal.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {

namespace {

using namespace tc;

constexpr int SM_ = 128;        // tokens per tile (MMA M)
constexpr int SN = 256;         // widest tile (MMA N); shape rules refer to it
constexpr int SKS = 64;         // k per stage (128 bytes of bf16)
constexpr int SS = 4;           // stage ring
constexpr int kSA = SM_ * SKS * 2;   // 16 KB
template <int NT>
struct SGeo {
    static constexpr int kSB = NT * SKS * 2;
    static constexpr int kStage = kSA + kSB;
    static constexpr int kSmem = 1024 + SS * kStage;
};
constexpr int kSThreads = 256;
enum { SH_SWIGLU = 0, SH_ADD = 1 };

struct SharedArgs {
    CUtensorMap tmap_a, tmap_b0, tmap_b1;  // A rows; B rows (gate/up: two maps; down: one map, two boxes)
    int T, K, N;                           // N: h features (gate/up) or d (down)
    uint16_t* out;                         // gate/up: h [T, N]; down: out [T, N] (read and written)
    int32_t* status;
};

// kind::f16 instruction descriptor with bf16 A and B, f32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <int EPI, int NT>
__global__ void __launch_bounds__(kSThreads, 1) shared_kernel(const __grid_constant__ SharedArgs a) {
    constexpr int kSB = SGeo<NT>::kSB, kSStage = SGeo<NT>::kStage;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bar_full[SS], bar_done[SS], bar_acc;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    grid_dep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SS; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_done[s]), 1);
        }
        mbar_init(smem_u32(&bar_acc), 1);
        s_abort = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), NT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;
    const int nk = a.K / SKS;
    constexpr int kCols = EPI == SH_SWIGLU ? NT / 2 : NT;  // output columns per tile
    const int n_tiles = a.N / kCols;
    const int t0 = (blockIdx.x / n_tiles) * SM_;  // tiles of one token block are adjacent (A stays in L2)
    const int c0 = (blockIdx.x % n_tiles) * kCols;

    if (warp == 0) {
        // ---------------- MMA: warp-uniform loop, one elected lane issues ----------------
        int s = 0;
        uint32_t par = 0;
        for (int kc = 0; kc < nk; ++kc) {
            if (!warp_wait(smem_u32(&bar_full[s]), par, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * kSStage), sb = sa + kSA;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < SKS / 16; ++kk)
                    mma_f16(tmem, sdesc_sw128(sa) + 2 * kk, sdesc_sw128(sb) + 2 * kk, idesc_bf16(SM_, NT),
                            (kc | kk) != 0);
                mma_commit(smem_u32(&bar_done[s]));
            }
            __syncwarp();
            if (++s == SS) {
                s = 0;
                par ^= 1;
            }
        }
        if (elect_one()) mma_commit(smem_u32(&bar_acc));
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- operands by TMA (one thread) ----------------
        if (lane == 0) {
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % SS;
                if (kc >= SS &&
                    !mbar_wait(smem_u32(&bar_done[s]), (uint32_t)(((kc - SS) / SS) & 1), abort_flag, a.status))
                    break;
                const uint32_t bar = smem_u32(&bar_full[s]);
                const uint32_t dst = smem_u32(smem + s * kSStage);
                mbar_arrive_expect_tx(bar, (uint32_t)kSStage);
                tma_load_2d(dst, &a.tmap_a, kc * (SKS * 2), t0, bar);
                if (EPI == SH_SWIGLU) {
                    tma_load_2d(dst + kSA, &a.tmap_b0, kc * (SKS * 2), c0, bar);
                    tma_load_2d(dst + kSA + kSB / 2, &a.tmap_b1, kc * (SKS * 2), c0, bar);
                } else {
                    tma_load_2d(dst + kSA, &a.tmap_b0, kc * (SKS * 2), c0, bar);
                    tma_load_2d(dst + kSA + kSB / 2, &a.tmap_b0, kc * (SKS * 2), c0 + NT / 2, bar);
                }
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------- epilogue: one token per TMEM lane ----------------
        const int q = warp - 4;
        const int row = t0 + q * 32 + lane;
        if (warp_wait(smem_u32(&bar_acc), 0, abort_flag, a.status, 64)) {
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16);
            if constexpr (EPI == SH_SWIGLU) {
                for (int cb = 0; cb < NT / 2; cb += 16) {
                    uint32_t g[16], u[16];
                    tmem_ld16(tb + cb, g);
                    tmem_ld16(tb + NT / 2 + cb, u);
                    tmem_ld_wait();
                    if (row < a.T) {
                        uint32_t packed[8];
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            float hv[2];
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                const float G = round_bf16(__uint_as_float(g[j + t]));
                                const float U = round_bf16(__uint_as_float(u[j + t]));
                                hv[t] = G / (1.0f + expf(-G)) * U;
                            }
                            packed[j / 2] =
                                (uint32_t)f32_to_bf16_bits(hv[0]) | ((uint32_t)f32_to_bf16_bits(hv[1]) << 16);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(a.out + (size_t)row * a.N + c0 + cb);
                        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                    }
                }
            } else {
                for (int cb = 0; cb < NT; cb += 32) {
                    uint32_t r[32];
                    tmem_ld32(tb + cb, r);
                    tmem_ld_wait();
                    if (row < a.T) {
                        uint4* p = reinterpret_cast<uint4*>(a.out + (size_t)row * a.N + c0 + cb);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const uint4 o = p[v];
                            const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
                            uint32_t nw[4];
#pragma unroll
                            for (int w2 = 0; w2 < 4; ++w2) {
                                const float lo = bf16_bits_to_f32(ow[w2] & 0xFFFFu) + __uint_as_float(r[8 * v + 2 * w2]);
                                const float hi = bf16_bits_to_f32(ow[w2] >> 16) + __uint_as_float(r[8 * v + 2 * w2 + 1]);
                                nw[w2] = (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hi) << 16);
                            }
                            p[v] = make_uint4(nw[0], nw[1], nw[2], nw[3]);
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, NT);
    }
    grid_dep_launch();
}

template <int EPI, int NT>
nvfp4_status launch_shared(const SharedArgs& a, cudaStream_t s, const char* name) {
    auto kern = shared_kernel<EPI, NT>;
    constexpr int smem = SGeo<NT>::kSmem;
    static bool init = false;
    if (!init) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        init = true;
    }
    constexpr int kCols = EPI == SH_SWIGLU ? NT / 2 : NT;
    const int grid = ((a.T + SM_ - 1) / SM_) * (a.N / kCols);
    NVFP4_LAUNCH(name, s, launch_pdl(kern, dim3(grid), dim3(kSThreads), (size_t)smem, s, a));
    return last_launch_status();
}

}  // namespace

}  // namespace nvfp4

using namespace nvfp4;

extern "C" size_t moe_shared_expert_workspace_size(int T, int Fs) {
    if (T < 0 || Fs < 1) return 0;
    return align_up((size_t)T * Fs * 2, 256);
}

extern "C" nvfp4_status moe_shared_expert(const uint16_t* x_bf16, int T, int d, const uint16_t* w_gate_bf16,
                                          const uint16_t* w_up_bf16, const uint16_t* w_down_bf16, int Fs,
                                          uint16_t* out_bf16, void* ws, size_t ws_bytes, int32_t* d_status,
                                          cudaStream_t stream) {
    if (T < 0 || d < 1 || Fs < 1) return NVFP4_ERR_INVALID_ARG;
    if (d % SN != 0 || Fs % (SN / 2) != 0) return NVFP4_ERR_SHAPE;
    if (T == 0) return NVFP4_OK;
    if (!x_bf16 || !w_gate_bf16 || !w_up_bf16 || !w_down_bf16 || !out_bf16 || !ws) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(w_gate_bf16) || !aligned16(w_up_bf16) || !aligned16(w_down_bf16) ||
        !aligned16(out_bf16) || !aligned16(ws) || (d_status && !aligned16(d_status)))
        return NVFP4_ERR_ALIGN;
    if (ws_bytes < moe_shared_expert_workspace_size(T, Fs)) return NVFP4_ERR_WORKSPACE;
    uint16_t* h = static_cast<uint16_t*>(ws);
    // 64-wide tiles when the 256-wide down tiles would leave half the SMs idle
    const int m_tiles = (T + SM_ - 1) / SM_;
    const bool narrow = (long long)m_tiles * (d / SN) * 2 < num_sms();
    const unsigned bh = narrow ? 32 : SN / 2;  // B rows per TMA box
    // gate/up + SwiGLU -> h [T, Fs]
    SharedArgs g{};
    g.T = T;
    g.K = d;
    g.N = Fs;
    g.out = h;
    g.status = d_status;
    if (!encode_tmap_u8(&g.tmap_a, x_bf16, (unsigned long long)d * 2, (unsigned long long)T, SKS * 2, SM_, true) ||
        !encode_tmap_u8(&g.tmap_b0, w_gate_bf16, (unsigned long long)d * 2, (unsigned long long)Fs, SKS * 2, bh,
                        true) ||
        !encode_tmap_u8(&g.tmap_b1, w_up_bf16, (unsigned long long)d * 2, (unsigned long long)Fs, SKS * 2, bh, true))
        return NVFP4_ERR_CUDA;
    nvfp4_status st = narrow ? launch_shared<SH_SWIGLU, 64>(g, stream, "shared_gateup")
                             : launch_shared<SH_SWIGLU, SN>(g, stream, "shared_gateup");
    if (st != NVFP4_OK) return st;
    // down, added into the routed output
    SharedArgs u{};
    u.T = T;
    u.K = Fs;
    u.N = d;
    u.out = out_bf16;
    u.status = d_status;
    if (!encode_tmap_u8(&u.tmap_a, h, (unsigned long long)Fs * 2, (unsigned long long)T, SKS * 2, SM_, true) ||
        !encode_tmap_u8(&u.tmap_b0, w_down_bf16, (unsigned long long)Fs * 2, (unsigned long long)d, SKS * 2, bh, true))
        return NVFP4_ERR_CUDA;
    return narrow ? launch_shared<SH_ADD, 64>(u, stream, "shared_down") : launch_shared<SH_ADD, SN>(u, stream, "shared_down");
}
