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
// the weights are then spread over 4x as many CTAs); when even that leaves
// SMs idle, K is split over a thread-block cluster of KS <= 8 CTAs, which
// store their fp32 partial tiles in shared memory and, after a cluster
// barrier, sum them in rank order through distributed shared memory, each
// CTA for a slice of the tile's rows (deterministic, no workspace);
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
constexpr int kSA = SM_ * SKS * 2;   // 16 KB
// Stage ring: 4 deep for the 256-wide tiles; 8 deep for the 64-wide ones
// (a decode batch), whose stages carry only 8 KB of weights next to the
// 16 KB row tile, so that enough weight bytes are in flight per SM.
template <int NT>
struct SGeo {
    static constexpr int kSB = NT * SKS * 2;
    static constexpr int kStage = kSA + kSB;
    static constexpr int SS = NT <= 64 ? 8 : 4;
    static constexpr int kPart = SM_ * (NT + 1) * 4;        // fp32 partial tile (split K), padded rows
    static constexpr int kSmem = 1024 + SS * kStage + (NT <= 64 ? kPart : 0);
};
constexpr int kMaxClusterSplit = 8;
constexpr int kSThreads = 256;
enum { SH_SWIGLU = 0, SH_ADD = 1 };

struct SharedArgs {
    CUtensorMap tmap_a, tmap_b0, tmap_b1;  // A rows; B rows (gate/up: two maps; down: one map, two boxes)
    int T, K, N;                           // N: h features (gate/up) or d (down)
    int ksplit;                            // CTAs of a cluster splitting K (1: no cluster)
    int a_rows;                            // rows of the A box: T rounded up to 8, at most 128
                                           // (the MMA's other rows hold stale data and are never stored)
    uint16_t* out;                         // gate/up: h [T, N]; down: out [T, N] (read and written)
    int32_t* status;
};

// kind::f16 instruction descriptor with bf16 A and B, f32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <int EPI, int NT>
__global__ void __launch_bounds__(kSThreads, 1) shared_kernel(const __grid_constant__ SharedArgs a) {
    constexpr int kSB = SGeo<NT>::kSB, kSStage = SGeo<NT>::kStage, SS = SGeo<NT>::SS;
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
    // CTAs of one cluster (k slices) are adjacent, then the tiles of one token block
    const int KS = a.ksplit;
    const int ks = blockIdx.x % KS, tile = blockIdx.x / KS;
    const int nk_all = a.K / SKS;
    const int kc0 = ks * nk_all / KS, nk = (ks + 1) * nk_all / KS - kc0;  // this CTA's k-stages
    constexpr int kCols = EPI == SH_SWIGLU ? NT / 2 : NT;  // output columns per tile
    const int n_tiles = a.N / kCols;
    const int t0 = (tile / n_tiles) * SM_;  // tiles of one token block are adjacent (A stays in L2)
    const int c0 = (tile % n_tiles) * kCols;
    float* part = reinterpret_cast<float*>(smem + SS * kSStage);  // [SM_][NT + 1] when KS > 1

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
                mbar_arrive_expect_tx(bar, (uint32_t)(a.a_rows * SKS * 2 + kSB));
                const int kx = (kc0 + kc) * (SKS * 2);
                tma_load_2d(dst, &a.tmap_a, kx, t0, bar);
                if (EPI == SH_SWIGLU) {
                    tma_load_2d(dst + kSA, &a.tmap_b0, kx, c0, bar);
                    tma_load_2d(dst + kSA + kSB / 2, &a.tmap_b1, kx, c0, bar);
                } else {
                    tma_load_2d(dst + kSA, &a.tmap_b0, kx, c0, bar);
                    tma_load_2d(dst + kSA + kSB / 2, &a.tmap_b0, kx, c0 + NT / 2, bar);
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
            if (NT <= 64 && KS > 1) {
                // the partial tile, one padded row per lane (no bank conflicts)
                for (int cb = 0; cb < NT; cb += 32) {
                    uint32_t r[32];
                    tmem_ld32(tb + cb, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) part[(q * 32 + lane) * (NT + 1) + cb + j] = __uint_as_float(r[j]);
                }
            } else if constexpr (EPI == SH_SWIGLU) {
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
    if (NT <= 64 && KS > 1) {
        // every CTA of the cluster gets here (no early exit); the partials are
        // summed in rank order, each CTA taking a slice of the tile's valid
        // rows; consecutive threads take consecutive columns of a row
        cluster_barrier();
        const int vr = min(SM_, a.T - t0), per = (vr + KS - 1) / KS;
        const int r0 = ks * per, r1 = min(vr, r0 + per);
        const uint32_t pl = smem_u32(part);
        constexpr int kOut = EPI == SH_SWIGLU ? NT / 2 : NT;
        for (int i = threadIdx.x; i < (r1 - r0) * kOut; i += kSThreads) {
            const int rr = r0 + i / kOut, j = i % kOut, row = t0 + rr;
            const uint32_t o0 = pl + (uint32_t)((rr * (NT + 1) + j) * 4);
            // every rank's value is loaded first (all in flight), then summed in rank order
            float v0[kMaxClusterSplit], v1[kMaxClusterSplit];
#pragma unroll
            for (int p = 0; p < kMaxClusterSplit; ++p)
                if (p < KS) {
                    v0[p] = ld_dsmem(dsmem_addr(o0, (uint32_t)p));
                    if (EPI == SH_SWIGLU) v1[p] = ld_dsmem(dsmem_addr(o0 + (uint32_t)(NT / 2 * 4), (uint32_t)p));
                }
            float y0 = 0.0f, y1 = 0.0f;
#pragma unroll
            for (int p = 0; p < kMaxClusterSplit; ++p)
                if (p < KS) {
                    y0 += v0[p];
                    if (EPI == SH_SWIGLU) y1 += v1[p];
                }
            if constexpr (EPI == SH_SWIGLU) {
                const float G = round_bf16(y0), U = round_bf16(y1);
                a.out[(size_t)row * a.N + c0 + j] = f32_to_bf16_bits(G / (1.0f + expf(-G)) * U);
            } else {
                uint16_t* o = a.out + (size_t)row * a.N + c0 + j;
                *o = f32_to_bf16_bits(bf16_bits_to_f32(*o) + y0);
            }
        }
        cluster_barrier();  // no CTA leaves while another still reads its partial
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, NT);
    }
    grid_dep_launch();
}

// Clusters of `ks` CTAs of this kernel that can be resident at once (the
// shared memory allows one CTA per SM; a cluster's CTAs share a GPC).
template <int EPI, int NT>
int max_active_clusters(int ks) {
    auto kern = shared_kernel<EPI, NT>;
    constexpr int smem = SGeo<NT>::kSmem;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ks * num_sms());
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = ks;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
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
    const int grid = ((a.T + SM_ - 1) / SM_) * (a.N / kCols) * a.ksplit;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (a.ksplit > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = a.ksplit;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl_enabled()) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    NVFP4_LAUNCH(name, s, cudaLaunchKernelEx(&cfg, kern, a));
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
    // narrow tiles: split K over a cluster, the widest split whose clusters
    // are all resident at once (one wave) and that leaves every CTA at least
    // two k-stages (measured on GB300: a second wave of a few clusters
    // doubles the launch's time)
    static int clusters_gu[kMaxClusterSplit + 1] = {}, clusters_dn[kMaxClusterSplit + 1] = {};
    auto pick_split = [&](long long ctas, int K, int* cache, bool gateup) {
        int ks = 1;
        if (!narrow) return ks;
        for (int c = 2; c <= kMaxClusterSplit; ++c) {
            if (K / SKS < 2 * c || ctas * c > num_sms()) continue;
            if (cache[c] == 0)
                cache[c] = gateup ? max_active_clusters<SH_SWIGLU, 64>(c) : max_active_clusters<SH_ADD, 64>(c);
            if (ctas <= cache[c]) ks = c;
        }
        return ks;
    };
    const unsigned bh = narrow ? 32 : SN / 2;  // B rows per TMA box
    // gate/up + SwiGLU -> h [T, Fs]
    SharedArgs g{};
    g.T = T;
    g.K = d;
    g.N = Fs;
    g.out = h;
    g.status = d_status;
    const int a_rows = std::min(SM_, (T + 7) / 8 * 8);
    g.a_rows = a_rows;
    g.ksplit = pick_split((long long)m_tiles * (Fs / 32), d, clusters_gu, true);
    if (!encode_tmap_u8(&g.tmap_a, x_bf16, (unsigned long long)d * 2, (unsigned long long)T, SKS * 2, a_rows, true) ||
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
    u.a_rows = a_rows;
    u.ksplit = pick_split((long long)m_tiles * (d / 64), Fs, clusters_dn, false);
    if (!encode_tmap_u8(&u.tmap_a, h, (unsigned long long)Fs * 2, (unsigned long long)T, SKS * 2, a_rows, true) ||
        !encode_tmap_u8(&u.tmap_b0, w_down_bf16, (unsigned long long)Fs * 2, (unsigned long long)d, SKS * 2, bh, true))
        return NVFP4_ERR_CUDA;
    return narrow ? launch_shared<SH_ADD, 64>(u, stream, "shared_down") : launch_shared<SH_ADD, SN>(u, stream, "shared_down");
}
