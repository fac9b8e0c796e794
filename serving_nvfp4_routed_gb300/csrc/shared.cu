// shared.cu -- the BF16 shared-expert MLP after the weighted combine:
//   G = bf16(x Wg^T)   U = bf16(x Wu^T)   h = bf16(silu(G) * U)
//   out = bf16(out + h Wd^T)          (out holds the routed layer's result)
//
// TensorFold issue #308, "The checkpoint": the shared experts stay BF16 next
// to the NVFP4 routed experts; "What the branch does": the shared expert runs
// as a BF16 MLP.  It runs on every token, so it is two dense GEMMs.
//
// Both GEMMs run on tcgen05.mma kind::f16 with bf16 operands exactly as
// stored, moved by TMA (128-byte swizzle, k-stages of 64), an fp32
// accumulator in tensor memory; warp 0 runs the MMA loop (one elected lane
// issues), warp 1's lane 0 the TMA ring, warps 4-7 the epilogue.  mbarrier
// waits are bounded and report NVFP4_ERR_TIMEOUT.
//
// Wide tiles (a prompt batch): one CTA per (128 tokens, 256 output columns)
// tile, the tokens as the MMA's M and the weight rows as N (gate/up: B rows
// 0..127 = Wg rows f0.., 128..255 = Wu rows f0.., so a token's gate and up
// values for a feature share one TMEM lane and the SwiGLU is local to the
// thread); a ring of 4 stages.
//
// Narrow tiles (a decode batch, whose 256-wide tiles would leave most SMs
// idle): the weight rows are the MMA's M (128 rows: 64 gate + 64 up rows of
// 64 features, or 128 down rows) and up to 128 tokens its N, so that a
// stage carries 16 KB of weights next to the token rows and a deep ring
// keeps ~150 KB of weights in flight per SM.  K is split over a
// thread-block cluster of up to 8 CTAs (the widest split whose clusters are
// all resident at once); each CTA stores its fp32 partial tile in shared
// memory (over its drained ring) and, after a cluster barrier, the CTAs sum
// the partials in rank order through distributed shared memory, each for a
// slice of the tile's outputs (deterministic, no workspace).  The down
// launch issues its first weight stages before it waits for the gate/up
// launch (only the h rows depend on it).
#include "common.cuh"
#include "internal.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {

namespace {

using namespace tc;

constexpr int SM_ = 128;        // wide tiles: tokens per tile (MMA M); narrow tiles: weight rows (MMA M)
constexpr int SN = 256;         // wide tiles: output columns per tile (MMA N); shape rules refer to it
constexpr int SKS = 64;         // k per stage (128 bytes of bf16)
constexpr int kSA = SM_ * SKS * 2;   // 16 KB: the M-side operand of a stage
constexpr int kSB = SN * SKS * 2;    // 32 KB: the wide tiles' weight rows of a stage
constexpr int kWideStages = 4;
constexpr int kWideSmem = 1024 + kWideStages * (kSA + kSB);
constexpr int kSThreads = 256;
enum { SH_SWIGLU = 0, SH_ADD = 1 };

// Narrow tiles: ring stages of 16 KB of weights + NB token rows, as many as
// fit in kNarrowRing (at most kNarrowMaxStages); the fp32 partial tile
// [128][NB + 1] reuses the ring once the MMAs are done.
constexpr int kNarrowMaxStages = 12;
constexpr int kNarrowRing = 216 * 1024;
constexpr int kNarrowSmemMax = 1024 + kNarrowRing;
constexpr int kMaxClusterSplit = 8;
__host__ __device__ constexpr int narrow_stage_bytes(int nb) { return kSA + nb * SKS * 2; }

struct SharedArgs {
    CUtensorMap tmap_a, tmap_b0, tmap_b1;  // wide: A token rows, B weight rows (gate/up: two maps; down: one map,
                                           // two boxes); narrow: A weight rows (gate/up: gate, up; down: b0),
                                           // B token rows in tmap_a
    int T, K, N;                           // N: h features (gate/up) or d (down)
    int a_rows;                            // wide: rows of the token box (T rounded up to 8, at most 128; the
                                           // MMA's other rows hold stale data and are never stored)
    int nb;                                // narrow: tokens per tile (MMA N: 16, 32, 64 or 128)
    int t_tiles;                           // narrow: token tiles
    int ss;                                // narrow: ring stages
    int ksplit;                            // narrow: CTAs of a cluster splitting K (1: no cluster)
    uint16_t* out;                         // gate/up: h [T, N]; down: out [T, N] (read and written)
    int32_t* status;
};

// kind::f16 instruction descriptor with bf16 A and B, f32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// A bounded wait for a TMA copy still in flight when a CTA gives up, so that
// no copy lands in the shared memory of a later CTA.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try(bar, parity) && clock64() - t0 < kWaitCycles) {
    }
}

template <int EPI>
__global__ void __launch_bounds__(kSThreads, 1) shared_wide_kernel(const __grid_constant__ SharedArgs a) {
    constexpr int SS = kWideStages, NT = SN, kStage = kSA + kSB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bar_full[SS], bar_done[SS], bar_acc;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort, s_consumed, s_issued;

    grid_dep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SS; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_done[s]), 1);
        }
        mbar_init(smem_u32(&bar_acc), 1);
        s_abort = 0;
        s_consumed = 0;
        s_issued = 0;
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
        int s = 0, kc = 0;
        uint32_t par = 0;
        for (; kc < nk; ++kc) {
            if (!warp_wait(smem_u32(&bar_full[s]), par, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * kStage), sb = sa + kSA;
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
        if (lane == 0) s_consumed = kc;
        if (elect_one()) mma_commit(smem_u32(&bar_acc));
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- operands by TMA (one thread) ----------------
        if (lane == 0) {
            int kc = 0;
            for (; kc < nk; ++kc) {
                const int s = kc % SS;
                if (kc >= SS &&
                    !mbar_wait(smem_u32(&bar_done[s]), (uint32_t)(((kc - SS) / SS) & 1), abort_flag, a.status))
                    break;
                const uint32_t bar = smem_u32(&bar_full[s]);
                const uint32_t dst = smem_u32(smem + s * kStage);
                mbar_arrive_expect_tx(bar, (uint32_t)(a.a_rows * SKS * 2 + kSB));
                const int kx = kc * (SKS * 2);
                tma_load_2d(dst, &a.tmap_a, kx, t0, bar);
                if (EPI == SH_SWIGLU) {
                    tma_load_2d(dst + kSA, &a.tmap_b0, kx, c0, bar);
                    tma_load_2d(dst + kSA + kSB / 2, &a.tmap_b1, kx, c0, bar);
                } else {
                    tma_load_2d(dst + kSA, &a.tmap_b0, kx, c0, bar);
                    tma_load_2d(dst + kSA + kSB / 2, &a.tmap_b0, kx, c0 + NT / 2, bar);
                }
            }
            s_issued = kc;
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
    if (threadIdx.x == 32 && *abort_flag)  // copies still in flight land before the CTA leaves
        for (int kc = s_consumed; kc < s_issued; ++kc) drain_wait(smem_u32(&bar_full[kc % SS]), (uint32_t)((kc / SS) & 1));
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, NT);
    }
    grid_dep_launch();
}

template <int EPI>
__global__ void __launch_bounds__(kSThreads, 1) shared_narrow_kernel(const __grid_constant__ SharedArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bar_full[kNarrowMaxStages], bar_done[kNarrowMaxStages], bar_acc;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort, s_consumed, s_issued;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NB = a.nb, SS = a.ss, KS = a.ksplit;
    const int kStage = narrow_stage_bytes(NB);
    const uint32_t tcols = NB < 32 ? 32u : (uint32_t)NB;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SS; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_done[s]), 1);
        }
        mbar_init(smem_u32(&bar_acc), 1);
        s_abort = 0;
        s_consumed = 0;
        s_issued = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), tcols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;
    // the CTAs of one cluster (k slices) are adjacent, then the token tiles
    // of one weight tile (its rows stay in L2 for them)
    const int ks = blockIdx.x % KS, tile = blockIdx.x / KS;
    const int tt = tile % a.t_tiles, wt = tile / a.t_tiles;
    const int t0 = tt * NB;
    constexpr int kRows = EPI == SH_SWIGLU ? SM_ / 2 : SM_;  // output features per tile
    const int r0 = wt * kRows;                                // first output feature (= weight row of each map)
    const int nk_all = a.K / SKS;
    const int kc0 = ks * nk_all / KS, nk = (ks + 1) * nk_all / KS - kc0;  // this CTA's k-stages
    const uint32_t stage_tx = (uint32_t)kStage;                          // whole boxes (rows past T are zero-filled)

    if (warp == 0) {
        // ---------------- MMA: warp-uniform loop, one elected lane issues ----------------
        int s = 0, kc = 0;
        uint32_t par = 0;
        for (; kc < nk; ++kc) {
            if (!warp_wait(smem_u32(&bar_full[s]), par, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t sw = smem_u32(smem + s * kStage), sx = sw + kSA;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < SKS / 16; ++kk)
                    mma_f16(tmem, sdesc_sw128(sw) + 2 * kk, sdesc_sw128(sx) + 2 * kk, idesc_bf16(SM_, NB),
                            (kc | kk) != 0);
                mma_commit(smem_u32(&bar_done[s]));
            }
            __syncwarp();
            if (++s == SS) {
                s = 0;
                par ^= 1;
            }
        }
        if (lane == 0) s_consumed = kc;
        if (elect_one()) mma_commit(smem_u32(&bar_acc));
        __syncwarp();
        grid_dep_wait();  // (this warp reads no global memory before the output phase)
    } else if (warp == 1) {
        // ---------------- operands by TMA (one thread) ----------------
        if (lane != 0) grid_dep_wait();
        if (lane == 0) {
            auto load_w = [&](int kc) {
                const uint32_t bar = smem_u32(&bar_full[kc % SS]);
                const uint32_t dst = smem_u32(smem + (kc % SS) * kStage);
                const int kx = (kc0 + kc) * (SKS * 2);
                if (EPI == SH_SWIGLU) {
                    tma_load_2d(dst, &a.tmap_b0, kx, r0, bar);
                    tma_load_2d(dst + kSA / 2, &a.tmap_b1, kx, r0, bar);
                } else {
                    tma_load_2d(dst, &a.tmap_b0, kx, r0, bar);
                }
            };
            auto load_x = [&](int kc) {
                const uint32_t bar = smem_u32(&bar_full[kc % SS]);
                const uint32_t dst = smem_u32(smem + (kc % SS) * kStage) + kSA;
                tma_load_2d(dst, &a.tmap_a, (kc0 + kc) * (SKS * 2), t0, bar);
            };
            // the down launch: its first weight stages do not depend on the
            // gate/up launch, only the h rows do
            const int pre = EPI == SH_ADD ? min(SS, nk) : 0;
            for (int kc = 0; kc < pre; ++kc) {
                mbar_arrive_expect_tx(smem_u32(&bar_full[kc]), stage_tx);
                load_w(kc);
            }
            grid_dep_wait();
            for (int kc = 0; kc < pre; ++kc) load_x(kc);
            int kc = pre;
            for (; kc < nk; ++kc) {
                const int s = kc % SS;
                if (kc >= SS &&
                    !mbar_wait(smem_u32(&bar_done[s]), (uint32_t)(((kc - SS) / SS) & 1), abort_flag, a.status))
                    break;
                mbar_arrive_expect_tx(smem_u32(&bar_full[s]), stage_tx);
                load_w(kc);
                load_x(kc);
            }
            s_issued = kc;
        }
        __syncwarp();
    } else {
        grid_dep_wait();
    }

    // ---------------- the accumulator (or this CTA's partial) to shared memory ----------------
    // part[t][r], t = token of the tile, r = weight row (TMEM lane): a warp's
    // stores of one token are 32 consecutive floats; it reuses the ring,
    // whose copies the MMAs have all consumed
    float* part = reinterpret_cast<float*>(smem);
    if (warp >= 4) {
        const int q = warp - 4, r = q * 32 + lane;
        if (warp_wait(smem_u32(&bar_acc), 0, abort_flag, a.status, 64)) {
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16);
            for (int cb = 0; cb < NB; cb += 16) {
                uint32_t v[16];
                tmem_ld16(tb + cb, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) part[(cb + j) * SM_ + r] = __uint_as_float(v[j]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    grid_dep_launch();
    if (KS > 1) cluster_barrier();

    // ---------------- the tile's outputs: partials summed in rank order ----------------
    // unit u of the tile: token t = u / (kRows / 4), features 4 (u % (kRows /
    // 4)) .. +3 (consecutive threads, consecutive features of a token row:
    // 16-byte loads of the partials, 8-byte stores); CTA ks of the cluster
    // takes a contiguous slice of the units
    {
        constexpr int kUPT = kRows / 4;  // units per token
        const int vt = min(NB, a.T - t0), total = kUPT * vt;
        const int per = (total + KS - 1) / KS, u0 = ks * per, u1 = min(total, u0 + per);
        const uint32_t pl = smem_u32(part);
        auto ld_part = [&](int p, int t, int r) -> float4 {
            const uint32_t o = pl + (uint32_t)((t * SM_ + r) * 4);
            return KS > 1 ? ld_dsmem4(dsmem_addr(o, (uint32_t)p)) : *reinterpret_cast<const float4*>(part + t * SM_ + r);
        };
        constexpr int kBatch = 2;  // units per thread with all their loads in flight
        for (int ub = u0 + threadIdx.x; ub < u1; ub += kBatch * kSThreads) {
            float4 v0[kBatch][kMaxClusterSplit], v1[kBatch][kMaxClusterSplit];
            uint2 ov[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int u = ub + b * kSThreads;
                if (u < u1) {
                    const int t = u / kUPT, f = (u % kUPT) * 4;
#pragma unroll
                    for (int p = 0; p < kMaxClusterSplit; ++p)
                        if (p < KS) {
                            v0[b][p] = ld_part(p, t, f);
                            if (EPI == SH_SWIGLU) v1[b][p] = ld_part(p, t, kRows + f);
                        }
                    if (EPI == SH_ADD)
                        ov[b] = *reinterpret_cast<const uint2*>(a.out + (size_t)(t0 + t) * a.N + r0 + f);
                }
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int u = ub + b * kSThreads;
                if (u < u1) {
                    const int t = u / kUPT, f = (u % kUPT) * 4;
                    float4 y0 = make_float4(0.f, 0.f, 0.f, 0.f), y1 = y0;
#pragma unroll
                    for (int p = 0; p < kMaxClusterSplit; ++p)
                        if (p < KS) {
                            y0.x += v0[b][p].x;
                            y0.y += v0[b][p].y;
                            y0.z += v0[b][p].z;
                            y0.w += v0[b][p].w;
                            if (EPI == SH_SWIGLU) {
                                y1.x += v1[b][p].x;
                                y1.y += v1[b][p].y;
                                y1.z += v1[b][p].z;
                                y1.w += v1[b][p].w;
                            }
                        }
                    const float g4[4] = {y0.x, y0.y, y0.z, y0.w};
                    uint32_t hw[4];
                    if constexpr (EPI == SH_SWIGLU) {
                        const float u4[4] = {y1.x, y1.y, y1.z, y1.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float G = round_bf16(g4[j]), U = round_bf16(u4[j]);
                            hw[j] = f32_to_bf16_bits(G / (1.0f + expf(-G)) * U);
                        }
                    } else {
                        const uint32_t o2[2] = {ov[b].x, ov[b].y};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t ob = (o2[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
                            hw[j] = f32_to_bf16_bits(bf16_bits_to_f32(ob) + g4[j]);
                        }
                    }
                    *reinterpret_cast<uint2*>(a.out + (size_t)(t0 + t) * a.N + r0 + f) =
                        make_uint2(hw[0] | (hw[1] << 16), hw[2] | (hw[3] << 16));
                }
            }
        }
    }
    if (KS > 1) cluster_barrier();  // no CTA leaves while another still reads its partial
    if (threadIdx.x == 32 && *abort_flag)  // copies still in flight land before the CTA leaves
        for (int kc = s_consumed; kc < s_issued; ++kc) drain_wait(smem_u32(&bar_full[kc % SS]), (uint32_t)((kc / SS) & 1));
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, tcols);
    }
}

// Clusters of `ks` narrow CTAs with `smem` bytes of dynamic shared memory
// that can be resident at once (a cluster's CTAs share a GPC).
template <int EPI>
int max_active_clusters(int ks, int smem) {
    auto kern = shared_narrow_kernel<EPI>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kNarrowSmemMax);
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

nvfp4_status launch_cfg(void (*kern)(SharedArgs), int grid, int smem, int cluster, const SharedArgs& a,
                        cudaStream_t s, const char* name) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster;
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

template <int EPI>
nvfp4_status launch_wide(const SharedArgs& a, cudaStream_t s, const char* name) {
    static bool init = false;
    if (!init) {
        cudaFuncSetAttribute(shared_wide_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kWideSmem);
        init = true;
    }
    constexpr int kCols = EPI == SH_SWIGLU ? SN / 2 : SN;
    const int grid = ((a.T + SM_ - 1) / SM_) * (a.N / kCols);
    return launch_cfg(shared_wide_kernel<EPI>, grid, kWideSmem, 1, a, s, name);
}

template <int EPI>
nvfp4_status launch_narrow(const SharedArgs& a, cudaStream_t s, const char* name) {
    static bool init = false;
    if (!init) {
        cudaFuncSetAttribute(shared_narrow_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, kNarrowSmemMax);
        init = true;
    }
    const int smem = 1024 + a.ss * narrow_stage_bytes(a.nb);
    constexpr int kRows = EPI == SH_SWIGLU ? SM_ / 2 : SM_;
    const int grid = (a.N / kRows) * a.t_tiles * a.ksplit;
    return launch_cfg(shared_narrow_kernel<EPI>, grid, smem, a.ksplit, a, s, name);
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
    const int m_tiles = (T + SM_ - 1) / SM_;
    // narrow tiles when the 256-wide down tiles would leave half the SMs idle
    const bool narrow = (long long)m_tiles * (d / SN) * 2 < num_sms();
    if (!narrow) {
        SharedArgs g{};  // gate/up + SwiGLU -> h [T, Fs]
        g.T = T;
        g.K = d;
        g.N = Fs;
        g.out = h;
        g.status = d_status;
        g.a_rows = std::min(SM_, (T + 7) / 8 * 8);
        if (!encode_tmap_u8(&g.tmap_a, x_bf16, (unsigned long long)d * 2, (unsigned long long)T, SKS * 2, g.a_rows,
                            true) ||
            !encode_tmap_u8(&g.tmap_b0, w_gate_bf16, (unsigned long long)d * 2, (unsigned long long)Fs, SKS * 2,
                            SN / 2, true) ||
            !encode_tmap_u8(&g.tmap_b1, w_up_bf16, (unsigned long long)d * 2, (unsigned long long)Fs, SKS * 2,
                            SN / 2, true))
            return NVFP4_ERR_CUDA;
        nvfp4_status st = launch_wide<SH_SWIGLU>(g, stream, "shared_gateup");
        if (st != NVFP4_OK) return st;
        SharedArgs u{};  // down, added into the routed output
        u.T = T;
        u.K = Fs;
        u.N = d;
        u.out = out_bf16;
        u.status = d_status;
        u.a_rows = g.a_rows;
        if (!encode_tmap_u8(&u.tmap_a, h, (unsigned long long)Fs * 2, (unsigned long long)T, SKS * 2, u.a_rows,
                            true) ||
            !encode_tmap_u8(&u.tmap_b0, w_down_bf16, (unsigned long long)Fs * 2, (unsigned long long)d, SKS * 2,
                            SN / 2, true))
            return NVFP4_ERR_CUDA;
        return launch_wide<SH_ADD>(u, stream, "shared_down");
    }
    // narrow tiles: tokens per tile, ring depth, and K split over a cluster
    // -- the widest split whose clusters are all resident at once (one wave:
    // measured on GB300, a second wave of a few clusters doubles a launch's
    // time) and that leaves every CTA at least two k-stages
    const int nb = T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : SM_;
    const int nbi = nb == 16 ? 0 : nb == 32 ? 1 : nb == 64 ? 2 : 3;
    const int t_tiles = (T + nb - 1) / nb;
    const int ss = std::min(kNarrowMaxStages, kNarrowRing / narrow_stage_bytes(nb));
    const int smem = 1024 + ss * narrow_stage_bytes(nb);
    static int clusters[2][4][kMaxClusterSplit + 1] = {};
    auto pick_split = [&](long long tiles, int K, int epi) {
        int ks = 1;
        for (int c = 2; c <= kMaxClusterSplit; ++c) {
            if (K / SKS < 2 * c || tiles * c > num_sms()) continue;
            int& n = clusters[epi][nbi][c];
            if (n == 0)
                n = epi == SH_SWIGLU ? max_active_clusters<SH_SWIGLU>(c, smem) : max_active_clusters<SH_ADD>(c, smem);
            if (tiles <= n) ks = c;
        }
        return ks;
    };
    SharedArgs g{};  // gate/up + SwiGLU -> h [T, Fs]
    g.T = T;
    g.K = d;
    g.N = Fs;
    g.nb = nb;
    g.t_tiles = t_tiles;
    g.ss = ss;
    g.out = h;
    g.status = d_status;
    g.ksplit = pick_split((long long)(Fs / (SM_ / 2)) * t_tiles, d, SH_SWIGLU);
    if (!encode_tmap_u8(&g.tmap_a, x_bf16, (unsigned long long)d * 2, (unsigned long long)T, SKS * 2, nb, true) ||
        !encode_tmap_u8(&g.tmap_b0, w_gate_bf16, (unsigned long long)d * 2, (unsigned long long)Fs, SKS * 2, SM_ / 2,
                        true) ||
        !encode_tmap_u8(&g.tmap_b1, w_up_bf16, (unsigned long long)d * 2, (unsigned long long)Fs, SKS * 2, SM_ / 2,
                        true))
        return NVFP4_ERR_CUDA;
    nvfp4_status st = launch_narrow<SH_SWIGLU>(g, stream, "shared_gateup");
    if (st != NVFP4_OK) return st;
    SharedArgs u{};  // down, added into the routed output
    u.T = T;
    u.K = Fs;
    u.N = d;
    u.nb = nb;
    u.t_tiles = t_tiles;
    u.ss = ss;
    u.out = out_bf16;
    u.status = d_status;
    u.ksplit = pick_split((long long)(d / SM_) * t_tiles, Fs, SH_ADD);
    if (!encode_tmap_u8(&u.tmap_a, h, (unsigned long long)Fs * 2, (unsigned long long)T, SKS * 2, nb, true) ||
        !encode_tmap_u8(&u.tmap_b0, w_down_bf16, (unsigned long long)Fs * 2, (unsigned long long)d, SKS * 2, SM_,
                        true))
        return NVFP4_ERR_CUDA;
    return launch_narrow<SH_ADD>(u, stream, "shared_down");
}
