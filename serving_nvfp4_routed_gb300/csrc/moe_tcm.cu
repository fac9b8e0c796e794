// moe_tcm.cu -- prompt-shaped gate/up + SwiGLU with the routed rows as the
// MMA's M dimension and gate and up stacked as one N = 256 operand.
//
// TensorFold issue #308 "GLM-5.3-Flash on CUDA: read nvidia/GLM-5.3-Flash-NVFP4
// (ModelOpt NVFP4) as stored, W4A16": "What the branch does" (routed experts
// as one grouped kernel over bf16 rows, weight_scale_2 per expert) and
// "Questions", item 4 (prompts get their own kernel).
//
// Unit = (expert e, 128 features f0.., 128 routed rows row0.. of e):
//   D[j, n] = sum_k X[row0 + j, k] * Wn[k],  n < 128: gate row f0 + n,
//                                           n >= 128: up row f0 + n - 128
// One tcgen05.mma kind::f16 (M = 128, N = 256, K = 16) costs about the same
// as one with N = 128, so stacking gate and up in N halves the instruction
// count, and makes both halves of a SwiGLU pair land in the same TMEM lane.
// A (rows): f16 copies of x in expert order, one 128 x 64 tile per k-stage
//    by TMA (128-byte swizzle) -- one elected thread, async proxy.
// B (weights): eight producer warps, one weight row per thread, stream the
//    row's e2m1 codes and e4m3 scales through a register ring, dequantise to
//    f16 (exact) and store the row into the 128-byte-swizzled K-major tile.
// One thread issues the MMAs into fp32 accumulators in TMEM (two buffers of
// 256 columns); four epilogue warps read them (one row per thread: G in
// columns 0..127, U in 128..255) and write h = bf16(silu(bf16 G) * bf16 U).
// mbarrier waits are bounded (about 2 s) and report NVFP4_ERR_TIMEOUT.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {

namespace {

using namespace tc;

constexpr int BM = 128;           // routed rows per unit (MMA M)
constexpr int BF = 128;           // features per unit (gate + up = MMA N = 256)
constexpr int BN = 2 * BF;
constexpr int BK = 64;            // K per stage
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;  // 16 KB
constexpr int kBBytes = BN * BK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmem = kStages * kStageBytes + 1024;
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kWarpMma = 0, kWarpTma = 1, kWarpEpi = 4, kWarpDeq = 8, kDeqWarps = 8;
constexpr int kPD = 6;            // k-stages of weight codes in flight per dequant thread
constexpr uint32_t kTmemCols = 512;  // two 256-column accumulators

struct Unit {
    int e, row0, row_end, f0;
};

__device__ __forceinline__ Unit decode_unit(const TcmArgs& a, int u, int n_active, int n_ft) {
    int lo = 0, hi = n_active;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a.tile_start[mid] * n_ft <= u) lo = mid; else hi = mid;
    }
    const int e = a.active[lo];
    const int ntt = a.tile_start[lo + 1] - a.tile_start[lo];
    const int local = u - a.tile_start[lo] * n_ft;
    Unit un;
    un.e = e;
    un.f0 = (local / ntt) * BF;
    un.row0 = a.offsets[e] + (local % ntt) * BM;
    un.row_end = a.offsets[e + 1];
    return un;
}

__global__ void __launch_bounds__(kThreads, 1) tcm_gateup_kernel(const __grid_constant__ TcmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bar_full[kStages], bar_empty[kStages], bar_acc_full[2], bar_acc_empty[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    grid_dep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1 + kDeqWarps);  // TMA producer + one arrive per dequant warp
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_acc_full[b]), 1);
            mbar_init(smem_u32(&bar_acc_empty[b]), 4);
        }
        s_abort = 0;
        mbar_fence_init();
    }
    if (warp == kWarpMma) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;

    const int n_active = *a.n_active;
    const int n_ft = a.F / BF;
    const int total = a.tile_start[n_active] * n_ft;
    const int nk = a.K / BK;
    const int my_units = blockIdx.x < total ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const long long n_items = (long long)my_units * nk;  // (unit, k-stage) pairs of this CTA

    if (warp == kWarpMma) {
        // ---------------- MMA issue ----------------
        const uint32_t idesc = idesc_f16_f32(BM, BN);
        long long i = 0;
        for (int it = 0; it < my_units; ++it) {
            const int acc = it & 1;
            if (!warp_wait(smem_u32(&bar_acc_empty[acc]), ((it >> 1) & 1) ^ 1, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t d = tmem + acc * BN;
            for (int kc = 0; kc < nk; ++kc, ++i) {
                const int s = (int)(i % kStages);
                if (!warp_wait(smem_u32(&bar_full[s]), (uint32_t)((i / kStages) & 1), abort_flag, a.status))
                    goto mma_done;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sa = smem_u32(smem + s * kStageBytes);
                    const uint64_t adesc = sdesc_sw128(sa), bdesc = sdesc_sw128(sa + kABytes);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_f16(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kc | kk) != 0);
                    mma_commit(smem_u32(&bar_empty[s]));
                }
                __syncwarp();
            }
            if (lane == 0) mma_commit(smem_u32(&bar_acc_full[acc]));
            __syncwarp();
        }
    mma_done:;
    } else if (warp == kWarpTma) {
        // ---------------- A producer: routed rows by TMA ----------------
        long long i = 0;
        for (int it = 0; it < my_units; ++it) {
            const Unit un = decode_unit(a, blockIdx.x + it * gridDim.x, n_active, n_ft);
            for (int kc = 0; kc < nk; ++kc, ++i) {
                const int s = (int)(i % kStages);
                if (!warp_wait(smem_u32(&bar_empty[s]), (uint32_t)(((i / kStages) & 1) ^ 1), abort_flag, a.status))
                    goto tma_done;
                if (lane == 0) {
                    const uint32_t bar = smem_u32(&bar_full[s]);
                    mbar_arrive_expect_tx(bar, kABytes);
                    tma_load_2d(smem_u32(smem + s * kStageBytes), &a.tmap_x, kc * BK, un.row0, bar);
                }
                __syncwarp();
            }
        }
    tma_done:;
    } else if (warp >= kWarpEpi && warp < kWarpEpi + 4) {
        // ---------------- epilogue: one routed row per thread ----------------
        const int q = warp - kWarpEpi;
        const int rr = q * 32 + lane;  // row within the unit = TMEM lane
        for (int it = 0; it < my_units; ++it) {
            const Unit un = decode_unit(a, blockIdx.x + it * gridDim.x, n_active, n_ft);
            const int acc = it & 1;
            const int row = un.row0 + rr;
            const bool valid = row < un.row_end;
            const float rs = valid ? exp2i(a.x_exp[row]) : 0.0f;
            const float wg = a.a_ws2[0][un.e], wu = a.a_ws2[1][un.e];
            if (!warp_wait(smem_u32(&bar_acc_full[acc]), (it >> 1) & 1, abort_flag, a.status, 128)) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + acc * BN;
            for (int cb = 0; cb < BF / 32; ++cb) {
                uint32_t g[32], u[32];
                tmem_ld32(tb + cb * 32, g);
                tmem_ld32(tb + BF + cb * 32, u);
                tmem_ld_wait();
                if (valid) {
                    uint32_t packed[16];
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        float hv[2];
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const float G = round_bf16(__fmul_rn(__fmul_rn(__uint_as_float(g[j + t]), rs), wg));
                            const float U = round_bf16(__fmul_rn(__fmul_rn(__uint_as_float(u[j + t]), rs), wu));
                            hv[t] = G / (1.0f + expf(-G)) * U;
                        }
                        packed[j / 2] = (uint32_t)f32_to_bf16_bits(hv[0]) | ((uint32_t)f32_to_bf16_bits(hv[1]) << 16);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(a.h_out + (size_t)row * a.F + un.f0 + cb * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_acc_empty[acc]));
        }
    } else if (warp >= kWarpDeq) {
        // ---------------- B producer: NVFP4 weight rows -> f16 tile rows ----------------
        const int j = threadIdx.x - kWarpDeq * 32;  // B row: 0..127 gate, 128..255 up
        const int p = j / BF;
        const size_t K2 = (size_t)a.K / 2, K16 = (size_t)a.K / 16;
        // issue side of the register ring, kPD (unit, k-stage) items ahead
        int iu = 0, ikc = 0;
        const uint8_t* icp = nullptr;
        const uint8_t* isp = nullptr;
        auto set_unit = [&]() {
            if (iu < my_units) {
                const Unit un = decode_unit(a, blockIdx.x + iu * gridDim.x, n_active, n_ft);
                const size_t rowg = (size_t)un.e * a.F + un.f0 + (j % BF);
                icp = a.a_codes[p] + rowg * K2;
                isp = a.a_scales[p] + rowg * K16;
            }
        };
        uint32_t ring[kPD][9];
        auto issue = [&](uint32_t (&r)[9]) {
            if (iu < my_units) {
                const uint4 c0 = __ldg(reinterpret_cast<const uint4*>(icp + (size_t)ikc * 32));
                const uint4 c1 = __ldg(reinterpret_cast<const uint4*>(icp + (size_t)ikc * 32) + 1);
                r[0] = c0.x; r[1] = c0.y; r[2] = c0.z; r[3] = c0.w;
                r[4] = c1.x; r[5] = c1.y; r[6] = c1.z; r[7] = c1.w;
                r[8] = __ldg(reinterpret_cast<const uint32_t*>(isp + (size_t)ikc * 4));
                if (++ikc == nk) {
                    ikc = 0;
                    ++iu;
                    set_unit();
                }
            }
        };
        set_unit();
#pragma unroll
        for (int uu = 0; uu < kPD; ++uu) issue(ring[uu]);
        for (long long i0 = 0; i0 < n_items; i0 += kPD) {
#pragma unroll
            for (int uu = 0; uu < kPD; ++uu) {
                const long long i = i0 + uu;
                if (i >= n_items) break;
                const int s = (int)(i % kStages);
                if (!warp_wait(smem_u32(&bar_empty[s]), (uint32_t)(((i / kStages) & 1) ^ 1), abort_flag, a.status))
                    goto deq_done;
                uint8_t* rowp = smem + s * kStageBytes + kABytes + j * 128;
                const uint32_t sw = ring[uu][8];
                const uint32_t S01 = e4m3x2_to_f16x2(sw & 0xFFFFu), S23 = e4m3x2_to_f16x2(sw >> 16);
                const uint32_t Sb[4] = {f16x2_bcast(S01, 0), f16x2_bcast(S01, 1), f16x2_bcast(S23, 0),
                                        f16x2_bcast(S23, 1)};
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    uint32_t f[4];
                    e2m1x8_to_f16x8(ring[uu][w], f);
                    const uint32_t S2 = Sb[w >> 1];
                    *reinterpret_cast<uint4*>(rowp + ((w ^ (j & 7)) << 4)) =
                        make_uint4(hmul2_u32(f[0], S2), hmul2_u32(f[1], S2), hmul2_u32(f[2], S2), hmul2_u32(f[3], S2));
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bar_full[s]));
                issue(ring[uu]);
            }
        }
    deq_done:;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    grid_dep_launch();
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

}  // namespace

bool make_tmap_rows_f16(CUtensorMap* map, const void* base, int rows, int K) {
    std::call_once(g_encode_once, []() {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!g_encode) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {BK, BM};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void launch_tcm_gateup(const TcmArgs& a, int max_units, cudaStream_t s) {
    static bool init = false;
    if (!init) {
        cudaFuncSetAttribute(tcm_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        init = true;
    }
    const int grid = std::max(1, std::min(max_units, num_sms()));
    NVFP4_LAUNCH("tcm_gateup_w4a16", s,
                 launch_pdl(tcm_gateup_kernel, dim3(grid), dim3(kThreads), (size_t)kSmem, s, a));
}

}  // namespace nvfp4
