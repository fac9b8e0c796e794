// moe_tc.cu -- prompt-shaped grouped NVFP4 expert GEMM on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// TensorFold issue #308 "GLM-5.3-Flash on CUDA: read nvidia/GLM-5.3-Flash-NVFP4
// (ModelOpt NVFP4) as stored, W4A16": "What the branch does" (routed experts
// as one grouped kernel over bf16 rows, weight_scale_2 per expert; dense MLP
// with gate and up apart) and "Questions", item 4 (prompts get their own
// kernel, whose sums run in a different order from decode's).
//
// Work unit = (expert e, 128 output features f0.., 128 routed rows row0..):
//   D[f, j] = sum_k W[e, f, k] * B[row0 + j, k]         (swap-AB: weights are A)
// A: the NVFP4 weights.  Each of four producer warps owns 32 tile rows; a
//    thread streams its row's codes and scales through a private cp.async
//    ring in shared memory, dequantises e2m1*e4m3 -> f16 (exact) in
//    registers and writes the f16 row straight into tensor memory with
//    tcgen05.st -- the A operand never occupies shared memory, which keeps
//    shared-memory capacity and bandwidth for the B rows.
// B: f16 rows (x or h times a per-row power of two, exact for the inputs
//    here) gathered by cp.async into the 128-byte-swizzled K-major smem
//    layout.  Both operands flow through mbarrier-guarded stage rings.
// One thread issues tcgen05.mma kind::f16 (M=128, N=128, K=16, A from
// TMEM) into fp32 accumulators in TMEM; four epilogue warps (one TMEM lane
// quarter each) read them with tcgen05.ld and apply SwiGLU or store bf16
// rows (the routed layer's down projection: y by routed row, summed per
// token in slot order by a second kernel).
// Every mbarrier wait is bounded (about 2 s): on expiry the kernel records
// NVFP4_ERR_TIMEOUT in the status word, every role leaves its loop, and the
// CTA still frees its tensor memory before it exits.
#include "common.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {

namespace {

using namespace tc;

constexpr int BM = 128, BN = kTcTokTile, BK = 64;  // features, rows, K per stage
constexpr int kTileBytes = 128 * 128;                  // 128 rows x 64 f16
constexpr int kTcWarps = 12;
constexpr int kTcThreads = kTcWarps * 32;
// warp roles: 0 MMA issue, 1-2 B gather, 3 idle, 4-7 epilogue, 8-11 A dequant
constexpr int kWarpMma = 0, kWarpB = 1, kNumBWarps = 2, kWarpEpi = 4, kWarpDeq = 8;

// Tensor memory (512 columns x 128 lanes x 32 bit): the fp32 accumulators
// (NPROJ x BN columns per buffer) and a ring of f16 weight stages (A operand,
// NPROJ x 32 columns per stage: 64 K values of each of the 128 rows).
template <int NPROJ>
struct Cfg {
    static constexpr int kNAcc = NPROJ == 2 ? 1 : 2;      // accumulator buffers
    static constexpr int kSA = NPROJ == 2 ? 4 : 8;        // f16 weight stages in TMEM
    static constexpr int kAccCols = NPROJ * BN;
    static constexpr int kACols = NPROJ * (BK / 2);
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kNAcc * kAccCols + kSA * kACols <= 512, "TMEM budget");
    static constexpr int kSB = NPROJ == 2 ? 6 : 8;        // token-row stages in smem (gathered from L2)
    static constexpr int kRaw = NPROJ == 2 ? 10 : 12;     // weight-code stages in flight per thread
    static constexpr int kRawSlot = NPROJ * (2 * 128 * 16 + 128 * 4);
    static constexpr int kSmem = kSB * kTileBytes + kRaw * kRawSlot + 1024;
};

struct Unit {
    int e, row0, row_end, f0;
};

__device__ __forceinline__ Unit decode_unit(const TcArgs& a, int u, int n_active, int n_ft) {
    int lo = 0, hi = n_active;  // largest ai with tile_start[ai] * n_ft <= u
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a.tile_start[mid] * n_ft <= u) lo = mid; else hi = mid;
    }
    const int e = a.active[lo];
    const int ntt = a.tile_start[lo + 1] - a.tile_start[lo];
    const int local = u - a.tile_start[lo] * n_ft;
    Unit un;
    un.e = e;
    un.f0 = (local / ntt) * BM;
    un.row0 = a.offsets[e] + (local % ntt) * BN;
    un.row_end = a.offsets[e + 1];
    return un;
}

__device__ __forceinline__ int brow_of(const TcArgs& a, int row) {
    return a.b_by_token ? (a.row_to_slot ? a.row_to_slot[row] / a.top_k : row) : row;
}

template <int OUT, int NPROJ>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const TcArgs a) {
    using CF = Cfg<NPROJ>;
    constexpr int SA = CF::kSA, SB = CF::kSB, NACC = CF::kNAcc;
    constexpr int RD = CF::kRaw;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smem_b = smem;                              // [SB] f16 token-row tiles
    uint8_t* raw = smem_b + SB * kTileBytes;             // per-thread weight-code ring
    __shared__ __align__(8) uint64_t bar_full_a[SA], bar_empty_a[SA], bar_full_b[SB], bar_empty_b[SB];
    __shared__ __align__(8) uint64_t bar_acc_full[2], bar_acc_empty[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ int s_brow[BN];
    __shared__ float s_rs[2][BN];   // epilogue: 2^exp of the column's B row (0 if the column is empty)

    grid_dep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(smem_u32(&bar_full_a[s]), 4);  // one arrive per dequant warp (its 32 rows)
            mbar_init(smem_u32(&bar_empty_a[s]), 1);
        }
        for (int s = 0; s < SB; ++s) {
            mbar_init(smem_u32(&bar_full_b[s]), 32 * kNumBWarps);
            mbar_init(smem_u32(&bar_empty_b[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_acc_full[b]), 1);
            mbar_init(smem_u32(&bar_acc_empty[b]), 4);  // one arrive per epilogue warp
        }
        s_abort = 0;
        mbar_fence_init();
    }
    if (warp == kWarpMma) tmem_alloc(smem_u32(&s_tmem), CF::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t tmem_a = tmem + NACC * CF::kAccCols;  // first column of the weight stages
    volatile int* abort_flag = &s_abort;

    const int n_active = *a.n_active;
    const int n_ft = a.N / BM;
    const int total = a.tile_start[n_active] * n_ft;
    const int nk = a.K / BK;

    if (warp == kWarpMma) {
        // ---------------- MMA issue (one elected lane) ----------------
        const uint32_t idesc = idesc_f16_f32(BM, BN);
        int kcg = 0, it = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x, ++it) {
            const int as = it % NACC;
            if (!warp_wait(smem_u32(&bar_acc_empty[as]), ((it / NACC) & 1) ^ 1, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t d_base = tmem + as * CF::kAccCols;
            for (int kc = 0; kc < nk; ++kc, ++kcg) {
                const int sa = kcg % SA, sb = kcg % SB;
                if (!warp_wait(smem_u32(&bar_full_a[sa]), (kcg / SA) & 1, abort_flag, a.status) ||
                    !warp_wait(smem_u32(&bar_full_b[sb]), (kcg / SB) & 1, abort_flag, a.status))
                    goto mma_done;
                tc_fence_after();
                fence_proxy_async();
                if (lane == 0) {
                    const uint32_t a_stage = tmem_a + sa * CF::kACols;
                    const uint64_t bdesc = sdesc_sw128(smem_u32(smem_b + sb * kTileBytes));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
#pragma unroll
                        for (int p = 0; p < NPROJ; ++p)
                            mma_f16_ta(d_base + p * BN, a_stage + p * (BK / 2) + kk * 8, bdesc + 2 * kk, idesc,
                                       (kc | kk) != 0);
                    mma_commit(smem_u32(&bar_empty_a[sa]));
                    mma_commit(smem_u32(&bar_empty_b[sb]));
                }
                __syncwarp();
            }
            if (lane == 0) mma_commit(smem_u32(&bar_acc_full[as]));
            __syncwarp();
        }
    mma_done:;
    } else if (warp >= kWarpB && warp < kWarpB + kNumBWarps) {
        // ---------------- B producers: gathered f16 rows via cp.async ----------------
        const int wb = warp - kWarpB;  // rows wb*64 .. wb*64+63
        int kcg = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            const Unit un = decode_unit(a, u, n_active, n_ft);
            __syncwarp();
            for (int i = lane; i < BN / kNumBWarps; i += 32) {
                const int rr = wb * (BN / kNumBWarps) + i;
                const int row = un.row0 + rr;
                s_brow[rr] = row < un.row_end ? brow_of(a, row) : -1;
            }
            __syncwarp();
            for (int kc = 0; kc < nk; ++kc, ++kcg) {
                const int s = kcg % SB;
                if (!warp_wait(smem_u32(&bar_empty_b[s]), ((kcg / SB) & 1) ^ 1, abort_flag, a.status)) goto b_done;
                const uint32_t bt = smem_u32(smem_b + s * kTileBytes);
                const int c = lane & 7;
#pragma unroll
                for (int i = 0; i < BN / kNumBWarps / 4; ++i) {
                    const int rr = wb * (BN / kNumBWarps) + (lane >> 3) + 4 * i;
                    const int br = s_brow[rr];
                    const uint16_t* src = a.b_f16 + (size_t)(br < 0 ? 0 : br) * a.K + (size_t)kc * BK + c * 8;
                    cp_async16(bt + rr * 128 + ((c ^ (rr & 7)) << 4), src, br < 0 ? 0u : 16u);
                }
                cp_async_arrive_noinc(smem_u32(&bar_full_b[s]));
            }
        }
    b_done:;
    } else if (warp >= kWarpEpi && warp < kWarpEpi + 4) {
        // ---------------- epilogue: TMEM -> registers -> global ----------------
        const int q = warp - kWarpEpi;  // TMEM lane quarter
        const int et = q * 32 + lane;   // feature within the unit, and the column this thread describes
        int it = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x, ++it) {
            const Unit un = decode_unit(a, u, n_active, n_ft);
            const int as = it & 1;           // column-table buffer
            const int acc = it % NACC;       // accumulator buffer
            {   // per-column row data of this unit, one column per thread
                const int row = un.row0 + et;
                float rs = 0.0f;
                if (row < un.row_end) rs = exp2i(a.b_exp[brow_of(a, row)]);
                s_rs[as][et] = rs;
            }
            named_bar(1, 128);
            if (!warp_wait(smem_u32(&bar_acc_full[acc]), (it / NACC) & 1, abort_flag, a.status, 128)) break;
            tc_fence_after();
            const int f = un.f0 + et;
            const float w0 = a.a_ws2[0][un.e];
            const float w1 = a.a_ws2[NPROJ - 1][un.e];
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + acc * CF::kAccCols;
            const int ncol = min(BN, un.row_end - un.row0);
            for (int cb = 0; cb < BN / 32; ++cb) {
                if (cb * 32 >= ncol) break;  // warp-uniform
                uint32_t r0[32], r1[32];
                tmem_ld32(tb + cb * 32, r0);
                if constexpr (NPROJ == 2) tmem_ld32(tb + BN + cb * 32, r1);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int col = cb * 32 + j;
                    if (col >= ncol) continue;
                    const int row = un.row0 + col;
                    const float rs = s_rs[as][col];
                    if constexpr (OUT == TC_OUT_H) {
                        const float G = round_bf16(__fmul_rn(__fmul_rn(__uint_as_float(r0[j]), rs), w0));
                        const float U = round_bf16(__fmul_rn(__fmul_rn(__uint_as_float(r1[j]), rs), w1));
                        const float h = round_bf16(G / (1.0f + expf(-G)) * U);
                        a.h_out[(size_t)row * a.N + f] = f32_to_bf16_bits(h);
                    } else {
                        a.y_out[(size_t)row * a.N + f] =
                            f32_to_bf16_bits(__fmul_rn(__fmul_rn(__uint_as_float(r0[j]), rs), w0));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_acc_empty[acc]));
        }
    } else if (warp >= kWarpDeq) {
        // ---------------- A producer: NVFP4 weights -> f16 smem tiles ----------------
        // Each thread owns one tile row.  Its codes and scales stream through
        // a private ring of RD smem slots by cp.async (RD - 1 k-stages ahead),
        // then are dequantised into the shared f16 stage.
        const int dt = threadIdx.x - kWarpDeq * 32;  // tile row
        const int dwarp = warp - kWarpDeq;            // TMEM lane quarter of this warp
        const size_t K2 = (size_t)a.K / 2, K16 = (size_t)a.K / 16;
        auto raw_codes = [&](int slot, int p, int part) -> uint8_t* {
            return raw + slot * CF::kRawSlot + ((p * 2 + part) * 128 + dt) * 16;
        };
        auto raw_scale = [&](int slot, int p) -> uint8_t* {
            return raw + slot * CF::kRawSlot + NPROJ * 2 * 128 * 16 + (p * 128 + dt) * 4;
        };
        // issue side of the ring: walks this CTA's units and k-stages ahead of the consumer
        int iu = blockIdx.x, ikc = 0;
        const uint8_t* icp[NPROJ];
        const uint8_t* isp[NPROJ];
        auto set_issue_unit = [&]() {
            if (iu < total) {
                const Unit un = decode_unit(a, iu, n_active, n_ft);
                const size_t rowg = (size_t)un.e * a.N + un.f0 + dt;
#pragma unroll
                for (int p = 0; p < NPROJ; ++p) {
                    icp[p] = a.a_codes[p] + rowg * K2;
                    isp[p] = a.a_scales[p] + rowg * K16;
                }
            }
        };
        auto issue = [&](int slot) {
            if (iu < total) {
#pragma unroll
                for (int p = 0; p < NPROJ; ++p) {
                    const uint8_t* c = icp[p] + (size_t)ikc * 32;
                    cp_async16(smem_u32(raw_codes(slot, p, 0)), c, 16u);
                    cp_async16(smem_u32(raw_codes(slot, p, 1)), c + 16, 16u);
                    cp_async4(smem_u32(raw_scale(slot, p)), isp[p] + (size_t)ikc * 4);
                }
                if (++ikc == nk) {
                    ikc = 0;
                    iu += gridDim.x;
                    set_issue_unit();
                }
            }
            cp_async_commit();
        };
        set_issue_unit();
        for (int i = 0; i < RD - 1; ++i) issue(i);
        int kcg = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            for (int kc = 0; kc < nk; ++kc, ++kcg) {
                issue((kcg + RD - 1) % RD);
                cp_async_wait<RD - 1>();
                const int s = kcg % SA;
                if (!warp_wait(smem_u32(&bar_empty_a[s]), ((kcg / SA) & 1) ^ 1, abort_flag, a.status)) goto deq_done;
                tc_fence_after();
                const int slot = kcg % RD;
                // TMEM lane = this thread's tile row; 32 columns per projection
                const uint32_t ta = tmem_a + ((uint32_t)(dwarp * 32) << 16) + s * CF::kACols;
#pragma unroll
                for (int p = 0; p < NPROJ; ++p) {
                    const uint4 c0 = *reinterpret_cast<const uint4*>(raw_codes(slot, p, 0));
                    const uint4 c1 = *reinterpret_cast<const uint4*>(raw_codes(slot, p, 1));
                    const uint32_t sw = *reinterpret_cast<const uint32_t*>(raw_scale(slot, p));
                    const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    const uint32_t S01 = e4m3x2_to_f16x2(sw & 0xFFFFu), S23 = e4m3x2_to_f16x2(sw >> 16);
                    const uint32_t Sb[4] = {f16x2_bcast(S01, 0), f16x2_bcast(S01, 1), f16x2_bcast(S23, 0),
                                            f16x2_bcast(S23, 1)};
                    uint32_t v[32];
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        uint32_t f[4];
                        e2m1x8_to_f16x8(cw[w], f);
                        const uint32_t S2 = Sb[w >> 1];
#pragma unroll
                        for (int i = 0; i < 4; ++i) v[4 * w + i] = hmul2_u32(f[i], S2);
                    }
                    tmem_st32(ta + p * (BK / 2), v);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bar_full_a[s]));
            }
        }
    deq_done:
        cp_async_wait<0>();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, CF::kTmemCols);
    }
    grid_dep_launch();
}

template <int OUT, int NPROJ>
void launch_tc_t(const TcArgs& a, int max_units, cudaStream_t s, const char* name) {
    auto kern = tc_gemm_kernel<OUT, NPROJ>;
    static bool init = false;
    if (!init) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<NPROJ>::kSmem);
        init = true;
    }
    const int grid = std::max(1, std::min(max_units, num_sms()));
    NVFP4_LAUNCH(name, s, launch_pdl(kern, dim3(grid), dim3(kTcThreads), (size_t)Cfg<NPROJ>::kSmem, s, a));
}

// ---------------------------------------------------------------------------
// bf16 rows -> f16 rows times 2^-s(row), s from the row's max |v| so that the
// row max lands in [2^14, 2^15); exp[row] = s.  Optionally zeroes a float
// row of the same index (the combine accumulator).
// ---------------------------------------------------------------------------
__global__ void rows_to_f16_kernel(const uint16_t* __restrict__ src, int rows, int K, uint16_t* __restrict__ dst,
                                   int32_t* __restrict__ exps, float* __restrict__ zero_rows, int zero_len,
                                   const int32_t* __restrict__ map, int map_div, int zero_count) {
    grid_dep_wait();
    __shared__ float red[32];
    for (int r = blockIdx.x; r < rows; r += gridDim.x) {
        const int sr = map ? map[r] / map_div : r;
        const uint4* s4 = reinterpret_cast<const uint4*>(src + (size_t)sr * K);
        float m = 0.0f;
        for (int i = threadIdx.x; i < K / 8; i += blockDim.x) {
            const uint4 u = __ldg(s4 + i);
            const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_f32(ww[j] & 0xFFFFu)), fabsf(bf16_bits_to_f32(ww[j] >> 16))));
        }
        m = warp_max(m);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
        float v = (threadIdx.x & 31) < (blockDim.x >> 5) ? red[threadIdx.x & 31] : 0.0f;
        v = warp_max(v);
        const int sexp = row_exponent(v);
        const float down = exp2i(-sexp);
        if (threadIdx.x == 0) exps[r] = sexp;
        uint4* d4 = reinterpret_cast<uint4*>(dst + (size_t)r * K);
        for (int i = threadIdx.x; i < K / 8; i += blockDim.x) {
            const uint4 u = __ldg(s4 + i);
            uint4 o;
            o.x = f32x2_to_f16x2(bf16_bits_to_f32(u.x & 0xFFFFu) * down, bf16_bits_to_f32(u.x >> 16) * down);
            o.y = f32x2_to_f16x2(bf16_bits_to_f32(u.y & 0xFFFFu) * down, bf16_bits_to_f32(u.y >> 16) * down);
            o.z = f32x2_to_f16x2(bf16_bits_to_f32(u.z & 0xFFFFu) * down, bf16_bits_to_f32(u.z >> 16) * down);
            o.w = f32x2_to_f16x2(bf16_bits_to_f32(u.w & 0xFFFFu) * down, bf16_bits_to_f32(u.w >> 16) * down);
            d4[i] = o;
        }
        if (zero_rows && r < zero_count) {
            float4* z = reinterpret_cast<float4*>(zero_rows + (size_t)r * zero_len);
            for (int i = threadIdx.x; i < zero_len / 4; i += blockDim.x) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();
    }
    grid_dep_launch();
}

// One warp per row for K <= 32 * 8 * kRowRegs: the row stays in registers
// between its amax (a warp reduction) and its conversion, so it is read once
// and no block barrier is needed.
constexpr int kRowRegs = 16;  // 16-byte words per lane
constexpr int kRowWarps = 8;

__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float down) {
    return f32x2_to_f16x2(bf16_bits_to_f32(w & 0xFFFFu) * down, bf16_bits_to_f32(w >> 16) * down);
}

__global__ void __launch_bounds__(kRowWarps * 32) rows_to_f16_warp_kernel(
    const uint16_t* __restrict__ src, int rows, int K, uint16_t* __restrict__ dst, int32_t* __restrict__ exps,
    float* __restrict__ zero_rows, int zero_len, const int32_t* __restrict__ map, int map_div, int zero_count) {
    grid_dep_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = K / 8;  // 16-byte words per row
    for (int r = blockIdx.x * kRowWarps + warp; r < rows; r += gridDim.x * kRowWarps) {
        const int sr = map ? map[r] / map_div : r;
        const uint4* s4 = reinterpret_cast<const uint4*>(src + (size_t)sr * K);
        uint4 u[kRowRegs];
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < kRowRegs; ++j) {
            const int i = lane + 32 * j;
            if (i < nw) {
                u[j] = __ldg(s4 + i);
                const uint32_t ww[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_f32(ww[q] & 0xFFFFu)), fabsf(bf16_bits_to_f32(ww[q] >> 16))));
            }
        }
        m = warp_max(m);
        const int sexp = row_exponent(m);
        const float down = exp2i(-sexp);
        if (lane == 0) exps[r] = sexp;
        uint4* d4 = reinterpret_cast<uint4*>(dst + (size_t)r * K);
#pragma unroll
        for (int j = 0; j < kRowRegs; ++j) {
            const int i = lane + 32 * j;
            if (i < nw)
                d4[i] = make_uint4(bf16x2_to_f16x2_scaled(u[j].x, down), bf16x2_to_f16x2_scaled(u[j].y, down),
                                   bf16x2_to_f16x2_scaled(u[j].z, down), bf16x2_to_f16x2_scaled(u[j].w, down));
        }
        if (zero_rows && r < zero_count) {
            float4* z = reinterpret_cast<float4*>(zero_rows + (size_t)r * zero_len);
            for (int i = lane; i < zero_len / 4; i += 32) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    grid_dep_launch();
}


}  // namespace

size_t tc_smem_bytes(int nproj) { return nproj == 2 ? Cfg<2>::kSmem : Cfg<1>::kSmem; }

void launch_tc_gemm(int outmode, int nproj, const TcArgs& a, int max_units, cudaStream_t s, bool routed_down) {
    if (outmode == TC_OUT_H && nproj == 2) return launch_tc_t<TC_OUT_H, 2>(a, max_units, s, "tc_gateup_w4a16");
    if (outmode == TC_OUT_BF16)
        return launch_tc_t<TC_OUT_BF16, 1>(a, max_units, s, routed_down ? "tc_down_w4a16" : "tc_linear_w4a16");
}

void launch_rows_to_f16(const uint16_t* src, int rows, int K, uint16_t* dst, int32_t* exps, float* zero_rows,
                        int zero_len, cudaStream_t s, const int32_t* map, int map_div, int zero_count) {
    if (rows <= 0) return;
    if (zero_count < 0) zero_count = rows;
    if (K <= 32 * 8 * kRowRegs) {
        const int grid = std::min((rows + kRowWarps - 1) / kRowWarps, num_sms() * 8);
        NVFP4_LAUNCH("rows_to_f16", s,
                     launch_pdl(rows_to_f16_warp_kernel, dim3(grid), dim3(kRowWarps * 32), 0, s, src, rows, K, dst,
                                exps, zero_rows, zero_len, map, map_div, zero_count));
        return;
    }
    const int grid = std::min(rows, num_sms() * 8);
    NVFP4_LAUNCH("rows_to_f16", s,
                 launch_pdl(rows_to_f16_kernel, dim3(grid), dim3(256), 0, s, src, rows, K, dst, exps, zero_rows,
                            zero_len, map, map_div, zero_count));
}


}  // namespace nvfp4
