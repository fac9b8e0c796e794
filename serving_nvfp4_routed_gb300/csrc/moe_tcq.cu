// moe_tcq.cu -- W4A4 prompt-shaped grouped GEMMs on the block-scaled FP4
// tensor cores: tcgen05.mma kind::mxf4nvf4 with e4m3 scales per 16 values
// (scale_vec::4X), both operands exactly as stored.
//
// W4A4 model card "GLM-5.3-Flash-NVFP4-W4A4-Experts", "Quantization
// boundary" (routed experts quantise their inputs with a static per-expert
// input_scale to the checkpoint's e2m1 + e4m3 format) and TensorFold issue
// #308, "The checkpoint" (weights: e2m1 codes, e4m3 scale per 16 inputs,
// fp32 weight_scale_2).  Each product of an e2m1 code pair and its two block
// scales is exact; the MMA sums them in fp32 and the epilogue applies the
// two fp32 tensor scales, as for the f16 kernels.
//
// Unit = (expert e, 192 B rows, 128 routed rows of e):
//   D[j, n] = sum_k X[row0 + j, k] * B[n, k]
//   SwiGLU: B rows 0..95 = gate rows f0.., 96..191 = up rows f0..;
//   down: B rows = 192 consecutive rows f0.. of the down projection (the
//   last unit of a row tile may reach past the expert's rows: those columns
//   are computed and dropped); the epilogue writes bf16 rows y by routed row
//   (staged through shared memory, two 64-byte row segments per store) and a
//   second kernel adds each token's slots, weighted, in slot order.
// One MMA has M = 128, N = 192, K = 64 (96 cycles at the full FP4 rate).
// N = 192 rather than 128: a single issuing warp spends ~100 cycles per MMA
// on issue, barrier and commit work, which a 64-cycle N = 128 MMA cannot
// hide (measured on GB300: 2-3x slower than the FP4 rate), while two N = 256
// accumulators would leave no tensor memory for the scales.
// A k-stage covers K = 256: the rows' codes (128 bytes per row, 128-byte
// swizzle) and e4m3 scales (16 bytes per row) of A and B arrive by TMA into
// one smem slot of a ring of S.  Two groups of four scale warps (alternate
// k-stages) copy the stage's scales into one of three tensor-memory scale
// slots, where the MMA reads them:
//   A scales of row m, MMA j: lane m, column 4j + m/32 of the slot's area;
//   B scales of row n, MMA j: lanes n%32 (every lane quarter), column
//   16 + 6j + n/32.
// Every scale address the MMA takes and every multi-column tcgen05.st here
// starts on a multiple of 4 columns (B scales: of 2): a layout packing the A
// scales at column j + m/32 (4-column stores at odd columns, MMA scale
// addresses at odd columns) stopped with "misaligned address" on GB300.
// Each 32-bit TMEM word holds the four block scales of one row and one MMA
// (bytes = blocks in k order), which is the stored order of the scales.
// One warp runs the MMA loop (one elected lane issues) into two 192-column
// fp32 accumulators; eight epilogue warps read them (one routed row and half
// the columns per thread).  mbarrier waits are bounded (about 2 s) and
// report NVFP4_ERR_TIMEOUT.
#include "common.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {

namespace {

using namespace tc;

constexpr int BM = 128, BN = 192;
constexpr int BH = BN / 2;                 // B rows per TMA box (gate or up half)
constexpr int KS = 256;                    // k per stage
constexpr int S = 4;                       // stage ring depth (even: each slot has one scale group)
constexpr int kA = BM * KS / 2;            // 16 KB codes
constexpr int kB = BN * KS / 2;            // 24 KB codes
constexpr int kSA = BM * KS / 16;          // 2 KB scales
constexpr int kSB = BN * KS / 16;          // 3 KB scales
constexpr int kStage = kA + kB + kSA + kSB;  // 45 KB
static_assert(kStage % 1024 == 0 && (kB / 2) % 1024 == 0, "stage slots and B halves keep 1024-byte alignment");
constexpr int kMaxUnits = 320;
constexpr int kTileCopy = kMaxExperts + 1;
constexpr int kStageRow = 33;               // epilogue staging: 32 rows x 32 floats, padded
constexpr int kSmem = 1024 + S * kStage + kMaxUnits * 16 + kTileCopy * 4 + 8 * 32 * kStageRow * 4;
constexpr int kWarps = 20;
constexpr int kThreads = kWarps * 32;
constexpr int kWarpMma = 0, kWarpTma = 1, kWarpEpi = 4, kWarpSf = 8, kSfGroups = 2, kWarpEpi2 = 16;
static_assert(S % kSfGroups == 0, "each stage slot belongs to one scale group");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol0 = 2 * BN;       // scale slots after the two accumulators
constexpr int kSfSlots = 3;                // tensor-memory scale slots (stage i uses slot i % 3)
constexpr uint32_t kSfB = 16;              // B scales after A's 4 MMAs x 4 columns
constexpr uint32_t kSfBPerMma = BN / 32;   // 6 columns of B scales per MMA
constexpr uint32_t kSfCols = kSfB + 4 * kSfBPerMma;  // 40 columns per slot
static_assert(kSfCol0 + kSfSlots * kSfCols <= kTmemCols, "tensor memory budget");
static_assert(kSmem <= 227 * 1024, "shared memory budget");

// Instruction descriptor, kind::mxf4nvf4: A and B e2m1 (format 1, bits 7-9
// and 10-12), K-major, N >> 3 in bits 17-22, scale type ue4m3 (bit 23 = 0),
// M >> 4 in bits 24-28; scale-factor selectors 0.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_fp4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t sfa, uint32_t sfb,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %5, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %6, [%3], [%4], p;\n}" ::"r"(
            d),
        "l"(adesc), "l"(bdesc), "r"(sfa), "r"(sfb), "r"(accumulate), "n"(kIdesc)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ bool wait_done(const uint64_t* done, long long j, volatile int* abort_flag,
                                          int32_t* status) {
    if (j < 0) return true;
    return mbar_wait(smem_u32(&done[j % S]), (uint32_t)((j / S) & 1), abort_flag, status);
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1) tcq_kernel(const __grid_constant__ TcmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int4* s_units = reinterpret_cast<int4*>(smem + S * kStage);  // {e, row0, row_end, f0}
    int* s_tiles = reinterpret_cast<int*>(s_units + kMaxUnits);
    float* s_stage = reinterpret_cast<float*>(s_tiles + kTileCopy);  // [8 warps][32][kStageRow]
    __shared__ __align__(8) uint64_t bar_full[S], bar_sf[S], bar_done[S], bar_acc_full[2], bar_acc_empty[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    grid_dep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_sf[s]), 4);
            mbar_init(smem_u32(&bar_done[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_acc_full[b]), 1);
            mbar_init(smem_u32(&bar_acc_empty[b]), 8);
        }
        s_abort = 0;
        mbar_fence_init();
    }
    if (warp == kWarpMma) tmem_alloc(smem_u32(&s_tmem), kTmemCols);

    // ---- this CTA's work list ----
    constexpr bool kPair = EPI == TCM_SWIGLU_Q;
    constexpr int kSlice = kPair ? BN / 2 : BN;  // output features per unit
    const int n_active = *a.n_active;
    const int n_nt = (a.N + kSlice - 1) / kSlice;
    for (int i = threadIdx.x; i <= n_active; i += kThreads) s_tiles[i] = a.tile_start[i];
    __syncthreads();
    const int total = s_tiles[n_active] * n_nt;
    const int my_units = blockIdx.x < total ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    for (int t = threadIdx.x; t < my_units && t < kMaxUnits; t += kThreads) {
        const int u = blockIdx.x + t * gridDim.x;
        int lo = 0, hi = n_active;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_tiles[mid] * n_nt <= u) lo = mid; else hi = mid;
        }
        const int e = a.active[lo];
        const int ntt = s_tiles[lo + 1] - s_tiles[lo];
        const int local = u - s_tiles[lo] * n_nt;
        s_units[t] = make_int4(e, a.offsets[e] + (local % ntt) * BM, a.offsets[e + 1], (local / ntt) * kSlice);
    }
    if (threadIdx.x == 0 && my_units > kMaxUnits) {
        s_abort = 1;
        if (a.status) atomicExch(a.status, (int)NVFP4_ERR_SHAPE);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;
    const int n_units = *abort_flag ? 0 : my_units;
    const int nk = a.K / KS;

    if (warp == kWarpMma) {
        // ---------------- MMA issue: the warp runs the loop, one lane issues ----------------
        // The scale warps arrive on bar_sf[s] only after the slot's TMA bytes
        // landed (they wait on bar_full[s]), so one wait per stage covers both.
        const uint32_t smem0 = smem_u32(smem);
        int s = 0, t = 0;
        uint32_t par = 0;
        for (int it = 0; it < n_units; ++it) {
            const int acc = it & 1;
            if (!warp_wait(smem_u32(&bar_acc_empty[acc]), ((it >> 1) & 1) ^ 1, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t d = tmem + acc * BN;
            bool ok = true;
            for (int kc = 0; kc < nk; ++kc) {
                if (!warp_wait(smem_u32(&bar_sf[s]), par, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = smem0 + s * kStage;
                const uint64_t adesc = sdesc_sw128(sa), bdesc = sdesc_sw128(sa + kA);
                const uint32_t sf = tmem + kSfCol0 + t * kSfCols;
                if (elect_one()) {
#pragma unroll
                    for (int j = 0; j < KS / 64; ++j)
                        mma_fp4(d, adesc + 2 * j, bdesc + 2 * j, sf + 4 * j, sf + kSfB + kSfBPerMma * j, (kc | j) != 0);
                    mma_commit(smem_u32(&bar_done[s]));
                }
                __syncwarp();
                if (++s == S) {
                    s = 0;
                    par ^= 1;
                }
                if (++t == kSfSlots) t = 0;
            }
            if (!ok) break;
            if (elect_one()) mma_commit(smem_u32(&bar_acc_full[acc]));
            __syncwarp();
        }
    } else if (warp == kWarpTma) {
        // ---------------- operands by TMA (one thread) ----------------
        if (lane == 0) {
            const void* mc1 = kPair ? (const void*)&a.tmap_wc[1] : (const void*)&a.tmap_wc[0];
            const void* ms1 = kPair ? (const void*)&a.tmap_ws[1] : (const void*)&a.tmap_ws[0];
            long long i = 0;
            bool ok = true;
            for (int it = 0; it < n_units && ok; ++it) {
                const int4 un = s_units[it];
                const int y0 = un.x * a.N + un.w;
                const int y1 = kPair ? y0 : y0 + BH;
                for (int kc = 0; kc < nk; ++kc, ++i) {
                    if (!wait_done(bar_done, i - S, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    const int s = (int)(i % S);
                    const uint32_t bar = smem_u32(&bar_full[s]);
                    const uint32_t dst = smem_u32(smem + s * kStage);
                    mbar_arrive_expect_tx(bar, kStage);
                    tma_load_2d(dst, &a.tmap_ac, kc * (KS / 2), un.y, bar);
                    tma_load_2d(dst + kA, &a.tmap_wc[0], kc * (KS / 2), y0, bar);
                    tma_load_2d(dst + kA + kB / 2, mc1, kc * (KS / 2), y1, bar);
                    tma_load_2d(dst + kA + kB, &a.tmap_as, kc * (KS / 16), un.y, bar);
                    tma_load_2d(dst + kA + kB + kSA, &a.tmap_ws[0], kc * (KS / 16), y0, bar);
                    tma_load_2d(dst + kA + kB + kSA + kSB / 2, ms1, kc * (KS / 16), y1, bar);
                }
            }
        }
        __syncwarp();
    } else if (warp >= kWarpSf && warp < kWarpEpi2) {
        // ---------------- scales: smem -> tensor memory ----------------
        const int q = (warp - kWarpSf) & 3;  // lane quarter
        const int grp = (warp - kWarpSf) >> 2;  // takes the k-stages i = grp mod kSfGroups
        const int m = q * 32 + lane;           // A row of this thread
        const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
        long long i = 0;
        bool ok = true;
        for (int it = 0; it < n_units && ok; ++it) {
            for (int kc = 0; kc < nk; ++kc, ++i) {
                if ((int)(i % kSfGroups) != grp) continue;
                const int s = (int)(i % S);
                // the scale slot i % 3 was last read by the MMAs of stage i - 3
                if (!mbar_wait(smem_u32(&bar_full[s]), (uint32_t)((i / S) & 1), abort_flag, a.status) ||
                    !wait_done(bar_done, i - kSfSlots, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                const uint8_t* sc = smem + s * kStage + kA + kB;
                const uint4 va = *reinterpret_cast<const uint4*>(sc + m * 16);
                uint4 vb[BN / 32];
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) vb[c] = *reinterpret_cast<const uint4*>(sc + kSA + (c * 32 + lane) * 16);
                // the slot is refilled by TMA (async proxy) once these MMAs are done
                fence_proxy_async();
                uint32_t ra[16], rb[16], rb2[8];
                const uint32_t wa[4] = {va.x, va.y, va.z, va.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int c = 0; c < 4; ++c) ra[4 * j + c] = wa[j];  // column 4j + quarter holds this row's MMA-j scales
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
                        // column 6j + c holds row 32c + lane
                        const uint32_t wb[4] = {vb[c].x, vb[c].y, vb[c].z, vb[c].w};
                        const int k = (int)kSfBPerMma * j + c;
                        if (k < 16) rb[k] = wb[j]; else rb2[k - 16] = wb[j];
                    }
                const uint32_t col = kSfCol0 + (uint32_t)(i % kSfSlots) * kSfCols;
                tmem_st16(tq + col, ra);
                tmem_st16(tq + col + kSfB, rb);
                tmem_st8(tq + col + kSfB + 16, rb2);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bar_sf[s]));
            }
        }
    } else if ((warp >= kWarpEpi && warp < kWarpEpi + 4) || warp >= kWarpEpi2) {
        // ---------------- epilogue: one routed row per thread ----------------
        const int q = warp & 3;                // TMEM lane quarter
        const int half = warp >= kWarpEpi2;    // which half of the unit's columns
        const int rr = q * 32 + lane;
        for (int it = 0; it < n_units; ++it) {
            const int4 un = s_units[it];
            const int acc = it & 1;
            const int row = un.y + rr;
            const bool valid = row < un.z;
            const float rs = a.x_gs[un.x];
            const float w0 = a.a_ws2[0][un.x], w1 = a.a_ws2[1][un.x];
            if (!mbar_wait(smem_u32(&bar_acc_full[acc]), (it >> 1) & 1, abort_flag, a.status, 64)) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + acc * BN;
            if constexpr (EPI == TCM_SWIGLU_Q) {
                // h in 16-feature blocks, requantised to NVFP4 under hq_gs[e];
                // each half of the warps takes 3 of the unit's 6 blocks
                const float gs2 = a.hq_gs[un.x];
                for (int cb = 3 * half; cb < 3 * half + 3; ++cb) {
                    const int f = un.w + cb * 16;
                    if (f >= a.N) break;  // last unit of a row tile: features past ffn
                    uint32_t g[16], u[16];
                    tmem_ld16(tb + cb * 16, g);
                    tmem_ld16(tb + BH + cb * 16, u);
                    tmem_ld_wait();
                    if (valid) {
                        float hv[16];
                        float mx = 0.0f;
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            const float G = round_bf16(__fmul_rn(__fmul_rn(__uint_as_float(g[t]), rs), w0));
                            const float U = round_bf16(__fmul_rn(__fmul_rn(__uint_as_float(u[t]), rs), w1));
                            hv[t] = round_bf16(G / (1.0f + expf(-G)) * U);
                            mx = fmaxf(mx, fabsf(hv[t]));
                        }
                        uint32_t sbyte = 0, q0 = 0, q1 = 0;
                        if (gs2 > 0.0f) {
                            sbyte = f32_to_e4m3(__fdiv_rn(__fdiv_rn(mx, 6.0f), gs2));
                            const float Sv = e4m3_to_f32(sbyte);
                            if (Sv != 0.0f) {
                                const float den = __fmul_rn(Sv, gs2), rden = __frcp_rn(den);
#pragma unroll
                                for (int t = 0; t < 8; t += 2) {
                                    q0 |= e2m1x2_byte(e2m1_quotient(hv[t], den, rden),
                                                      e2m1_quotient(hv[t + 1], den, rden)) << (4 * t);
                                    q1 |= e2m1x2_byte(e2m1_quotient(hv[8 + t], den, rden),
                                                      e2m1_quotient(hv[9 + t], den, rden)) << (4 * t);
                                }
                            }
                        }
                        *reinterpret_cast<uint2*>(a.hq_out + (size_t)row * (a.N / 2) + f / 2) = make_uint2(q0, q1);
                        a.hs_out[(size_t)row * (a.N / 16) + f / 16] = (uint8_t)sbyte;
                    }
                }
            } else if constexpr (EPI == TCM_ROWS) {
                // 32 rows x 32 columns per warp and chunk: y (fp32) through shared
                // memory, then two bf16 rows (2 x 64 bytes) per store instruction
                float* st = s_stage + (size_t)(half * 4 + q) * 32 * kStageRow;
                const int nvalid = min(32, un.z - (un.y + q * 32));  // rows of this warp in the unit
                const int hr = lane >> 4, cl = (lane & 15) * 2;
                for (int cb = 3 * half; cb < 3 * half + 3; ++cb) {
                    if (un.w + cb * 32 >= a.N) break;  // columns past the expert's rows
                    uint32_t r[32];
                    tmem_ld32(tb + cb * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        st[lane * kStageRow + c] = __fmul_rn(__fmul_rn(__uint_as_float(r[c]), rs), w0);
                    __syncwarp();
                    uint16_t* ybase = a.y_rows + (size_t)(un.y + q * 32) * a.N + un.w + cb * 32 + cl;
                    for (int j = hr; j < nvalid; j += 2)
                        *reinterpret_cast<uint32_t*>(ybase + (size_t)j * a.N) =
                            (uint32_t)f32_to_bf16_bits(st[j * kStageRow + cl]) |
                            ((uint32_t)f32_to_bf16_bits(st[j * kStageRow + cl + 1]) << 16);
                    __syncwarp();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_acc_empty[acc]));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    grid_dep_launch();
}

// out[t][f] = bf16(sum_j w[t*k + j] * y[slot_to_row[t*k + j]][f]), the
// fp32 sum in slot order over bf16 y rows; 8 features per thread.  KT = k
// at compile time (0: any k): all of a token's row loads are then in flight
// together.
template <int KT>
__global__ void sum_rows_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ slot_to_row,
                                const float* __restrict__ topk_w, int T, int k_rt, int d, uint16_t* __restrict__ out) {
    grid_dep_wait();
    const int k = KT > 0 ? KT : k_rt;
    const int per_row = d / 8;
    const unsigned n = (unsigned)T * (unsigned)per_row;  // below 2^31: the launch splits T
    for (unsigned i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const size_t t = i / (unsigned)per_row, f = (i % (unsigned)per_row) * 8;
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
        auto add = [&](const uint4 p, float wj) {
            const uint32_t pw[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[2 * q] += wj * bf16_bits_to_f32(pw[q] & 0xFFFFu);
                acc[2 * q + 1] += wj * bf16_bits_to_f32(pw[q] >> 16);
            }
        };
        if constexpr (KT > 0) {
            uint4 p[KT];
            float wv[KT];
#pragma unroll
            for (int j = 0; j < KT; ++j) {
                const size_t r = (size_t)slot_to_row[t * KT + j];
                wv[j] = topk_w[t * KT + j];
                p[j] = __ldcs(reinterpret_cast<const uint4*>(y + r * d + f));
            }
#pragma unroll
            for (int j = 0; j < KT; ++j) add(p[j], wv[j]);
        } else {
            for (int j = 0; j < k; ++j) {
                const size_t r = (size_t)slot_to_row[t * k + j];
                add(__ldcs(reinterpret_cast<const uint4*>(y + r * d + f)), topk_w[t * k + j]);
            }
        }
        uint4 o;
        o.x = (uint32_t)f32_to_bf16_bits(acc[0]) | ((uint32_t)f32_to_bf16_bits(acc[1]) << 16);
        o.y = (uint32_t)f32_to_bf16_bits(acc[2]) | ((uint32_t)f32_to_bf16_bits(acc[3]) << 16);
        o.z = (uint32_t)f32_to_bf16_bits(acc[4]) | ((uint32_t)f32_to_bf16_bits(acc[5]) << 16);
        o.w = (uint32_t)f32_to_bf16_bits(acc[6]) | ((uint32_t)f32_to_bf16_bits(acc[7]) << 16);
        *reinterpret_cast<uint4*>(out + t * d + f) = o;
    }
    grid_dep_launch();
}

template <int EPI>
void launch_tcq_t(const TcmArgs& a, int max_units, cudaStream_t s, const char* name) {
    auto kern = tcq_kernel<EPI>;
    static bool init = false;
    if (!init) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        init = true;
    }
    int grid = std::max(1, std::min(max_units, num_sms()));
    grid = std::max(grid, (max_units + kMaxUnits - 1) / kMaxUnits);
    NVFP4_LAUNCH(name, s, launch_pdl(kern, dim3(grid), dim3(kThreads), (size_t)kSmem, s, a));
}

}  // namespace

bool tcq_supported(int epi, int N, int K) {
    return K % KS == 0 && N > 0 && (epi == TCM_SWIGLU_Q ? N % 16 == 0 : N % 32 == 0);
}

bool tcq_set_maps(TcmArgs* a, const uint8_t* x_codes, const uint8_t* x_scales, long long rows_x, long long rows_w) {
    const unsigned long long K = (unsigned long long)a->K;
    if (!encode_tmap_u8(&a->tmap_ac, x_codes, K / 2, rows_x, KS / 2, BM, true) ||
        !encode_tmap_u8(&a->tmap_as, x_scales, K / 16, rows_x, KS / 16, BM, false))
        return false;
    for (int p = 0; p < 2; ++p)
        if (!encode_tmap_u8(&a->tmap_wc[p], a->a_codes[p], K / 2, rows_w, KS / 2, BH, true) ||
            !encode_tmap_u8(&a->tmap_ws[p], a->a_scales[p], K / 16, rows_w, KS / 16, BH, false))
            return false;
    return true;
}

void launch_tcq(int epi, const TcmArgs& a, int max_tiles, cudaStream_t s) {
    const int slice = epi == TCM_SWIGLU_Q ? BH : BN;
    const int max_units = max_tiles * ((a.N + slice - 1) / slice);
    if (epi == TCM_SWIGLU_Q) return launch_tcq_t<TCM_SWIGLU_Q>(a, max_units, s, "tcq_gateup_w4a4");
    if (epi == TCM_ROWS) return launch_tcq_t<TCM_ROWS>(a, max_units, s, "tcq_down_w4a4");
}

void launch_sum_rows(const uint16_t* y, const int32_t* slot_to_row, const float* topk_w, int T, int k, int d,
                     uint16_t* out, cudaStream_t s) {
    if ((size_t)T * (d / 8) == 0) return;
    // the kernel indexes (token, 8 features) in 32 bits: tokens in chunks
    // of at most 2^31 such items
    const int chunk = (int)std::min<size_t>((size_t)T, ((size_t)1 << 31) / (size_t)(d / 8));
    for (int t0 = 0; t0 < T; t0 += chunk) {
        const int tc = std::min(chunk, T - t0);
        const size_t n = (size_t)tc * (d / 8);
        const int grid = (int)std::min<size_t>((n + 255) / 256, (size_t)num_sms() * 16);
        const int32_t* str = slot_to_row + (size_t)t0 * k;
        const float* tw = topk_w + (size_t)t0 * k;
        uint16_t* o = out + (size_t)t0 * d;
        if (k == 8) {
            NVFP4_LAUNCH("sum_rows", s,
                         launch_pdl(sum_rows_kernel<8>, dim3(grid), dim3(256), 0, s, y, str, tw, tc, k, d, o));
        } else {
            NVFP4_LAUNCH("sum_rows", s,
                         launch_pdl(sum_rows_kernel<0>, dim3(grid), dim3(256), 0, s, y, str, tw, tc, k, d, o));
        }
    }
}

}  // namespace nvfp4
