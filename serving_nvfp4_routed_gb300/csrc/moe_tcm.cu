// moe_tcm.cu -- prompt-shaped grouped NVFP4 expert GEMMs on the 5th-generation
// tensor cores with the routed rows as the MMA's M dimension.
//
// TensorFold issue #308 "GLM-5.3-Flash on CUDA: read nvidia/GLM-5.3-Flash-NVFP4
// (ModelOpt NVFP4) as stored, W4A16": "What the branch does" (routed experts
// as one grouped kernel over bf16 rows, weight_scale_2 per expert; dense MLP
// with gate and up apart) and "Questions", item 4 (prompts get their own
// kernel, whose sums run in a different order from decode's).
//
// Unit = (expert e, one 256-wide slice of B rows, 128 routed rows of e):
//   D[j, n] = sum_k X[row0 + j, k] * B[n, k]
//   SwiGLU: B rows 0..127 = gate rows f0.., 128..255 = up rows f0.. of e, so
//           the two halves of a SwiGLU pair sit in one TMEM lane;
//   down (bf16 y rows) / bf16: B rows = 256 consecutive rows f0.. of one projection.
// One tcgen05.mma kind::f16 with M = 128, N = 256, K = 16 runs at the full
// dense rate; N = 128 takes the same time, hence the 256-wide B.
// A (rows): f16 copies of the activations (a per-row power of two taken out,
//    exact), a 128 x 64 tile per k-stage by TMA with 128-byte swizzle, in a
//    ring of SA stages.
// B (weights): the stored e2m1 codes (128 rows x 32 bytes per box) and e4m3
//    scales (128 rows x 16 bytes, four k-stages) arrive by TMA in rings of
//    SR and SS slots; sixteen producer warps in four groups, each taking
//    every fourth k-stage (so four stages are in flight), two B rows per
//    thread, dequantise them to f16 (exact) into the 128-byte-swizzled
//    K-major tile, ring of SB.
// One thread issues the MMAs into fp32 accumulators in TMEM (two buffers of
// 256 columns) and commits each k-stage to one "stage done" barrier that
// frees both rings.  Four epilogue warps read a buffer (one row per thread).
// A producer that reads a TMA-filled slot with ordinary loads issues a proxy
// fence before it releases the slot: without it the slot's next TMA fill was
// seen to land before those loads had read it.
// The CTA's work list (expert, rows, slice) is decoded once into shared
// memory at the start.  Every mbarrier wait is bounded (about 2 s): on
// expiry the kernel records NVFP4_ERR_TIMEOUT, every role leaves its loop
// and the CTA still frees its tensor memory.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "tc.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {

namespace {

using namespace tc;

constexpr int BM = 128;            // routed rows per unit (MMA M)
constexpr int BN = 256;            // B rows per unit (MMA N)
constexpr int BK = 64;             // K per stage (one 128-byte swizzle row of f16)
constexpr int SR = 4;              // raw codes ring depth (k-stages)
constexpr int SS = 2;              // raw scales ring depth (groups of four k-stages)
constexpr int kABytes = BM * BK * 2;   // 16 KB
constexpr int kBBytes = BN * BK * 2;   // 32 KB
constexpr int kRawB = BN * BK / 2;     // 8 KB: two boxes of 128 weight rows x 32 bytes
constexpr int kScB = BN * 16;          // 4 KB: two boxes of 128 weight rows x 16 bytes
constexpr int kMaxUnits = 256;         // units per CTA (the host sizes the grid for it)
constexpr int kTileCopy = kMaxExperts + 1;
constexpr int kGroups = 4;                      // producer groups, one per k-stage residue
constexpr int kGroupWarps = 16 / kGroups;  // warps that produce one k-stage
static_assert(SR % kGroups == 0, "each raw slot must belong to one producer group");
// Ring geometry.
struct Geo {
    static constexpr int SA = 4;  // A (row) tiles
    static constexpr int SB = 3;  // f16 weight tiles
    static constexpr int SD0 = SA > SB ? SA : SB;
    // "stage done" barriers: at least every ring depth and the k-stage stride
    // between two waits of one producer group, so that parity waits stay in phase
    static constexpr int SD = SD0 > kGroups ? SD0 : kGroups;
    static constexpr int kRaw = kRawB;
    static constexpr int kSc = kScB;
    // fp32 row staging of the TCM_ROWS epilogue: 4 warps x 32 rows x 33 floats
    static constexpr int kStaging = 4 * 32 * 33 * 4;
    static constexpr int kSmem =
        1024 + SA * kABytes + SB * kBBytes + SR * kRaw + SS * kSc + kMaxUnits * 16 + kTileCopy * 4 + kStaging;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};
constexpr int kWarps = 24;
constexpr int kThreads = kWarps * 32;
constexpr int kWarpMma = 0, kWarpTmaA = 1, kWarpTmaB = 2, kWarpEpi = 4, kWarpDeq = 8, kDeqWarps = 16;

constexpr uint32_t kTmemCols = 512;    // two 256-column accumulators

// Waits until k-stage j's MMAs completed (j < 0: nothing to wait for).
template <int SD>
__device__ __forceinline__ bool wait_done(const uint64_t* done, long long j, volatile int* abort_flag,
                                          int32_t* status) {
    if (j < 0) return true;
    return mbar_wait(smem_u32(&done[j % SD]), (uint32_t)((j / SD) & 1), abort_flag, status);
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1) tcm_kernel(const __grid_constant__ TcmArgs a) {
    using G = Geo;
    constexpr int SA = G::SA, SB = G::SB, SD = G::SD, kRaw = G::kRaw, kSc = G::kSc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring_a = smem;
    uint8_t* ring_b = ring_a + SA * kABytes;
    uint8_t* ring_r = ring_b + SB * kBBytes;
    uint8_t* ring_s = ring_r + SR * kRaw;
    int4* s_units = reinterpret_cast<int4*>(ring_s + SS * kSc);  // {e, row0, row_end, f0}
    int* s_tiles = reinterpret_cast<int*>(s_units + kMaxUnits);
    float* s_stage = reinterpret_cast<float*>(s_tiles + kTileCopy);  // [4 warps][32][33] (TCM_ROWS)
    __shared__ __align__(8) uint64_t bar_afull[SA], bar_bfull[SB], bar_done[SD], bar_acc_full[2], bar_acc_empty[2];
    __shared__ __align__(8) uint64_t bar_rfull[SR], bar_rempty[SR], bar_sfull[SS], bar_sempty[SS];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    grid_dep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; ++s) mbar_init(smem_u32(&bar_afull[s]), 1);
        for (int s = 0; s < SB; ++s) mbar_init(smem_u32(&bar_bfull[s]), kGroupWarps);
        for (int s = 0; s < SD; ++s) mbar_init(smem_u32(&bar_done[s]), 1);
        for (int s = 0; s < SR; ++s) {
            mbar_init(smem_u32(&bar_rfull[s]), 1);
            mbar_init(smem_u32(&bar_rempty[s]), kGroupWarps);
        }
        for (int s = 0; s < SS; ++s) {
            mbar_init(smem_u32(&bar_sfull[s]), 1);
            mbar_init(smem_u32(&bar_sempty[s]), kDeqWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_acc_full[b]), 1);
            mbar_init(smem_u32(&bar_acc_empty[b]), 4);
        }
        s_abort = 0;
        mbar_fence_init();
    }
    if (warp == kWarpMma) tmem_alloc(smem_u32(&s_tmem), kTmemCols);

    // ---- this CTA's work list ----
    const int n_active = *a.n_active;
    constexpr bool kPair = EPI == TCM_SWIGLU;  // gate + up halves
    const int n_nt = kPair ? a.N / (BN / 2) : a.N / BN;  // B slices per expert
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
        const int f0 = (local / ntt) * (kPair ? BN / 2 : BN);
        const int row0 = a.offsets[e] + (local % ntt) * BM;
        s_units[t] = make_int4(e, row0, a.offsets[e + 1], f0);
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
    const int nk = a.K / BK;

    if (warp == kWarpMma) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(BM, BN);
            long long i = 0;
            for (int it = 0; it < n_units; ++it) {
                const int acc = it & 1;
                if (!mbar_wait(smem_u32(&bar_acc_empty[acc]), ((it >> 1) & 1) ^ 1, abort_flag, a.status)) break;
                tc_fence_after();
                const uint32_t d = tmem + acc * BN;
                bool ok = true;
                for (int kc = 0; kc < nk; ++kc, ++i) {
                    const int sa = (int)(i % SA), sb = (int)(i % SB);
                    if (!mbar_wait(smem_u32(&bar_afull[sa]), (uint32_t)((i / SA) & 1), abort_flag, a.status) ||
                        !mbar_wait(smem_u32(&bar_bfull[sb]), (uint32_t)((i / SB) & 1), abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = sdesc_sw128(smem_u32(ring_a + sa * kABytes));
                    const uint64_t bdesc = sdesc_sw128(smem_u32(ring_b + sb * kBBytes));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_f16(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kc | kk) != 0);
                    mma_commit(smem_u32(&bar_done[i % SD]));
                }
                if (!ok) break;
                mma_commit(smem_u32(&bar_acc_full[acc]));
            }
        }
        __syncwarp();
    } else if (warp == kWarpTmaB) {
        // ---------------- raw weights by TMA (one thread) ----------------
        if (lane == 0) {
            long long i = 0, g = 0;
            bool ok = true;
            for (int it = 0; it < n_units && ok; ++it) {
                const int4 un = s_units[it];
                // B rows 0..127 and 128..255: (map, row) of each half
                const int y0 = un.x * a.N + un.w;
                const int y1 = kPair ? y0 : y0 + BN / 2;
                const void* mc1 = kPair ? (const void*)&a.tmap_wc[1] : (const void*)&a.tmap_wc[0];
                const void* ms1 = kPair ? (const void*)&a.tmap_ws[1] : (const void*)&a.tmap_ws[0];
                for (int kc = 0; kc < nk; ++kc, ++i) {
                    if ((kc & 3) == 0) {
                        const int ss = (int)(g % SS);
                        if (!mbar_wait(smem_u32(&bar_sempty[ss]), (uint32_t)(((g / SS) & 1) ^ 1), abort_flag,
                                       a.status)) {
                            ok = false;
                            break;
                        }
                        const uint32_t bar = smem_u32(&bar_sfull[ss]);
                        mbar_arrive_expect_tx(bar, kSc);
                        uint8_t* dst = ring_s + ss * kSc;
                        tma_load_2d(smem_u32(dst), &a.tmap_ws[0], kc * 4, y0, bar);
                        tma_load_2d(smem_u32(dst + kScB / 2), ms1, kc * 4, y1, bar);
                        ++g;
                    }
                    const int sr = (int)(i % SR);
                    if (!mbar_wait(smem_u32(&bar_rempty[sr]), (uint32_t)(((i / SR) & 1) ^ 1), abort_flag,
                                   a.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bar = smem_u32(&bar_rfull[sr]);
                    mbar_arrive_expect_tx(bar, kRaw);
                    uint8_t* dst = ring_r + sr * kRaw;
                    tma_load_2d(smem_u32(dst), &a.tmap_wc[0], kc * 32, y0, bar);
                    tma_load_2d(smem_u32(dst + kRawB / 2), mc1, kc * 32, y1, bar);
                }
            }
        }
        __syncwarp();
    } else if (warp == kWarpTmaA) {
        // ---------------- A producer: routed f16 rows by TMA (one thread) ----------------
        if (lane == 0) {
            long long i = 0;
            for (int it = 0; it < n_units; ++it) {
                const int row0 = s_units[it].y;
                bool ok = true;
                for (int kc = 0; kc < nk; ++kc, ++i) {
                    if (!wait_done<SD>(bar_done, i - SA, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bar = smem_u32(&bar_afull[i % SA]);
                    mbar_arrive_expect_tx(bar, kABytes);
                    tma_load_2d(smem_u32(ring_a + (i % SA) * kABytes), &a.tmap_x, kc * BK, row0, bar);
                }
                if (!ok) break;
            }
        }
        __syncwarp();
    } else if (warp >= kWarpEpi && warp < kWarpEpi + 4) {
        // ---------------- epilogue: one routed row per thread ----------------
        const int q = warp - kWarpEpi;
        const int rr = q * 32 + lane;  // row within the unit = TMEM lane
        for (int it = 0; it < n_units; ++it) {
            const int4 un = s_units[it];
            const int acc = it & 1;
            const int row = un.y + rr;
            const bool valid = row < un.z;
            const float rs = valid ? exp2i(a.x_exp[row]) : 0.0f;
            const float w0 = a.a_ws2[0][un.x], w1 = a.a_ws2[1][un.x];
            if (!mbar_wait(smem_u32(&bar_acc_full[acc]), (it >> 1) & 1, abort_flag, a.status, 64)) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + acc * BN;
            if constexpr (EPI == TCM_SWIGLU) {
                for (int cb = 0; cb < BN / 32; ++cb) {
                    uint32_t g[16], u[16];
                    tmem_ld16(tb + cb * 16, g);
                    tmem_ld16(tb + BN / 2 + cb * 16, u);
                    tmem_ld_wait();
                    if (valid) {
                        uint32_t packed[8];
#pragma unroll
                        for (int j = 0; j < 16; j += 2) {
                            float hv[2];
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                const float G = round_bf16(__fmul_rn(__fmul_rn(__uint_as_float(g[j + t]), rs), w0));
                                const float U = round_bf16(__fmul_rn(__fmul_rn(__uint_as_float(u[j + t]), rs), w1));
                                hv[t] = G / (1.0f + expf(-G)) * U;
                            }
                            packed[j / 2] =
                                (uint32_t)f32_to_bf16_bits(hv[0]) | ((uint32_t)f32_to_bf16_bits(hv[1]) << 16);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(a.h_out + (size_t)row * a.N + un.w + cb * 16);
                        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                    }
                }
            } else if constexpr (EPI == TCM_ROWS) {
                // y = ws2 * x W^T as bf16 rows by routed row: 32 rows x 32 columns
                // per chunk through shared memory, then two rows (2 x 64 bytes)
                // per store instruction; a second kernel adds each token's k
                // rows, weighted, in slot order (deterministic combine)
                float* st = s_stage + (size_t)q * 32 * 33;
                const int nvalid = min(32, un.z - (un.y + q * 32));  // rows of this warp in the unit
                const int hr = lane >> 4, cl = (lane & 15) * 2;
                for (int cb = 0; cb < BN / 32; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(tb + cb * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) st[lane * 33 + c] = __fmul_rn(__fmul_rn(__uint_as_float(r[c]), rs), w0);
                    __syncwarp();
                    uint16_t* ybase = a.y_rows + (size_t)(un.y + q * 32) * a.N + un.w + cb * 32 + cl;
                    for (int j = hr; j < nvalid; j += 2)
                        *reinterpret_cast<uint32_t*>(ybase + (size_t)j * a.N) =
                            (uint32_t)f32_to_bf16_bits(st[j * 33 + cl]) | ((uint32_t)f32_to_bf16_bits(st[j * 33 + cl + 1]) << 16);
                    __syncwarp();
                }
            } else {
                for (int cb = 0; cb < BN / 32; ++cb) {
                    uint32_t r[32];
                    tmem_ld32(tb + cb * 32, r);
                    tmem_ld_wait();
                    if (valid) {
                        uint32_t packed[16];
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            const float y0 = __fmul_rn(__fmul_rn(__uint_as_float(r[j]), rs), w0);
                            const float y1 = __fmul_rn(__fmul_rn(__uint_as_float(r[j + 1]), rs), w0);
                            packed[j / 2] = (uint32_t)f32_to_bf16_bits(y0) | ((uint32_t)f32_to_bf16_bits(y1) << 16);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(a.y_out + (size_t)row * a.N + un.w + cb * 32);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_acc_empty[acc]));
        }
    } else if (warp >= kWarpDeq) {
        // ---------------- producers: raw NVFP4 rows -> f16 tile rows ----------------
        // Group grp takes k-stage grp of every scale group (four k-stages);
        // its 128 threads own two B rows each.
        // The proxy fence after the stage's smem stores also orders the
        // reads of the TMA-filled raw slots before their next fill, so the
        // raw slots are released together with the f16 tiles.
        const int dw = warp - kWarpDeq;
        const int grp = dw / kGroupWarps;              // = the k-stage q of each scale group
        const int tg = (dw % kGroupWarps) * 32 + lane;  // 0..127: B rows tg and tg + 128, A row tg
        const int ng = nk / 4;
        long long gg = 0;
        bool ok = true;
        for (int it = 0; it < n_units && ok; ++it) {
            for (int kg = 0; kg < ng && ok; ++kg, ++gg) {
                const int ss = (int)(gg % SS);
                if (!mbar_wait(smem_u32(&bar_sfull[ss]), (uint32_t)((gg / SS) & 1), abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                const int q = grp;
                const uint32_t sw0 = *reinterpret_cast<const uint32_t*>(ring_s + ss * kSc + tg * 16 + q * 4);
                const uint32_t sw1 = *reinterpret_cast<const uint32_t*>(ring_s + ss * kSc + (tg + 128) * 16 + q * 4);
                const long long i = (long long)it * nk + kg * 4 + q;
                const int sr = (int)(i % SR);
                if (!mbar_wait(smem_u32(&bar_rfull[sr]), (uint32_t)((i / SR) & 1), abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                // 32-byte swizzle: half h of row r sits at h ^ (bit 2 of r)
                // (rows tg and tg + 128 share that bit)
                const int h0 = ((tg >> 2) & 1) << 4, h1 = 16 - h0;
                uint4 c[4];
                c[0] = *reinterpret_cast<const uint4*>(ring_r + sr * kRaw + tg * 32 + h0);
                c[1] = *reinterpret_cast<const uint4*>(ring_r + sr * kRaw + tg * 32 + h1);
                c[2] = *reinterpret_cast<const uint4*>(ring_r + sr * kRaw + (tg + 128) * 32 + h0);
                c[3] = *reinterpret_cast<const uint4*>(ring_r + sr * kRaw + (tg + 128) * 32 + h1);
                if (!wait_done<SD>(bar_done, i - SB, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int j = tg + rr * 128;
                    uint8_t* rowp = ring_b + (i % SB) * kBBytes + j * 128;
                    const uint32_t sw = rr ? sw1 : sw0;
                    const uint32_t S01 = e4m3x2_to_f16x2(sw & 0xFFFFu), S23 = e4m3x2_to_f16x2(sw >> 16);
                    const uint32_t Sb[4] = {f16x2_bcast(S01, 0), f16x2_bcast(S01, 1), f16x2_bcast(S23, 0),
                                            f16x2_bcast(S23, 1)};
                    const uint4 x0 = c[2 * rr], x1 = c[2 * rr + 1];
                    const uint32_t cw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        uint32_t f[4];
                        e2m1x8_to_f16x8(cw[w], f);
                        const uint32_t S2 = Sb[w >> 1];
                        *reinterpret_cast<uint4*>(rowp + ((w ^ (j & 7)) << 4)) = make_uint4(
                            hmul2_u32(f[0], S2), hmul2_u32(f[1], S2), hmul2_u32(f[2], S2), hmul2_u32(f[3], S2));
                    }
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&bar_bfull[i % SB]));
                    mbar_arrive(smem_u32(&bar_rempty[sr]));
                    mbar_arrive(smem_u32(&bar_sempty[ss]));
                }
            }
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

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

template <int EPI>
void launch_tcm_t(const TcmArgs& a, int max_units, cudaStream_t s, const char* name) {
    auto kern = tcm_kernel<EPI>;
    constexpr int smem = Geo::kSmem;
    static bool init = false;
    if (!init) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        init = true;
    }
    int grid = std::max(1, std::min(max_units, num_sms()));
    grid = std::max(grid, (max_units + kMaxUnits - 1) / kMaxUnits);
    NVFP4_LAUNCH(name, s, launch_pdl(kern, dim3(grid), dim3(kThreads), (size_t)smem, s, a));
}

}  // namespace

void init_encode() {
    std::call_once(g_encode_once, []() {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
}

bool encode_tmap_u8(CUtensorMap* map, const void* base, unsigned long long inner_bytes, unsigned long long rows,
                    unsigned box_inner, unsigned box_rows, bool swizzle128) {
    init_encode();
    if (!g_encode || rows < 1 || inner_bytes % 16 != 0 || !aligned16(base)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner_bytes, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)inner_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_rows_f16(CUtensorMap* map, const void* base, int rows, int K) {
    init_encode();
    if (!g_encode || rows < 1 || K % BK != 0 || !aligned16(base)) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {BK, BM};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The stored codes [rows, K/2] and scales [rows, K/16] of an NVFP4 tensor as
// uint8 tensor maps: boxes of 128 rows x 32 bytes (one k-stage of codes,
// with the 32-byte swizzle: the two 16-byte halves of row r swap places
// when bit 2 of r is set, so that the producers' 16-byte reads of eight
// consecutive rows hit eight distinct bank groups) and 128 rows x 16 bytes
// (four k-stages of scales), no swizzle.
bool make_tmap_weights(CUtensorMap* codes, CUtensorMap* scales, const uint8_t* c, const uint8_t* sc, long long rows,
                       int K) {
    if (!g_encode || rows < 1 || K % 256 != 0 || !aligned16(c) || !aligned16(sc)) return false;
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t cd[2] = {(cuuint64_t)K / 2, (cuuint64_t)rows};
    const cuuint64_t cs[1] = {(cuuint64_t)K / 2};
    const cuuint32_t cb[2] = {32, 128};
    if (g_encode(codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(c), cd, cs, cb, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    const cuuint64_t sd[2] = {(cuuint64_t)K / 16, (cuuint64_t)rows};
    const cuuint64_t ss[1] = {(cuuint64_t)K / 16};
    const cuuint32_t sb[2] = {16, 128};
    return g_encode(scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(sc), sd, ss, sb, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tcm_supported(int epi, int N, int K) {
    if (epi != TCM_SWIGLU && epi != TCM_ROWS && epi != TCM_BF16) return false;
    const bool pair = epi == TCM_SWIGLU;
    return K % 256 == 0 && (pair ? N % (BN / 2) == 0 : N % BN == 0);
}

bool tcm_set_weights(TcmArgs* a, long long rows) {
    init_encode();
    for (int p = 0; p < 2; ++p)
        if (!make_tmap_weights(&a->tmap_wc[p], &a->tmap_ws[p], a->a_codes[p], a->a_scales[p], rows, a->K))
            return false;
    return true;
}

void launch_tcm(int epi, const TcmArgs& a, int max_units, cudaStream_t s) {
    if (epi == TCM_SWIGLU) return launch_tcm_t<TCM_SWIGLU>(a, max_units, s, "tcm_gateup_w4a16");
    if (epi == TCM_ROWS) return launch_tcm_t<TCM_ROWS>(a, max_units, s, "tcm_down_w4a16");
    if (epi == TCM_BF16) return launch_tcm_t<TCM_BF16>(a, max_units, s, "tcm_linear_w4a16");
}

}  // namespace nvfp4
