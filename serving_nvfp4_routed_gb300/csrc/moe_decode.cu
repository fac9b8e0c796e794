// moe_decode.cu -- the decode-shaped routed-expert layer in one persistent
// launch: gate/up + SwiGLU, then down + the weighted top-k combine.
//
// TensorFold issue #308 "GLM-5.3-Flash on CUDA: read nvidia/GLM-5.3-Flash-NVFP4
// (ModelOpt NVFP4) as stored, W4A16", "What the branch does": the routed
// experts run through one grouped kernel over bf16 rows with weight_scale_2
// as the per-expert multiplier, and FP4 x FP4 (W4A4) is the checkpoint's own
// math; "Questions", item 4: decode and prompt shapes get their own kernels.
//
// With a few tokens per expert the layer is a stream of 4.5-bit weights
// (codes + e4m3 scales) from HBM, each read once for the handful of rows
// routed to its expert.  The stream is fed by TMA rather than by registers:
//   * one CTA per SM; work items come from a device counter in order: every
//     gate/up item (expert row tile of up to 8 routed rows x a group of
//     128-feature blocks), then every down item (row tile x a group of
//     256-output blocks);
//   * a producer warp loads each stage -- 256 weight rows (128 gate + 128
//     up rows of one feature block, or 256 down rows) x 256 K of the stored
//     codes and scales -- with tiled TMA into a ring of shared-memory slots,
//     running ahead across items;
//   * each of sixteen consumer warps owns 16 of the stage's rows (8 gate + 8
//     up rows of the same features, so that SwiGLU stays in its registers)
//     over every K chunk of the block: no partial sums to exchange.  It
//     loads its codes and scales from shared memory into mma.sync m16n8k16
//     A fragments (K permuted inside each 256-wide chunk so that every lane's
//     codes are contiguous; the B rows use the same permutation), dequantises
//     them in registers (cvt e2m1x2 -> f16x2, times the block scale: exact)
//     and multiplies the item's routed rows, staged once per item in shared
//     memory as f16 (bf16 rows with a per-row power of two taken out, or
//     NVFP4 rows dequantised exactly), on four accumulator chains;
//   * gate/up writes h = bf16(silu(G) * U) (W4A4: requantised to NVFP4 under
//     the down input scale) and, once an item is done, raises its row tile's
//     counter;
//   * a down item waits (bounded) for its tile's counter before it stages h,
//     while its weights are already streaming; it writes w * y per routed
//     row (fp32) and counts each (token, output group); the CTA that adds a
//     token's k-th contribution to a group sums the token's k rows in slot
//     order and writes the bf16 output: the same bits on every run.
// A down item waits only on gate/up items, all of which were handed out
// before it to CTAs that are running and wait on nothing, so the waits end.
// Every wait is bounded (about 2 s) and reports NVFP4_ERR_TIMEOUT; the
// producer then waits (bounded) for its copies in flight before it exits.
#include "common.cuh"
#include "internal.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {

namespace {

using namespace tc;

constexpr int kConsumers = 16;                   // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;  // + one producer warp
constexpr int kNS = 4;                           // ring slots
constexpr int kRows = 16 * kConsumers;           // weight rows per stage
constexpr int kFeatGU = kRows / 2;               // features per gate/up block (128 gate + 128 up rows)
constexpr int kChunk = 256;                      // K per stage (one 128-byte box row of codes)
constexpr int kBarConsumers = 1;                 // named barrier of the consumer warps
// Independent accumulator chains per warp (mma.sync has a long latency on
// this part).  Measured on GB300: with eight consumer warps the kernel was
// bound by instruction latency (14 % warps active, 37 % issue active), so
// sixteen warps share the stage, which caps a thread at 120 registers.
constexpr int kChains = 4;

struct Hdr {
    int kind;    // 0 gate/up, 1 down, -1 end of work
    int e, row0, nrows;
    int tile, grp;
    int f;       // first feature (gate/up) or output (down) of this stage's block
    int kc;      // K chunk of this stage
    int j;       // stage index within the item
    int nst;     // stages of the item
};

template <int CK>
struct Ch {
    static constexpr int TS = CK / 4;   // physical K per lane
    static constexpr int CB = CK / 8;   // code bytes per lane per row
    static constexpr int KS = CK / 16;  // mma k-steps per chunk
    static constexpr int CW = CB / 4;   // code words per lane per row
};

template <int CK>
__device__ __forceinline__ void lds_codes(const uint8_t* p, uint32_t* w) {
    if constexpr (CK == 256) {
        const uint4 u0 = *reinterpret_cast<const uint4*>(p);
        const uint4 u1 = *reinterpret_cast<const uint4*>(p + 16);
        w[0] = u0.x; w[1] = u0.y; w[2] = u0.z; w[3] = u0.w;
        w[4] = u1.x; w[5] = u1.y; w[6] = u1.z; w[7] = u1.w;
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        w[0] = u.x; w[1] = u.y;
    }
}

template <int CK>
__device__ __forceinline__ uint32_t lds_scales(const uint8_t* p) {
    if constexpr (CK == 256) return *reinterpret_cast<const uint32_t*>(p);
    else return *p;
}

// A lane's block scales as f16x2 pairs (the scale of block b in both
// halves of S[b]) from the 4 bytes (CK = 256) or 1 byte (CK = 64) it loaded.
template <int NB>
__device__ __forceinline__ void block_scales(uint32_t sw, uint32_t (&S)[NB]) {
    const uint32_t s01 = e4m3x2_to_f16x2(sw & 0xFFFFu);
    S[0] = f16x2_bcast(s01, 0);
    if constexpr (NB > 1) {
        const uint32_t s23 = e4m3x2_to_f16x2(sw >> 16);
        S[1] = f16x2_bcast(s01, 1);
        S[2] = f16x2_bcast(s23, 0);
        S[3] = f16x2_bcast(s23, 1);
    }
}

// Dequantised f16x2 words of one code word (8 codes of one 16-block, block
// scale S as f16x2): out[0] = phys 0..1, out[1] = 2..3, out[2] = 4..5, out[3] = 6..7.
__device__ __forceinline__ void deq_word(uint32_t word, uint32_t S, uint32_t out[4]) {
    uint32_t f[4];
    e2m1x8_to_f16x8(word, f);
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = hmul2_u32(f[i], S);
}

// Staged B rows: row g holds K f16 values as K/8 16-byte granules; granule
// q sits at bsw(q, g) so that the B-fragment reads of a quarter warp (lanes
// (g, c) read granule c*TS/8 + j of row g, g in a pair of rows) hit eight
// distinct 16-byte bank groups.
template <int CK>
__device__ __forceinline__ int bsw(int q, int g) {
    if constexpr (CK == 256) return q ^ ((((q >> 3) & 3) << 1) | (g & 1));
    else return q ^ (g & 1);
}

__device__ __forceinline__ uint32_t bf16x2_scaled_to_f16x2(uint32_t u, float sc) {
    return f32x2_to_f16x2(bf16_bits_to_f32(u & 0xFFFFu) * sc, bf16_bits_to_f32(u >> 16) * sc);
}

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void consumer_sync() { named_bar(kBarConsumers, kConsumers * 32); }

// Stage rows row0 .. row0 + nrows - 1 of the item as f16 into Bs (K values
// each, swizzled for chunk width CK); s_rowscale[j] receives the factor that
// takes an accumulator over row j back to x W^T (W4A16: the row's power of
// two; W4A4: 1, the input scale is applied in the epilogue).
template <int CK, int BMODE>
__device__ void stage_rows(const DecodeArgs& a, int K, int row0, int nrows, bool by_token, bool written_here,
                           const uint16_t* bf16_src, const uint8_t* q_src, const uint8_t* s_src, uint4* Bs,
                           float* s_rowscale, unsigned* s_amax, int warp, int lane) {
    const int Kg = K / 8;
    const int j = warp % nrows, gi = warp / nrows;
    const int gsz = (kConsumers - j + nrows - 1) / nrows;  // warps staging row j
    const int r = row0 + j;
    uint4* dst = Bs + (size_t)j * Kg;
    if constexpr (BMODE == B_BF16) {
        const int srow = by_token ? a.row_to_slot[r] / a.top_k : r;
        const uint4* src = reinterpret_cast<const uint4*>(bf16_src + (size_t)srow * K);
        float m = 0.0f;
        for (int q = gi * 32 + lane; q < Kg; q += gsz * 32) {
            const uint4 u = written_here ? __ldcg(src + q) : __ldg(src + q);
            const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_f32(ww[i] & 0xFFFFu)), fabsf(bf16_bits_to_f32(ww[i] >> 16))));
            dst[bsw<CK>(q, j)] = u;
        }
        m = warp_max(m);
        if (lane == 0) atomicMax(&s_amax[j], __float_as_uint(m));
        consumer_sync();
        const int sexp = row_exponent(__uint_as_float(s_amax[j]));
        const float down = exp2i(-sexp);
        if (gi == 0 && lane == 0) s_rowscale[j] = exp2i(sexp);
        for (int q = gi * 32 + lane; q < Kg; q += gsz * 32) {
            const int qs = bsw<CK>(q, j);
            const uint4 u = dst[qs];
            dst[qs] = make_uint4(bf16x2_scaled_to_f16x2(u.x, down), bf16x2_scaled_to_f16x2(u.y, down),
                                 bf16x2_scaled_to_f16x2(u.z, down), bf16x2_scaled_to_f16x2(u.w, down));
        }
    } else {
        const uint8_t* codes = q_src + (size_t)r * (K / 2);
        const uint8_t* scales = s_src + (size_t)r * (K / 16);
        for (int b = gi * 32 + lane; b < K / 16; b += gsz * 32) {  // 16-block: 8 code bytes, 1 scale
            const uint2 cw = written_here ? __ldcg(reinterpret_cast<const uint2*>(codes) + b)
                                          : __ldg(reinterpret_cast<const uint2*>(codes) + b);
            const uint32_t sb = written_here ? (uint32_t)__ldcg(scales + b) : (uint32_t)__ldg(scales + b);
            const uint32_t S = f16x2_bcast(e4m3x2_to_f16x2(sb), 0);
            uint32_t f0[4], f1[4];
            e2m1x8_to_f16x8(cw.x, f0);
            e2m1x8_to_f16x8(cw.y, f1);
            dst[bsw<CK>(2 * b, j)] =
                make_uint4(hmul2_u32(f0[0], S), hmul2_u32(f0[1], S), hmul2_u32(f0[2], S), hmul2_u32(f0[3], S));
            dst[bsw<CK>(2 * b + 1, j)] =
                make_uint4(hmul2_u32(f1[0], S), hmul2_u32(f1[1], S), hmul2_u32(f1[2], S), hmul2_u32(f1[3], S));
        }
        if (gi == 0 && lane == 0) s_rowscale[j] = 1.0f;
    }
}

// One warp's share of a stage: MMA row g from codes c0 / scales s0, row
// g + 8 from c1 / s1 (row pitches KC/2 and KC/16 bytes, as the TMA boxes
// land); the stage covers K [k0, k0 + KC) of the staged B rows (row length
// K); k-step i accumulates into chain i % kChains.
template <int CK>
__device__ __forceinline__ void stage_mma(const uint8_t* c0, const uint8_t* c1, const uint8_t* s0, const uint8_t* s1,
                                          int KC, int k0, const uint4* Bs, int K, int lane,
                                          float (&acc)[kChains][4]) {
    using C = Ch<CK>;
    const int g = lane >> 2, c = lane & 3;
    const int kb2 = KC / 2, ks16 = KC / 16;
    const uint8_t* r0c = c0 + g * kb2;
    const uint8_t* r1c = c1 + g * kb2;
    const uint8_t* r0s = s0 + g * ks16;
    const uint8_t* r1s = s1 + g * ks16;
    const uint4* brow = Bs + (size_t)g * (K / 8);
#pragma unroll 1
    for (int kc = 0; kc < KC; kc += CK) {
        const int kb = kc + c * C::TS;  // this lane's physical K inside the stage's chunk
        uint32_t w0[C::CW], w1[C::CW];
        lds_codes<CK>(r0c + kb / 2, w0);
        lds_codes<CK>(r1c + kb / 2, w1);
        constexpr int NB = C::TS / 16;  // 16-blocks per lane and chunk
        uint32_t S0[NB], S1[NB];
        block_scales<NB>(lds_scales<CK>(r0s + kb / 16), S0);
        block_scales<NB>(lds_scales<CK>(r1s + kb / 16), S1);
        const int qb = (k0 + kb) / 8;
#pragma unroll
        for (int jj = 0; jj < C::KS; jj += 2) {
            const uint4 bq = brow[bsw<CK>(qb + jj / 2, g)];
            const uint32_t b0[2] = {bq.x, bq.y};
            const uint32_t b1[2] = {bq.z, bq.w};
            uint32_t x0[4], x1[4];
            deq_word(w0[jj >> 1], S0[jj >> 2], x0);
            deq_word(w1[jj >> 1], S1[jj >> 2], x1);
            const uint32_t af0[4] = {x0[0], x1[0], x0[1], x1[1]};
            const uint32_t af1[4] = {x0[2], x1[2], x0[3], x1[3]};
            mma_16816(acc[jj % kChains], af0, b0);
            mma_16816(acc[(jj + 1) % kChains], af1, b1);
        }
    }
}

template <int BMODE, int CKG, int CKD>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint4* Bs = reinterpret_cast<uint4*>(ring + (size_t)kNS * a.slot_bytes);
    const int kmax = a.d > a.F ? a.d : a.F;
    // W4A4: h of one 64-feature block [8 rows][64], exchanged between warps for the requantisation
    float* s_hx = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(Bs) + (size_t)kGemvTokTile * kmax * 2);
    __shared__ __align__(8) uint64_t bar_full[kNS], bar_empty[kNS];
    __shared__ Hdr s_hdr[kNS];
    __shared__ float s_rowscale[kGemvTokTile];
    __shared__ unsigned s_amax[2][kGemvTokTile];
    __shared__ int s_fin[kGemvTokTile];
    __shared__ int s_abort, s_stop;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), kConsumers);
        }
        s_abort = 0;
        s_stop = 0;
        mbar_fence_init();
    }
    if (threadIdx.x < 2 * kGemvTokTile) (&s_amax[0][0])[threadIdx.x] = 0u;
    __syncthreads();
    grid_dep_wait();
    volatile int* abort_flag = &s_abort;

    const int n_active = *a.n_active;
    const int n_tiles = a.tile_start[n_active];
    const int nbu = a.F / kFeatGU, nbd = a.d / kRows;  // 64-feature / 128-output blocks
    const int ngu = nbu / a.gbu, ngd = nbd / a.gbd;    // item groups per tile
    const int nchu = a.d / kChunk, nchd = a.F / kChunk;  // K chunks per block
    const int nA = n_tiles * ngu, total = nA + n_tiles * ngd;

    if (warp == kConsumers) {
        // ---------------- producer: one lane issues the TMA loads ----------------
        if (lane == 0) {
            long long st = 0;
            bool ok = true;
            for (;;) {
                const int item = atomicAdd(a.counters, 1);
                Hdr h{};
                int nst = 1;
                if (item >= total || *abort_flag) {
                    h.kind = -1;
                } else {
                    const bool down = item >= nA;
                    const int it = down ? item - nA : item;
                    const int ng = down ? ngd : ngu;
                    h.kind = down ? 1 : 0;
                    h.tile = it / ng;
                    h.grp = it % ng;
                    int lo = 0, hi = n_active;  // largest lo with tile_start[lo] <= tile
                    while (hi - lo > 1) {
                        const int mid = (lo + hi) >> 1;
                        if (a.tile_start[mid] <= h.tile) lo = mid; else hi = mid;
                    }
                    h.e = a.active[lo];
                    h.row0 = a.offsets[h.e] + (h.tile - a.tile_start[lo]) * kGemvTokTile;
                    h.nrows = min(kGemvTokTile, a.offsets[h.e + 1] - h.row0);
                    nst = down ? a.gbd * nchd : a.gbu * nchu;
                    h.nst = nst;
                }
                for (int j = 0; j < nst; ++j, ++st) {
                    const int s = (int)(st % kNS);
                    if (!mbar_wait(smem_u32(&bar_empty[s]), (uint32_t)(((st / kNS) & 1) ^ 1), abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    h.j = j;
                    const uint32_t full = smem_u32(&bar_full[s]);
                    if (h.kind < 0) {
                        s_hdr[s] = h;
                        mbar_arrive(full);
                        continue;
                    }
                    const uint32_t dst = smem_u32(ring + (size_t)s * a.slot_bytes);
                    if (h.kind == 0) {
                        const int blk = h.grp * a.gbu + j / nchu;
                        h.kc = j % nchu;
                        h.f = blk * kFeatGU;
                        s_hdr[s] = h;
                        const int y = h.e * a.F + h.f;
                        const uint32_t cb = kFeatGU * kChunk / 2, sb = kFeatGU * kChunk / 16;
                        mbar_arrive_expect_tx(full, 2 * (cb + sb));
                        tma_load_2d(dst, &a.tm_gate_c, h.kc * (kChunk / 2), y, full);
                        tma_load_2d(dst + cb, &a.tm_up_c, h.kc * (kChunk / 2), y, full);
                        tma_load_2d(dst + 2 * cb, &a.tm_gate_s, h.kc * (kChunk / 16), y, full);
                        tma_load_2d(dst + 2 * cb + sb, &a.tm_up_s, h.kc * (kChunk / 16), y, full);
                    } else {
                        const int blk = h.grp * a.gbd + j / nchd;
                        h.kc = j % nchd;
                        h.f = blk * kRows;
                        s_hdr[s] = h;
                        const int y = h.e * a.d + h.f;
                        const uint32_t cb = kRows * kChunk / 2, sb = kRows * kChunk / 16;
                        mbar_arrive_expect_tx(full, cb + sb);
                        tma_load_2d(dst, &a.tm_down_c, h.kc * (kChunk / 2), y, full);
                        tma_load_2d(dst + cb, &a.tm_down_s, h.kc * (kChunk / 16), y, full);
                    }
                }
                if (!ok || h.kind < 0) break;
            }
            // before the CTA exits, every copy it issued must have landed (a
            // bounded wait that does not stop at the abort flag)
            volatile int keep_waiting = 0;
            for (long long i = st > kNS ? st - kNS : 0; i < st; ++i)
                mbar_wait(smem_u32(&bar_full[i % kNS]), (uint32_t)((i / kNS) & 1), &keep_waiting, nullptr);
        }
        __syncwarp();
    } else {
        // ---------------- consumers ----------------
        const int g = lane >> 2, c = lane & 3;
        float acc[kChains][4];
#pragma unroll
        for (int q = 0; q < kChains; ++q)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[q][i] = 0.0f;
        long long st = 0;
        int par = 0;
        Hdr cur{};
        for (;;) {
            const int s = (int)(st % kNS);
            if (!warp_wait(smem_u32(&bar_full[s]), (uint32_t)((st / kNS) & 1), abort_flag, a.status) || *abort_flag)
                break;
            const Hdr h = s_hdr[s];
            if (h.kind < 0) break;
            const bool down = h.kind == 1;
            if (h.j == 0) {
                // ---- a new item: stage its routed rows ----
                cur = h;
                consumer_sync();  // the previous item's readers of Bs / s_rowscale are done
                if (threadIdx.x < kGemvTokTile) s_amax[par ^ 1][threadIdx.x] = 0u;
                if (down) {
                    if (threadIdx.x == 0) {
                        const long long t0 = clock64();
                        int stop = 0;
                        while (ld_acquire(a.tile_ready + h.tile) < ngu) {
                            if (*abort_flag) {
                                stop = 1;
                                break;
                            }
                            if (clock64() - t0 > kWaitCycles) {
                                *abort_flag = 1;
                                if (a.status) atomicExch(a.status, (int)NVFP4_ERR_TIMEOUT);
                                stop = 1;
                                break;
                            }
                            __nanosleep(256);
                        }
                        s_stop = stop;
                    }
                    consumer_sync();
                    if (s_stop) break;
                    stage_rows<CKD, BMODE>(a, a.F, h.row0, h.nrows, false, true, a.h, a.hq, a.hs, Bs, s_rowscale,
                                           s_amax[par], warp, lane);
                } else {
                    stage_rows<CKG, BMODE>(a, a.d, h.row0, h.nrows, BMODE == B_BF16, false, a.x, a.xq, a.xs, Bs,
                                           s_rowscale, s_amax[par], warp, lane);
                }
                par ^= 1;
                consumer_sync();
            }
            // ---- this warp's 16 rows of the stage ----
            const int nch = down ? nchd : nchu;
            if (h.kc == 0) {
#pragma unroll
                for (int q = 0; q < kChains; ++q)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[q][i] = 0.0f;
            }
            const uint8_t* slot = ring + (size_t)s * a.slot_bytes;
            if (!down) {
                // MMA rows 0-7: gate rows 8w..8w+7 of the block, rows 8-15: the up rows of the same features
                const int cb = kFeatGU * kChunk / 2, sb = kFeatGU * kChunk / 16;
                const uint8_t* gc = slot + 8 * warp * (kChunk / 2);
                const uint8_t* gs = slot + 2 * cb + 8 * warp * (kChunk / 16);
                stage_mma<CKG>(gc, gc + cb, gs, gs + sb, kChunk, h.kc * kChunk, Bs, a.d, lane, acc);
            } else {
                const int cb = kRows * kChunk / 2;
                const uint8_t* dc = slot + 16 * warp * (kChunk / 2);
                const uint8_t* ds = slot + cb + 16 * warp * (kChunk / 16);
                stage_mma<CKD>(dc, dc + 8 * (kChunk / 2), ds, ds + 8 * (kChunk / 16), kChunk, h.kc * kChunk, Bs,
                               a.F, lane, acc);
            }
            // the slot is refilled by TMA (async proxy) after its release
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_empty[s]));

            if (h.kc == nch - 1) {
                // ---- this warp's rows of the block are complete: epilogue ----
                float t[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float v = acc[0][i];
#pragma unroll
                    for (int q = 1; q < kChains; ++q) v += acc[q][i];
                    t[i] = v;
                }
                const int e = cur.e;
                if (!down) {
                    // lane (g, c): feature f + 8w + g; gate in t[cc], up in t[2 + cc] for row 2c + cc
                    const int f = h.f + 8 * warp + g;
                    const float wg = a.gate_ws2[e], wu = a.up_ws2[e];
                    float hv[2];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int col = 2 * c + cc;
                        const bool valid = col < cur.nrows;
                        const float rs = BMODE == B_BF16 ? (valid ? s_rowscale[col] : 0.0f) : a.is13[e];
                        const float G = round_bf16(__fmul_rn(__fmul_rn(t[cc], rs), wg));
                        const float U = round_bf16(__fmul_rn(__fmul_rn(t[2 + cc], rs), wu));
                        hv[cc] = valid ? round_bf16(G / (1.0f + expf(-G)) * U) : 0.0f;
                        if constexpr (BMODE == B_BF16) {
                            if (valid) a.h[(size_t)(cur.row0 + col) * a.F + f] = f32_to_bf16_bits(hv[cc]);
                        }
                    }
                    if constexpr (BMODE == B_NVFP4) {
                        // an NVFP4 block of 16 features spans two warps: h goes
                        // through shared memory, then warp w requantises routed
                        // row w % 8 of the block, blocks 4 (w / 8) .. + 3 (lane b
                        // of those: features 16b .. 16b + 15)
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) s_hx[(2 * c + cc) * kFeatGU + 8 * warp + g] = hv[cc];
                        consumer_sync();
                        const int row = warp % kGemvTokTile;
                        constexpr int kBlkPerWarp = kFeatGU / 16 / (kConsumers / kGemvTokTile);
                        if (row < cur.nrows && lane < kBlkPerWarp) {
                            const int b = (warp / kGemvTokTile) * kBlkPerWarp + lane;
                            float v[16], m = 0.0f;
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                v[i] = s_hx[row * kFeatGU + 16 * b + i];
                                m = fmaxf(m, fabsf(v[i]));
                            }
                            const float gs2 = a.is2[e];
                            uint32_t sbyte = 0, q0 = 0, q1 = 0;
                            if (gs2 > 0.0f) {
                                sbyte = f32_to_e4m3(__fdiv_rn(__fdiv_rn(m, 6.0f), gs2));
                                const float S = e4m3_to_f32(sbyte);
                                if (S != 0.0f) {
                                    const float den = __fmul_rn(S, gs2), rden = __frcp_rn(den);
#pragma unroll
                                    for (int i = 0; i < 8; i += 2) {
                                        q0 |= e2m1x2_byte(e2m1_quotient(v[i], den, rden),
                                                          e2m1_quotient(v[i + 1], den, rden)) << (4 * i);
                                        q1 |= e2m1x2_byte(e2m1_quotient(v[8 + i], den, rden),
                                                          e2m1_quotient(v[9 + i], den, rden)) << (4 * i);
                                    }
                                }
                            }
                            const size_t r = (size_t)(cur.row0 + row);
                            const int fb = h.f + 16 * b;
                            *reinterpret_cast<uint2*>(a.hq + r * (a.F / 2) + fb / 2) = make_uint2(q0, q1);
                            a.hs[r * (a.F / 16) + fb / 16] = (uint8_t)sbyte;
                        }
                        consumer_sync();  // s_hx is rewritten by the next block
                    }
                } else {
                    // lane (g, c): outputs n0 + g and n0 + g + 8 for rows 2c + cc
                    const int n0 = h.f + 16 * warp;
                    const float wd = a.down_ws2[e];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int col = 2 * c + cc;
                        if (col < cur.nrows) {
                            const int r = cur.row0 + col;
                            const float rs = BMODE == B_BF16 ? s_rowscale[col] : a.is2[e];
                            const float wt = a.topk_w[a.row_to_slot[r]];
                            a.yrows[(size_t)r * a.d + n0 + g] = wt * __fmul_rn(__fmul_rn(t[cc], rs), wd);
                            a.yrows[(size_t)r * a.d + n0 + g + 8] = wt * __fmul_rn(__fmul_rn(t[2 + cc], rs), wd);
                        }
                    }
                }
                __threadfence();
            }

            if (h.j == h.nst - 1) {
                // ---- the item is complete ----
                consumer_sync();  // every epilogue write of the item is done (and fenced)
                if (!down) {
                    if (threadIdx.x == 0) atomicAdd(a.tile_ready + cur.tile, 1);
                } else {
                    if (threadIdx.x < kGemvTokTile) {
                        int t = -1;
                        if (threadIdx.x < cur.nrows) {
                            const int tt = a.row_to_slot[cur.row0 + threadIdx.x] / a.top_k;
                            if (atomicAdd(a.tok_done + (size_t)tt * ngd + cur.grp, 1) == a.top_k - 1) t = tt;
                        }
                        s_fin[threadIdx.x] = t;
                    }
                    consumer_sync();
                    const int n_out = a.gbd * kRows, f0 = cur.grp * n_out;
                    for (int i = 0; i < cur.nrows; ++i) {
                        const int t = s_fin[i];
                        if (t < 0) continue;
                        __threadfence();
                        for (int n = f0 + threadIdx.x; n < f0 + n_out; n += kConsumers * 32) {
                            float v = 0.0f;
                            for (int j = 0; j < a.top_k; ++j)
                                v += __ldcg(a.yrows + (size_t)a.slot_to_row[t * a.top_k + j] * a.d + n);
                            a.out[(size_t)t * a.d + n] = f32_to_bf16_bits(v);
                        }
                    }
                }
            }
            ++st;
        }
    }
    grid_dep_launch();
}

template <int BMODE, int CKG, int CKD>
void launch_t(const DecodeArgs& a, size_t smem, cudaStream_t s, const char* name) {
    auto kern = decode_kernel<BMODE, CKG, CKD>;
    // opt in to exactly the dynamic shared memory this shape needs (asking for
    // more than the limit minus the static shared memory fails)
    static size_t opted = 48 * 1024;
    if (smem > opted) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return;
        opted = smem;
    }
    NVFP4_LAUNCH(name, s, launch_pdl(kern, dim3(num_sms()), dim3(kThreads), smem, s, a));
}

template <int BMODE>
void launch_b(const DecodeArgs& a, size_t smem, cudaStream_t s, const char* name) {
    launch_t<BMODE, kChunk, kChunk>(a, smem, s, name);
}

int slot_bytes(int d, int F) {
    (void)d;
    (void)F;
    return kRows * kChunk * 9 / 16;
}

size_t decode_smem(int d, int F) {
    return 128 + (size_t)kNS * slot_bytes(d, F) + (size_t)kGemvTokTile * std::max(d, F) * 2 +
           (size_t)kGemvTokTile * kFeatGU * 4;
}

// Blocks per item: the most (a divisor of nb) that still gives every SM
// about `per_sm` items over `tiles` row tiles.
int pick_blocks(int tiles, int nb, int per_sm) {
    int best = 1;
    for (int g = 1; g <= nb; ++g)
        if (nb % g == 0 && (long long)tiles * (nb / g) >= (long long)per_sm * num_sms()) best = g;
    return best;
}

}  // namespace

bool decode_supported(int d, int F) {
    // the dynamic shared memory plus about 0.5 KB of static shared memory
    // within the 227 KB a CTA may opt in to
    return d % kChunk == 0 && F % kChunk == 0 && d % kRows == 0 && F % kFeatGU == 0 &&
           decode_smem(d, F) + 1024 <= 227 * 1024;
}

int decode_groups_d(int d) { return std::max(1, d / kRows); }

bool decode_set_maps(DecodeArgs* a, const nvfp4_moe_weights* w) {
    const unsigned long long E = (unsigned long long)w->E, d = a->d, F = a->F;
    return encode_tmap_u8(&a->tm_gate_c, w->gate.codes, d / 2, E * F, kChunk / 2, kFeatGU, false) &&
           encode_tmap_u8(&a->tm_up_c, w->up.codes, d / 2, E * F, kChunk / 2, kFeatGU, false) &&
           encode_tmap_u8(&a->tm_gate_s, w->gate.scales, d / 16, E * F, kChunk / 16, kFeatGU, false) &&
           encode_tmap_u8(&a->tm_up_s, w->up.scales, d / 16, E * F, kChunk / 16, kFeatGU, false) &&
           encode_tmap_u8(&a->tm_down_c, w->down.codes, F / 2, E * d, kChunk / 2, kRows, false) &&
           encode_tmap_u8(&a->tm_down_s, w->down.scales, F / 16, E * d, kChunk / 16, kRows, false);
}

void decode_pick_groups(int expected_tiles, int d, int F, int* gbu, int* gbd) {
    *gbu = pick_blocks(expected_tiles, F / kFeatGU, 12);
    *gbd = pick_blocks(expected_tiles, d / kRows, 12);
}

void launch_decode(int bmode, const DecodeArgs& args, cudaStream_t s) {
    DecodeArgs a = args;
    a.slot_bytes = slot_bytes(a.d, a.F);
    const size_t smem = decode_smem(a.d, a.F);
    if (bmode == B_BF16) launch_b<B_BF16>(a, smem, s, "gemv_gateup_down_w4a16");
    else launch_b<B_NVFP4>(a, smem, s, "gemv_gateup_down_w4a4");
}

}  // namespace nvfp4
