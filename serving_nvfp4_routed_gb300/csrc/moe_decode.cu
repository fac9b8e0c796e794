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
//   * one CTA per SM; work items come from two device counters in runs of
//     consecutive items: every gate/up item (expert row tile of up to 8
//     routed rows x a group of 128-feature blocks), then every down item
//     (row tile x a group of 256-output blocks); a CTA stages a row tile's
//     rows once for the consecutive items it takes on that tile;
//   * a producer warp loads each stage -- 256 weight rows (128 gate + 128
//     up rows of one feature block, or 256 down rows) x 256 K of the stored
//     codes and scales -- with tiled TMA into a ring of shared-memory slots
//     (codes with the 128-byte swizzle), running ahead across items;
//   * each of eight consumer warps owns 32 of the stage's rows as two m16
//     tiles (gate/up: 8 gate + 8 up rows of the same features per tile, so
//     that SwiGLU stays in its registers) over every K chunk of the block:
//     no partial sums to exchange.  It loads its codes and scales from
//     shared memory into mma.sync m16n8k16 A fragments (K permuted inside
//     each 256-wide chunk so that every lane's codes are contiguous; the B
//     rows use the same permutation), dequantises them in registers (cvt
//     e2m1x2 -> f16x2, times the block scale: exact) and multiplies the row
//     tile's routed rows, staged in shared memory as f16 (bf16 rows with a
//     per-row power of two taken out, or NVFP4 rows dequantised exactly);
//     each B fragment serves both tiles;
//   * gate/up writes h = bf16(silu(G) * U) (W4A4: requantised to NVFP4 under
//     the down input scale: a warp's 16 features are one NVFP4 block) and,
//     once an item is done, raises its row tile's counter;
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
#include "decode.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {

namespace {

using namespace tc;

constexpr int kConsumers = 8;                    // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;  // + one producer warp
constexpr int kNS = 4;                           // ring slots
constexpr int kWarpRows = 32;                    // weight rows per consumer warp: two m16 tiles
constexpr int kRows = kWarpRows * kConsumers;    // weight rows per stage
constexpr int kFeatGU = kRows / 2;               // features per gate/up block (128 gate + 128 up rows)
constexpr int kChunk = 256;                      // K per stage (one 128-byte box row of codes)
constexpr int kBarConsumers = 1;                 // named barrier of the consumer warps
// Measured on GB300 (one CTA per SM): the layer is bound by the consumer
// warps' instruction issue, not by the TMA stream (which alone reaches
// about 90 % of the copy bandwidth).  A warp therefore takes 32 rows as two
// m16 tiles: each B fragment it loads serves both, and the per-stage work
// of a warp (wait, header, release) is spread over twice the weights.

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

// A lane's codes of one stage row (CK = 256: 32 bytes, the 16-byte chunks
// 2c and 2c + 1 of the 128-byte row, stored by TMA with the 128-byte swizzle:
// chunk q of local row r at q ^ (r & 7), r & 7 == g for every warp's rows, so
// that the eight rows a quarter warp reads land in distinct bank groups).
template <int CK>
__device__ __forceinline__ void lds_codes(const uint8_t* row, int g, int c, uint32_t* w) {
    if constexpr (CK == 256) {
        const uint4 u0 = *reinterpret_cast<const uint4*>(row + (((2 * c) ^ g) << 4));
        const uint4 u1 = *reinterpret_cast<const uint4*>(row + (((2 * c + 1) ^ g) << 4));
        w[0] = u0.x; w[1] = u0.y; w[2] = u0.z; w[3] = u0.w;
        w[4] = u1.x; w[5] = u1.y; w[6] = u1.z; w[7] = u1.w;
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(row + 8 * c);
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

// One warp's share of a stage: two m16 tiles; tile t takes its MMA rows g
// and g + 8 from the 128-byte code rows cr[t][0] and cr[t][1] (swizzled) and
// the 16-byte scale rows sr[t][0] and sr[t][1].  The stage covers K
// [k0, k0 + 256) of the staged B rows (row length K); k-step i of tile t
// accumulates into acc[t][i & 1].
__device__ __forceinline__ void stage_mma2(const uint8_t* const (&cr)[2][2], const uint8_t* const (&sr)[2][2], int k0,
                                           const uint4* Bs, int K, int lane, float (&acc)[2][2][4]) {
    using C = Ch<kChunk>;
    const int g = lane >> 2, c = lane & 3;
    uint32_t w[2][2][C::CW];
    uint32_t S[2][2][4];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            lds_codes<kChunk>(cr[t][r], g, c, w[t][r]);
            block_scales<4>(lds_scales<kChunk>(sr[t][r] + 4 * c), S[t][r]);
        }
    const uint4* brow = Bs + (size_t)g * (K / 8);
    const int qb = (k0 + c * C::TS) / 8;
#pragma unroll
    for (int jj = 0; jj < C::KS; jj += 2) {
        const uint4 bq = brow[bsw<kChunk>(qb + jj / 2, g)];
        const uint32_t b0[2] = {bq.x, bq.y};
        const uint32_t b1[2] = {bq.z, bq.w};
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            uint32_t x0[4], x1[4];
            deq_word(w[t][0][jj >> 1], S[t][0][jj >> 2], x0);
            deq_word(w[t][1][jj >> 1], S[t][1][jj >> 2], x1);
            const uint32_t af0[4] = {x0[0], x1[0], x0[1], x1[1]};
            const uint32_t af1[4] = {x0[2], x1[2], x0[3], x1[3]};
            mma_16816(acc[t][0], af0, b0);
            mma_16816(acc[t][1], af1, b1);
        }
    }
}

template <int BMODE, int CKG, int CKD>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ DecodeArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the 128-byte swizzle repeats every 1024 bytes: slots start on that boundary
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint4* Bs = reinterpret_cast<uint4*>(ring + (size_t)kNS * a.slot_bytes);
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
            // items come in runs of consecutive indices (a.chu gate/up items,
            // then a.chd down items per grab), so that a CTA mostly keeps one
            // row tile's staged rows; every gate/up item is handed out before
            // the first down item
            int next = 0, run_end = 0;
            bool down_phase = false;
            for (;;) {
                int item = total;
                if (next < run_end) {
                    item = next++;
                } else {
                    if (!down_phase) {
                        const int b = atomicAdd(a.counters, a.chu);
                        if (b < nA) {
                            next = b;
                            run_end = min(nA, b + a.chu);
                            item = next++;
                        } else {
                            down_phase = true;
                        }
                    }
                    if (down_phase) {
                        const int b = atomicAdd(a.counters + 1, a.chd);
                        if (b < total - nA) {
                            next = nA + b;
                            run_end = nA + min(total - nA, b + a.chd);
                            item = next++;
                        }
                    }
                }
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
        float acc[2][2][4];  // [tile][chain][fragment]
        long long st = 0;
        int par = 0;
        int staged_tile = -1, staged_kind = -1;  // the rows now in Bs
        Hdr cur{};
        for (;;) {
            const int s = (int)(st % kNS);
            if (!warp_wait(smem_u32(&bar_full[s]), (uint32_t)((st / kNS) & 1), abort_flag, a.status) || *abort_flag)
                break;
            const Hdr h = s_hdr[s];
            if (h.kind < 0) break;
            const bool down = h.kind == 1;
            if (h.j == 0) cur = h;
            if (h.j == 0 && (h.tile != staged_tile || h.kind != staged_kind)) {
                // ---- a new row tile: stage its routed rows ----
                staged_tile = h.tile;
                staged_kind = h.kind;
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
            // ---- this warp's 32 rows of the stage ----
            const int nch = down ? nchd : nchu;
            if (h.kc == 0) {
#pragma unroll
                for (int t = 0; t < 2; ++t)
#pragma unroll
                    for (int q = 0; q < 2; ++q)
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[t][q][i] = 0.0f;
            }
            const uint8_t* slot = ring + (size_t)s * a.slot_bytes;
            if (!down) {
                // tile t: MMA rows 0-7 are gate rows 16w + 8t .. + 7 of the
                // block, rows 8-15 the up rows of the same features
                const int cb = kFeatGU * kChunk / 2, sb = kFeatGU * kChunk / 16;
                const int r0 = kWarpRows / 2 * warp + g;
                const uint8_t* const cr[2][2] = {{slot + r0 * (kChunk / 2), slot + cb + r0 * (kChunk / 2)},
                                                 {slot + (r0 + 8) * (kChunk / 2), slot + cb + (r0 + 8) * (kChunk / 2)}};
                const uint8_t* const sr[2][2] = {
                    {slot + 2 * cb + r0 * (kChunk / 16), slot + 2 * cb + sb + r0 * (kChunk / 16)},
                    {slot + 2 * cb + (r0 + 8) * (kChunk / 16), slot + 2 * cb + sb + (r0 + 8) * (kChunk / 16)}};
                stage_mma2(cr, sr, h.kc * kChunk, Bs, a.d, lane, acc);
            } else {
                // tile t: MMA rows g and g + 8 are rows 32w + 16t + g and + 8
                const int cb = kRows * kChunk / 2;
                const int r0 = kWarpRows * warp + g;
                const uint8_t* const cr[2][2] = {
                    {slot + r0 * (kChunk / 2), slot + (r0 + 8) * (kChunk / 2)},
                    {slot + (r0 + 16) * (kChunk / 2), slot + (r0 + 24) * (kChunk / 2)}};
                const uint8_t* const sr[2][2] = {
                    {slot + cb + r0 * (kChunk / 16), slot + cb + (r0 + 8) * (kChunk / 16)},
                    {slot + cb + (r0 + 16) * (kChunk / 16), slot + cb + (r0 + 24) * (kChunk / 16)}};
                stage_mma2(cr, sr, h.kc * kChunk, Bs, a.F, lane, acc);
            }
            // the slot is refilled by TMA (async proxy) after its release
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar_empty[s]));

            if (h.kc == nch - 1) {
                // ---- this warp's rows of the block are complete: epilogue ----
                float t4[2][4];
#pragma unroll
                for (int t = 0; t < 2; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i) t4[t][i] = acc[t][0][i] + acc[t][1][i];
                const int e = cur.e;
                if (!down) {
                    // lane (g, c), tile t: feature f + 16w + 8t + g; gate in
                    // t4[t][cc], up in t4[t][2 + cc] for row 2c + cc
                    const int f0 = h.f + kWarpRows / 2 * warp;
                    const float wg = a.gate_ws2[e], wu = a.up_ws2[e];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int col = 2 * c + cc;
                        const bool valid = col < cur.nrows;
                        const float rs = BMODE == B_BF16 ? (valid ? s_rowscale[col] : 0.0f) : a.is13[e];
                        float hv[2];
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const float G = round_bf16(__fmul_rn(__fmul_rn(t4[t][cc], rs), wg));
                            const float U = round_bf16(__fmul_rn(__fmul_rn(t4[t][2 + cc], rs), wu));
                            hv[t] = valid ? round_bf16(G / (1.0f + expf(-G)) * U) : 0.0f;
                            if constexpr (BMODE == B_BF16) {
                                if (valid) a.h[(size_t)(cur.row0 + col) * a.F + f0 + 8 * t + g] = f32_to_bf16_bits(hv[t]);
                            }
                        }
                        if constexpr (BMODE == B_NVFP4) {
                            // the warp's 16 features are one NVFP4 block of h
                            // for each row: tile t, lane g holds feature 8t + g
                            const float gs2 = a.is2[e];
                            float m = fmaxf(fabsf(hv[0]), fabsf(hv[1]));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                            uint32_t sbyte = 0, q[2] = {0u, 0u};
                            if (gs2 > 0.0f) {
                                sbyte = f32_to_e4m3(__fdiv_rn(__fdiv_rn(m, 6.0f), gs2));
                                const float S = e4m3_to_f32(sbyte);
                                if (S != 0.0f) {
                                    const float den = __fmul_rn(S, gs2), rden = __frcp_rn(den);
                                    const uint32_t byte = e2m1x2_byte(e2m1_quotient(hv[0], den, rden),
                                                                      e2m1_quotient(hv[1], den, rden));
                                    q[0] = byte & 0xFu;
                                    q[1] = byte >> 4;
                                }
                            }
                            // byte k of the block: features 2k, 2k + 1 (tile k / 4,
                            // lanes g = 2 (k % 4) and + 1); lane g = 0 gathers all eight
                            uint32_t by[2];
#pragma unroll
                            for (int t = 0; t < 2; ++t)
                                by[t] = q[t] | (__shfl_down_sync(0xffffffffu, q[t], 4) << 4);
                            uint32_t wd[2];
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                wd[t] = by[t];
#pragma unroll
                                for (int k = 1; k < 4; ++k) wd[t] |= __shfl_sync(0xffffffffu, by[t], c + 8 * k) << (8 * k);
                            }
                            if (valid && g == 0) {
                                const size_t r = (size_t)(cur.row0 + col);
                                *reinterpret_cast<uint2*>(a.hq + r * (a.F / 2) + f0 / 2) = make_uint2(wd[0], wd[1]);
                                a.hs[r * (a.F / 16) + f0 / 16] = (uint8_t)sbyte;
                            }
                        }
                    }
                } else {
                    // lane (g, c), tile t: outputs n0 + 16t + g and + 8 for rows 2c + cc
                    const int n0 = h.f + kWarpRows * warp;
                    const float wd = a.down_ws2[e];
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int col = 2 * c + cc;
                        if (col < cur.nrows) {
                            const int r = cur.row0 + col;
                            const float rs = BMODE == B_BF16 ? s_rowscale[col] : a.is2[e];
                            const float wt = a.topk_w[a.row_to_slot[r]];
                            float* yr = a.yrows + (size_t)r * a.d + n0 + g;
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                yr[16 * t] = wt * __fmul_rn(__fmul_rn(t4[t][cc], rs), wd);
                                yr[16 * t + 8] = wt * __fmul_rn(__fmul_rn(t4[t][2 + cc], rs), wd);
                            }
                        }
                    }
                }
            }

            if (h.j == h.nst - 1) {
                // ---- the item is complete ----
                // every epilogue write of the item is done; the barrier plus a
                // gpu-scope fence before each counter update publishes them
                // (release), and readers fence after seeing the count (acquire)
                consumer_sync();
                if (!down) {
                    if (threadIdx.x == 0) {
                        __threadfence();
                        atomicAdd(a.tile_ready + cur.tile, 1);
                    }
                } else {
                    if (threadIdx.x < kGemvTokTile) {
                        int t = -1;
                        if (threadIdx.x < cur.nrows) {
                            const int tt = a.row_to_slot[cur.row0 + threadIdx.x] / a.top_k;
                            __threadfence();
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
    return 1024 + (size_t)kNS * slot_bytes(d, F) + (size_t)kGemvTokTile * std::max(d, F) * 2;
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
    return encode_tmap_u8(&a->tm_gate_c, w->gate.codes, d / 2, E * F, kChunk / 2, kFeatGU, true) &&
           encode_tmap_u8(&a->tm_up_c, w->up.codes, d / 2, E * F, kChunk / 2, kFeatGU, true) &&
           encode_tmap_u8(&a->tm_gate_s, w->gate.scales, d / 16, E * F, kChunk / 16, kFeatGU, false) &&
           encode_tmap_u8(&a->tm_up_s, w->up.scales, d / 16, E * F, kChunk / 16, kFeatGU, false) &&
           encode_tmap_u8(&a->tm_down_c, w->down.codes, F / 2, E * d, kChunk / 2, kRows, true) &&
           encode_tmap_u8(&a->tm_down_s, w->down.scales, F / 16, E * d, kChunk / 16, kRows, false);
}

void decode_pick_work(int expected_tiles, DecodeArgs* a) {
    const int nbu = a->F / kFeatGU, nbd = a->d / kRows;
    a->gbu = pick_blocks(expected_tiles, nbu, 12);
    a->gbd = pick_blocks(expected_tiles, nbd, 12);
    // about six grabs per CTA and phase, never more than one tile's items
    const long long n_u = (long long)expected_tiles * (nbu / a->gbu), n_d = (long long)expected_tiles * (nbd / a->gbd);
    a->chu = (int)std::max(1LL, std::min<long long>(nbu / a->gbu, n_u / (6LL * num_sms())));
    a->chd = (int)std::max(1LL, std::min<long long>(nbd / a->gbd, n_d / (6LL * num_sms())));
}

void launch_decode(int bmode, const DecodeArgs& args, cudaStream_t s) {
    DecodeArgs a = args;
    a.slot_bytes = slot_bytes(a.d, a.F);
    const size_t smem = decode_smem(a.d, a.F);
    if (bmode == B_BF16) launch_b<B_BF16>(a, smem, s, "gemv_gateup_down_w4a16");
    else launch_b<B_NVFP4>(a, smem, s, "gemv_gateup_down_w4a4");
}

}  // namespace nvfp4
