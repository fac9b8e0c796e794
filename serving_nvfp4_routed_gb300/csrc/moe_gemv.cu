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
//   * work item = (expert, 16 x 8 / ksplit output features (down: up to 8
//     such blocks), up to 8 routed rows); a CTA's first item is its own
//     index, the others come from an atomic counter so that CTAs stay busy;
//     the routing metadata sits in shared memory, so that an item's decode
//     does no dependent global loads;
//   * each warp takes 16 output features; when too few items exist to fill
//     the GPU, ksplit warps split K and their partial sums (mma.sync
//     m16n8k16, f32 accumulate) meet in shared memory;
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
//   * epilogues: SwiGLU to bf16 h, SwiGLU + NVFP4 requantisation of h with
//     the down input_scale (W4A4), or (down projection) w * y per routed row
//     in fp32; the CTA that completes a token's last slot in a group of
//     outputs sums the token's k rows there in slot order (deterministic).
#include <type_traits>

#include "common.cuh"
#include "gemv.cuh"
#include "tc_ptx.cuh"

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


// Shared-memory layout of the staged B rows: row g holds K f16 values as K/8
// 16-byte granules; granule q is stored at bsw(q, g) so that the B-fragment
// reads of a warp (lane (g, c) reads granule c*CK/32 + j of its row) hit 8
// distinct 16-byte bank groups in every quarter-warp phase.
template <int CK>
__device__ __forceinline__ int bsw(int q, int g) {
    if constexpr (CK == 256) return q ^ ((((q >> 3) & 3) << 1) | (g & 1));
    else return q ^ (g & 1);
}

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Shared-memory weight ring of the routed down projection (one projection,
// 256-wide chunks): per warp kRingSlots slots of one chunk of its 16 rows
// (codes, then scales), filled with cp.async by the lanes that read them.
constexpr int kRingSlots = 4;
constexpr int kRingSlotBytes = 2 * 32 * 32 + 2 * 32 * 4;  // 2304
__host__ __device__ constexpr size_t ring_bytes() { return (size_t)kWarps * kRingSlots * kRingSlotBytes; }
// Dynamic shared memory: the row stage [kGemvTokTile][K] f16, the ring
// (kWarps x kRingSlots x 2304 B = 72 KB), the routing metadata (3 E + 2 ints).
__host__ __device__ constexpr size_t gemv_smem_bytes_dev(int K) { return (size_t)kGemvTokTile * K * 2; }
size_t meta_bytes(int E) { return ((size_t)(3 * E + 2) * 4 + 15) / 16 * 16; }
// The ring is used while two CTAs' row stage, ring and metadata (and ~4 KB
// of static shared memory each) fit in an SM: K up to ~2300 at E = 288.
bool ring_fits(int K, int E) {
    return 2 * (gemv_smem_bytes_dev(K) + ring_bytes() + meta_bytes(E) + 4096) <= 227 * 1024;
}
struct Item {
    int e, row0, nrows, fb, fb_end;  // feature blocks [fb, fb_end) share the staged rows
};

template <int CK, int BMODE, int OUTMODE, int NPROJ, bool RING = false>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const __grid_constant__ GemvArgs a) {
    using C = Chunk<CK>;
    // U chunks form a batch of weight loads; NBUF batches live in registers
    // as a ring, so that NBUF - 1 batches are in flight while one is consumed
    // (the next work item's first batches go out before the epilogue).  The
    // routed down projection keeps its batches in a shared-memory ring
    // instead (cp.async; no registers held by the loads in flight), four
    // slots deep: measured on GB300 its register ring left it bound by the
    // latency of its weight loads at two batches in flight.
    constexpr int U = 1;
    constexpr bool kRing = RING;
    static_assert(!RING || (OUTMODE == OUT_COMBINE && NPROJ == 1 && CK == 256), "the ring serves the down GEMV");
    constexpr int NBUF = kRing ? kRingSlots : (NPROJ == 2 ? 2 : 3);
    extern __shared__ uint4 Bs[];          // [kGemvTokTile][K/8] granules of f16
    __shared__ float s_red[kWarps - 1][NPROJ * 4][32];
    __shared__ float s_rowscale[kGemvTokTile];
    __shared__ unsigned s_amax[kGemvTokTile];
    __shared__ int s_next;
    __shared__ int s_fin[kGemvTokTile];
    __shared__ float s_wt[kGemvTokTile];  // OUT_COMBINE: the routing weight of each of the item's rows
    __shared__ int s_nact;

    // The routed layer's down projection (OUT_COMBINE) takes its first item
    // and starts that item's weight loads before it waits for the gate/up
    // launch: its routing arrays and work counter come from the route launch
    // before that one, complete by the time any gate/up CTA lets dependents
    // start; only the h rows it stages need the wait.
    constexpr bool kEarly = OUTMODE == OUT_COMBINE;
    if constexpr (!kEarly) grid_dep_wait();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    // The B-fragment reads of a chunk hit granules qb + j (qb = this lane's
    // first granule of the chunk, a multiple of 8 for CK = 256 and of 2 for
    // CK = 64; j < 8): there bsw() flips the low bits of j by a mask fixed
    // per lane, so the reads address qb + (j ^ kP).
    const int kP = CK == 256 ? ((c << 1) | (g & 1)) : (g & 1);
    const int KSPL = a.ksplit, WF = kWarps / KSPL;
    const int wf = warp / KSPL, ks = warp % KSPL;

    // the routing metadata, loaded once per CTA into the dynamic shared
    // memory after the row stage and the ring (an item's decode is then free
    // of dependent global loads): tile starts [E + 1], active experts [E],
    // row offsets [E + 1]
    int* s_ts = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(Bs) + gemv_smem_bytes_dev(a.K) +
                                       (kRing ? ring_bytes() : 0));
    int* s_act = s_ts + (a.E + 1);
    int* s_off = s_act + a.E;
    for (int i = tid; i <= a.E; i += kThreads) {
        s_ts[i] = a.tile_start[i];
        s_off[i] = a.offsets[i];
        if (i < a.E) s_act[i] = a.active[i];
    }
    if (tid == 0) s_nact = *a.n_active;
    if (tid < kGemvTokTile) s_amax[tid] = 0u;
    __syncthreads();
    const int n_active = s_nact;
    const int total_tiles = s_ts[n_active];
    const int FB = 16 * WF;
    const int n_fb = a.N / FB;
    const int G = a.fb_group > 0 ? a.fb_group : 1;  // feature blocks per work item
    const int n_grp = (n_fb + G - 1) / G;
    const int total = total_tiles * n_grp;
    const int nch = a.K / CK;
    const int Kg = a.K / 8;
    const size_t K2 = (size_t)a.K / 2, K16 = (size_t)a.K / 16;

    auto decode = [&](int item, Item& it) {
        it.fb = (item % n_grp) * G;
        it.fb_end = min(n_fb, it.fb + G);
        const int tile = item / n_grp;
        int lo = 0, hi = n_active;  // largest ai with tile_start[ai] <= tile
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_ts[mid] <= tile) lo = mid; else hi = mid;
        }
        it.e = s_act[lo];
        it.row0 = s_off[it.e] + (tile - s_ts[lo]) * kGemvTokTile;
        it.nrows = min(kGemvTokTile, s_off[it.e + 1] - it.row0);
    };

    // L2 prefetch (one thread, K not split over warps): chunk ch of the
    // item's feature rows of block fb, every projection, codes and scales;
    // past the block's last chunk, the item's next block
    auto l2_prefetch = [&](const Item& it, int fb, int ch) {
        if constexpr (CK == 256) {
            if (ch >= nch) {
                ch -= nch;
                ++fb;
            }
            if (ch < nch && fb < it.fb_end) {
                const int y = it.e * a.N + fb * FB;
#pragma unroll
                for (int p = 0; p < NPROJ; ++p) {
                    tc::tma_prefetch_2d(&a.pf_codes[p], ch * (CK / 2), y);
                    tc::tma_prefetch_2d(&a.pf_scales[p], ch * (CK / 16), y);
                }
            }
        }
    };
    uint32_t acw[kRing ? 1 : NBUF][U][NPROJ][2][C::CW];
    uint32_t asw[kRing ? 1 : NBUF][U][NPROJ][2];
    // ring slot b of this warp: codes [row half][lane][32 B] (the two 16-byte
    // halves of lane l at h ^ bit 2 of l: conflict-free 16-byte reads), then
    // scales [row half][lane][4 B]
    uint8_t* wring = reinterpret_cast<uint8_t*>(Bs + (size_t)kGemvTokTile * (a.K / 8)) +
                     (size_t)warp * kRingSlots * kRingSlotBytes;
    const int hsw = ((lane >> 2) & 1) << 4;
    auto load_batch = [&](auto buf, const Item& it, int chb) {
        constexpr int B = decltype(buf)::value;
        const int n0 = it.fb * FB + wf * 16;
        if constexpr (kRing) {
            // one commit group per call, empty past the end, so that a
            // batch is complete once NBUF - 1 later groups were committed
            const int ch = chb;
            if (a.pf_dist > 0 && tid == 0) l2_prefetch(it, it.fb, chb + a.pf_dist);
            if (ch < nch) {
                uint8_t* sl = wring + B * kRingSlotBytes;
                const size_t kb = (size_t)ch * CK + (size_t)c * C::TS;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const size_t row = (size_t)it.e * a.N + n0 + g + 8 * hf;
                    const uint8_t* src = a.a_codes[0] + row * K2 + kb / 2;
                    uint8_t* dst = sl + hf * 1024 + lane * 32;
                    tc::cp_async16(tc::smem_u32(dst + hsw), src, 16);
                    tc::cp_async16(tc::smem_u32(dst + (16 - hsw)), src + 16, 16);
                    tc::cp_async4(tc::smem_u32(sl + 2048 + hf * 128 + lane * 4), a.a_scales[0] + row * K16 + kb / 16);
                }
            }
            tc::cp_async_commit();
        } else {
            // (the CTA's chunks at that distance are the KSPL consecutive
            // ones; lane 0 of warp chb % 8 issues them, so that the warps
            // share the extra instructions)
            if (a.pf_dist > 0 && tid == 32 * (chb % kWarps))
                for (int q = 0; q < KSPL; ++q) l2_prefetch(it, it.fb, chb + a.pf_dist * KSPL + q);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int ch = chb + u * KSPL;
                if (ch < nch) {
                    const size_t kb = (size_t)ch * CK + (size_t)c * C::TS;
#pragma unroll
                    for (int p = 0; p < NPROJ; ++p)
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const size_t row = (size_t)it.e * a.N + n0 + g + 8 * hf;
                            load_codes<CK>(a.a_codes[p] + row * K2 + kb / 2, acw[B][u][p][hf]);
                            asw[B][u][p][hf] = load_scales<CK>(a.a_scales[p] + row * K16 + kb / 16);
                        }
                }
            }
        }
    };
    // the first NBUF - 1 batches of an item's (or feature block's) weights
    auto prefetch = [&](const Item& it) {
        load_batch(std::integral_constant<int, 0>{}, it, ks);
        if constexpr (NBUF > 2) load_batch(std::integral_constant<int, 1>{}, it, ks + U * KSPL);
        if constexpr (NBUF > 3) load_batch(std::integral_constant<int, 2>{}, it, ks + 2 * U * KSPL);
    };

    // the first item is the CTA's own index, the others come from the counter
    int item = blockIdx.x;
    Item cur{};
    if (item < total) {
        decode(item, cur);
        if (a.pf_dist > 0 && tid == 0)
            for (int ch = KSPL; ch < (a.pf_dist + 1) * KSPL; ++ch) l2_prefetch(cur, cur.fb, ch);
        prefetch(cur);
    }
    if constexpr (kEarly) grid_dep_wait();

    while (item < total) {
        // ---- the item's per-expert scales and (down) its rows' routing
        // weights, loaded once here for every epilogue of the item
        float it_ws[NPROJ];
#pragma unroll
        for (int p = 0; p < NPROJ; ++p) it_ws[p] = a.a_ws2[p][cur.e];
        const float it_bgs = BMODE == B_NVFP4 ? a.b_gs[cur.e] : 0.0f;
        const float it_hqgs = OUTMODE == OUT_HQ ? a.hq_gs[cur.e] : 0.0f;
        if constexpr (OUTMODE == OUT_COMBINE) {
            if (tid < cur.nrows) s_wt[tid] = a.topk_w[a.row_to_slot[cur.row0 + tid]];
        }
        // ---- stage the B rows of this item; the warps w with w % nrows == j stage row j
        {
            const int j = warp % cur.nrows, gi = warp / cur.nrows;
            const int gsz = (kWarps - j + cur.nrows - 1) / cur.nrows;
            const int r = cur.row0 + j;
            uint4* dst = Bs + (size_t)j * Kg;
            if constexpr (BMODE == B_BF16) {
                const int brow = a.b_by_token ? (a.row_to_slot ? a.row_to_slot[r] / a.top_k : r) : r;
                const uint4* src = reinterpret_cast<const uint4*>(a.b_bf16 + (size_t)brow * a.K);
                float m = 0.0f;
                for (int q = gi * 32 + lane; q < Kg; q += gsz * 32) {
                    const uint4 u = __ldg(src + q);
                    const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        m = fmaxf(m, fmaxf(fabsf(bf16_bits_to_f32(ww[i] & 0xFFFFu)),
                                           fabsf(bf16_bits_to_f32(ww[i] >> 16))));
                    dst[bsw<CK>(q, j)] = u;
                }
                m = warp_max(m);
                if (lane == 0) atomicMax(&s_amax[j], __float_as_uint(m));
                __syncthreads();
                const int sexp = row_exponent(__uint_as_float(s_amax[j]));
                const float down = exp2i(-sexp);
                if (gi == 0 && lane == 0) s_rowscale[j] = exp2i(sexp);
                for (int q = gi * 32 + lane; q < Kg; q += gsz * 32) {
                    const int qs = bsw<CK>(q, j);
                    const uint4 u = dst[qs];
                    uint4 o;
                    o.x = bf16x2_scaled_to_f16x2(u.x, down);
                    o.y = bf16x2_scaled_to_f16x2(u.y, down);
                    o.z = bf16x2_scaled_to_f16x2(u.z, down);
                    o.w = bf16x2_scaled_to_f16x2(u.w, down);
                    dst[qs] = o;
                }
            } else {
                const uint8_t* codes = a.b_codes + (size_t)r * K2;
                const uint8_t* scales = a.b_scales + (size_t)r * K16;
                for (int b = gi * 32 + lane; b < a.K / 16; b += gsz * 32) {  // 16-block: 8 code bytes, 1 scale
                    const uint2 cw = __ldg(reinterpret_cast<const uint2*>(codes) + b);
                    const uint32_t S = f16x2_bcast(e4m3x2_to_f16x2(__ldg(scales + b)), 0);
                    uint32_t f0[4], f1[4];
                    e2m1x8_to_f16x8(cw.x, f0);
                    e2m1x8_to_f16x8(cw.y, f1);
                    dst[bsw<CK>(2 * b, j)] =
                        make_uint4(hmul2_u32(f0[0], S), hmul2_u32(f0[1], S), hmul2_u32(f0[2], S), hmul2_u32(f0[3], S));
                    dst[bsw<CK>(2 * b + 1, j)] =
                        make_uint4(hmul2_u32(f1[0], S), hmul2_u32(f1[1], S), hmul2_u32(f1[2], S), hmul2_u32(f1[3], S));
                }
            }
        }
        __syncthreads();
        if (tid == 0) {
            const int nx = (int)gridDim.x + atomicAdd(a.work_counter, 1);  // next item, fetched while computing
            s_next = nx;
            // gate/up: a CTA on its last item lets the down launch start
            // filling the SMs that CTAs leave while the last items finish
            // (its CTAs wait for this launch's completion before they read h)
            if (NPROJ == 2 && nx >= total) grid_dep_launch();
        }
        int nitem = total;
        Item nxt{};
        for (;;) {  // the feature blocks of this item, all on the staged rows
            // ---- stream this warp's 16 features over its share of K
            const int n0 = cur.fb * FB + wf * 16;
            // two accumulator chains per projection (odd and even k-steps),
            // summed after the K loop: half the dependent mma.sync chain
            float acc[NPROJ][4], acc2[NPROJ][4];
#pragma unroll
            for (int p = 0; p < NPROJ; ++p)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[p][i] = acc2[p][i] = 0.0f;
            const uint4* brow_s = Bs + (size_t)g * Kg;
            auto compute = [&](auto buf, int chb) {
                constexpr int B = decltype(buf)::value;
                if constexpr (kRing) {
                    // this batch's copies have landed (NBUF - 1 later groups may not have)
                    tc::cp_async_wait<NBUF - 1>();
                    const uint8_t* sl = wring + B * kRingSlotBytes;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const uint4 u0 = *reinterpret_cast<const uint4*>(sl + hf * 1024 + lane * 32 + hsw);
                        const uint4 u1 = *reinterpret_cast<const uint4*>(sl + hf * 1024 + lane * 32 + (16 - hsw));
                        uint32_t* w = acw[0][0][0][hf];
                        w[0] = u0.x; w[1] = u0.y; w[2] = u0.z; w[3] = u0.w;
                        w[4] = u1.x; w[5] = u1.y; w[6] = u1.z; w[7] = u1.w;
                        asw[0][0][0][hf] = *reinterpret_cast<const uint32_t*>(sl + 2048 + hf * 128 + lane * 4);
                    }
                }
                constexpr int BR = kRing ? 0 : B;  // register buffer the batch sits in
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int ch = chb + u * KSPL;
                    if (ch >= nch) break;
                    const int qb = (ch * CK + c * C::TS) / 8;
#pragma unroll
                    for (int jj = 0; jj < C::KS; jj += 2) {
                        const uint4 bq = brow_s[qb + ((jj / 2) ^ kP)];  // = bsw(qb + jj / 2, g)
                        const uint32_t b0[2] = {bq.x, bq.y};
                        const uint32_t b1[2] = {bq.z, bq.w};
#pragma unroll
                        for (int p = 0; p < NPROJ; ++p) {
                            uint32_t r0[4], r1[4];
                            deq_word(acw[BR][u][p][0][jj >> 1], asw[BR][u][p][0], jj, r0);
                            deq_word(acw[BR][u][p][1][jj >> 1], asw[BR][u][p][1], jj, r1);
                            const uint32_t af0[4] = {r0[0], r1[0], r0[1], r1[1]};
                            const uint32_t af1[4] = {r0[2], r1[2], r0[3], r1[3]};
                            mma_16816(acc[p], af0, b0);
                            mma_16816(acc2[p], af1, b1);
                        }
                    }
                }
            };
            // batch b starts at chunk ks + b * step and lives in buffer b % NBUF;
            // batches 0 .. NBUF-2 were loaded by prefetch()
            {
                constexpr std::integral_constant<int, 0> kB0{};
                constexpr std::integral_constant<int, 1> kB1{};
                constexpr std::integral_constant<int, 2 % NBUF> kB2{};
                constexpr std::integral_constant<int, 3 % NBUF> kB3{};
                const int step = U * KSPL;
                // the ring's loads commit a group on every call (empty past the end)
                // the ring's loads of this block: the lane's row pointers
                // once, then one chunk stride per batch (one commit group
                // per call, empty past the end)
                const uint8_t* rcp[2];
                const uint8_t* rsp[2];
                if constexpr (kRing) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const size_t row = (size_t)cur.e * a.N + n0 + g + 8 * hf;
                        rcp[hf] = a.a_codes[0] + row * K2 + c * (C::TS / 2);
                        rsp[hf] = a.a_scales[0] + row * K16 + c * (C::TS / 16);
                    }
                }
                auto load_ahead = [&](auto buf, int ch) {
                    if constexpr (kRing) {
                        constexpr int B = decltype(buf)::value;
                        if (ch < nch) {
                            uint8_t* sl = wring + B * kRingSlotBytes;
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                const uint8_t* src = rcp[hf] + ch * (CK / 2);
                                uint8_t* dst = sl + hf * 1024 + lane * 32;
                                tc::cp_async16(tc::smem_u32(dst + hsw), src, 16);
                                tc::cp_async16(tc::smem_u32(dst + (16 - hsw)), src + 16, 16);
                                tc::cp_async4(tc::smem_u32(sl + 2048 + hf * 128 + lane * 4), rsp[hf] + ch * (CK / 16));
                            }
                        }
                        tc::cp_async_commit();
                    } else {
                        if (ch < nch) load_batch(buf, cur, ch);
                    }
                };
                for (int chb = ks; chb < nch; chb += NBUF * step) {
                    const int ld = (NBUF - 1) * step;  // distance of the batch loaded ahead
                    load_ahead(std::integral_constant<int, NBUF - 1>{}, chb + ld);
                    compute(kB0, chb);
                    if (chb + step >= nch) break;
                    load_ahead(kB0, chb + step + ld);
                    compute(kB1, chb + step);
                    if constexpr (NBUF >= 3) {
                        if (chb + 2 * step >= nch) break;
                        load_ahead(kB1, chb + 2 * step + ld);
                        compute(kB2, chb + 2 * step);
                    }
                    if constexpr (NBUF == 4) {
                        if (chb + 3 * step >= nch) break;
                        load_ahead(kB2, chb + 3 * step + ld);
                        compute(kB3, chb + 3 * step);
                    }
                }
            }
#pragma unroll
            for (int p = 0; p < NPROJ; ++p)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[p][i] += acc2[p][i];
            const bool owner = ks == 0;
            if (KSPL > 1 && !owner) {
#pragma unroll
                for (int p = 0; p < NPROJ; ++p)
#pragma unroll
                    for (int i = 0; i < 4; ++i) s_red[wf * (KSPL - 1) + ks - 1][p * 4 + i][lane] = acc[p][i];
            }
            // (gate/up items are never grouped: known at compile time)
            const bool last = NPROJ == 2 || cur.fb + 1 >= cur.fb_end;
            // Warps that do not split K are independent within a feature block:
            // they meet only to share partial sums (KSPL > 1) and, at an item's
            // last block, to read the next item's index.
            if (KSPL > 1 || last) __syncthreads();

            // ---- the next feature block's (or the next item's) first weight
            // batch goes out before this block's epilogue
            Item following = cur;
            if (!last) {
                following.fb = cur.fb + 1;
                prefetch(following);
            } else {
                nitem = s_next;
                if (nitem < total) {
                    decode(nitem, nxt);
                    if (a.pf_dist > 0 && tid == 0)
                        for (int ch = KSPL; ch < (a.pf_dist + 1) * KSPL; ++ch) l2_prefetch(nxt, nxt.fb, ch);
                    prefetch(nxt);
                }
            }
            if (KSPL > 1 && owner) {
                for (int k2 = 0; k2 < KSPL - 1; ++k2)
#pragma unroll
                    for (int p = 0; p < NPROJ; ++p)
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[p][i] += s_red[wf * (KSPL - 1) + k2][p * 4 + i][lane];
            }

            // ---- epilogue: column cc of this lane is permuted row row0 + 2c + cc
            const int e = cur.e, row0 = cur.row0, nrows = cur.nrows;
            if (owner) {
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int col = 2 * c + cc;
                    const bool valid = col < nrows;
                    const int r = row0 + (valid ? col : 0);
                    float rs;  // takes the accumulator to x W^T (without the tensor scale)
                    if constexpr (BMODE == B_BF16) rs = valid ? s_rowscale[col] : 0.0f;
                    else rs = it_bgs;
                    if constexpr (OUTMODE == OUT_H || OUTMODE == OUT_HQ) {
                        const float wg = it_ws[0], wu = it_ws[NPROJ - 1];
                        float hv[2];
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            const float G = round_bf16(__fmul_rn(__fmul_rn(acc[0][2 * hf + cc], rs), wg));
                            const float Uv = round_bf16(__fmul_rn(__fmul_rn(acc[NPROJ - 1][2 * hf + cc], rs), wu));
                            const float sg = G / (1.0f + expf(-G));
                            hv[hf] = valid ? round_bf16(sg * Uv) : 0.0f;
                        }
                        if constexpr (OUTMODE == OUT_H) {
                            if (valid) {
#pragma unroll
                                for (int hf = 0; hf < 2; ++hf)
                                    a.h_out[(size_t)r * a.N + n0 + g + 8 * hf] = f32_to_bf16_bits(hv[hf]);
                            }
                        } else {
                            // NVFP4 requantisation of h: this warp's 16 features are one block
                            const float gs2 = it_hqgs;
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
                                    const float den = __fmul_rn(S, gs2), rden = __frcp_rn(den);
                                    const uint32_t byte =
                                        e2m1x2_byte(e2m1_quotient(hv[0], den, rden), e2m1_quotient(hv[1], den, rden));
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
                            const float wt = s_wt[col];
                            const float ws = it_ws[0];
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                const float y = __fmul_rn(__fmul_rn(acc[0][2 * hf + cc], rs), ws);
                                a.y_rows[(size_t)r * a.N + n0 + g + 8 * hf] = wt * y;
                            }
                        }
                    } else {  // OUT_BF16
                        if (valid) {
                            const float ws = it_ws[0];
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf)
                                a.y_out[(size_t)r * a.N + n0 + g + 8 * hf] =
                                    f32_to_bf16_bits(__fmul_rn(__fmul_rn(acc[0][2 * hf + cc], rs), ws));
                        }
                    }
                }
            }


            if (last) {
                if constexpr (OUTMODE == OUT_COMBINE) {
                    // every slot of a token meets every item group once: the CTA
                    // that completes a token's k-th slot in this group sums the
                    // token's k rows over the group's outputs in slot order
                    // (the same bits on every run) and writes them as bf16
                    __threadfence();
                    __syncthreads();
                    const int grp = cur.fb / G;
                    if (tid < kGemvTokTile) {
                        int t = -1;
                        if (tid < nrows) {
                            const int tt = a.row_to_slot[row0 + tid] / a.top_k;
                            if (atomicAdd(a.tok_done + (size_t)tt * n_grp + grp, 1) == a.top_k - 1) t = tt;
                        }
                        s_fin[tid] = t;
                    }
                    __syncthreads();
                    const int q0 = grp * G * FB / 4, q1 = min(n_fb, (grp + 1) * G) * FB / 4;
                    for (int i = 0; i < nrows; ++i) {
                        const int t = s_fin[i];
                        if (t < 0) continue;
                        __threadfence();
                        uint2* dst = reinterpret_cast<uint2*>(a.out_bf16 + (size_t)t * a.N);
                        for (int jx = q0 + tid; jx < q1; jx += kThreads) {
                            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                            for (int j = 0; j < a.top_k; ++j) {
                                const float4 y = __ldcg(reinterpret_cast<const float4*>(
                                    a.y_rows + (size_t)a.slot_to_row[t * a.top_k + j] * a.N) + jx);
                                v.x += y.x;
                                v.y += y.y;
                                v.z += y.z;
                                v.w += y.w;
                            }
                            uint2 o;
                            o.x = (uint32_t)f32_to_bf16_bits(v.x) | ((uint32_t)f32_to_bf16_bits(v.y) << 16);
                            o.y = (uint32_t)f32_to_bf16_bits(v.z) | ((uint32_t)f32_to_bf16_bits(v.w) << 16);
                            dst[jx] = o;
                        }
                    }
                }
                break;
            }
            if (KSPL > 1) __syncthreads();  // s_red is read before the next block rewrites it
            cur = following;
        }
        if (tid < kGemvTokTile) s_amax[tid] = 0u;
        __syncthreads();
        item = nitem;
        cur = nxt;
    }
    grid_dep_launch();
}

template <int CK, int BMODE, int OUTMODE, int NPROJ, bool RING = false>
void launch_t(const GemvArgs& a, int max_work, cudaStream_t s, const char* name) {
    auto kern = gemv_kernel<CK, BMODE, OUTMODE, NPROJ, RING>;
    const size_t smem = gemv_smem_bytes(a.K) + (RING ? ring_bytes() : 0) + meta_bytes(a.E);
    // the occupancy probe: the row stage of a typical K (down 1536, gate/up
    // 4096) with the metadata of 288 experts
    const size_t probe = gemv_smem_bytes(RING ? 1536 : 4096) + (RING ? ring_bytes() : 0) + meta_bytes(288);
    // the dynamic shared-memory limit grows to the largest launch so far
    static size_t attr = 0;
    if (std::max(smem, probe) > attr) {
        attr = std::max(smem, probe);
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attr);
    }
    static int per_sm = 0;
    if (per_sm == 0) {
        int v = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kThreads, probe);
        per_sm = v > 0 ? v : 1;
    }
    // the ring kernel runs two CTAs per SM (ring_fits), the others two while
    // the row stage is at most 64 KB
    const int occ = RING ? std::min(per_sm, 2) : (2 * (smem + 8192) <= 227 * 1024 ? per_sm : 1);
    const int grid = std::max(1, std::min(max_work, occ * num_sms()));
    NVFP4_LAUNCH(name, s, launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a));
}

template <int CK>
void launch_ck(int bmode, int outmode, const GemvArgs& a, int max_work, cudaStream_t s) {
    const bool two = a.nproj == 2;
    if (bmode == B_BF16) {
        if (outmode == OUT_H && two) return launch_t<CK, B_BF16, OUT_H, 2>(a, max_work, s, "gemv_gateup_w4a16");
        if (outmode == OUT_COMBINE) {
            if (CK == 256 && ring_fits(a.K, a.E))
                return launch_t<CK, B_BF16, OUT_COMBINE, 1, CK == 256>(a, max_work, s, "gemv_down_w4a16");
            return launch_t<CK, B_BF16, OUT_COMBINE, 1>(a, max_work, s, "gemv_down_w4a16");
        }
        if (outmode == OUT_BF16) return launch_t<CK, B_BF16, OUT_BF16, 1>(a, max_work, s, "gemv_linear_w4a16");
    } else {
        if (outmode == OUT_HQ && two) return launch_t<CK, B_NVFP4, OUT_HQ, 2>(a, max_work, s, "gemv_gateup_w4a4");
        if (outmode == OUT_COMBINE) {
            if (CK == 256 && ring_fits(a.K, a.E))
                return launch_t<CK, B_NVFP4, OUT_COMBINE, 1, CK == 256>(a, max_work, s, "gemv_down_w4a4");
            return launch_t<CK, B_NVFP4, OUT_COMBINE, 1>(a, max_work, s, "gemv_down_w4a4");
        }
    }
}

}  // namespace

size_t gemv_smem_bytes(int K) { return (size_t)kGemvTokTile * K * 2; }

bool gemv_supported_k(int K) { return K > 0 && K % 64 == 0 && K <= 12288; }

// Feature blocks per work item: the down projection (short K) gains from
// staging its rows once for several blocks; gate/up items are long enough.
int gemv_pick_group(int expected_tiles, int N, int ksplit, int nproj) {
    if (nproj != 1) return 1;
    const int n_fb = N / (16 * (kWarps / ksplit));
    const long long want = 4LL * num_sms();  // keep about two items per resident CTA
    int g = 1;
    for (int c = 2; c <= 8; c *= 2)
        if ((long long)expected_tiles * ((n_fb + c - 1) / c) >= want) g = c;
    return g;
}

int gemv_item_groups(int N, int ksplit, int fb_group) {
    const int n_fb = N / (16 * (kWarps / ksplit));
    return (n_fb + fb_group - 1) / fb_group;
}

int gemv_pick_ksplit(int expected_tiles, int N, int nproj) {
    const long long want = num_sms();  // at least one work item per SM before K is split
    // gate/up with fewer than eight 128-feature items per SM (a few tokens):
    // smaller items with K split over the warps, so that the items spread
    // more evenly over the CTAs -- 64 features over two warp halves (T=8:
    // 111 -> 103 µs), 32 features over four warp quarters below two such
    // items per SM (T=2: 76.5 -> 72.6 µs; at T=8 it was slower)
    const long long items128 = (long long)expected_tiles * (N / 128);
    if (nproj == 2 && N % 128 == 0 && items128 >= want && items128 < 8LL * num_sms())
        return items128 < 2LL * num_sms() ? 4 : 2;
    for (int wf = kWarps; wf >= 1; wf >>= 1) {
        const int FB = 16 * wf;
        if (N % FB != 0) continue;
        if ((long long)expected_tiles * (N / FB) >= want) return kWarps / wf;
    }
    return kWarps;  // wf = 1: 16 features per CTA, K split over all warps
}

void launch_gemv(int bmode, int outmode, const GemvArgs& a, int max_work, cudaStream_t s) {
    if (a.K % 256 == 0) launch_ck<256>(bmode, outmode, a, max_work, s);
    else launch_ck<64>(bmode, outmode, a, max_work, s);
}

}  // namespace nvfp4
