// router.cu -- the BF16 router GEMM in front of routing:
//   logits[t, e] = sum_k x[t, k] * W[e, k]      (fp32)
//
// TensorFold issue #308, "The checkpoint": the router is BF16 (not NVFP4);
// its fp32 logits are what moe_route_permute and the layer calls take.
//
// One CTA computes the logits of 128 tokens for EB experts on the tensor
// cores: tcgen05.mma kind::f16 with bf16 A (x rows) and bf16 B (router
// rows), both exactly as stored and moved by TMA with 128-byte swizzle in
// k-stages of 64 (one box each); an fp32 accumulator of EB columns in tensor
// memory.  EB (a multiple of 32 dividing E rounded up to 32, at most 256) is
// the largest that still gives half the SMs a CTA, else 32: a decode batch
// (one token tile) spreads the router matrix over E / 32 CTAs instead of
// streaming it through one SM.  When that still leaves SMs idle, K is split
// over a thread-block cluster of KS <= 8 CTAs: each stores its fp32 partial
// tile in its shared memory and, after a cluster barrier, each CTA sums a
// slice of the tile's rows over the KS partials in rank order through
// distributed shared memory (ld.shared::cluster) -- deterministic, and no
// workspace.  Every bf16 x bf16 product is exact in fp32 and
// the k-sum is fp32.  Warp 0 runs the MMA loop (one elected lane issues),
// warp 1's lane 0 the TMA ring, warps 4-7 read one token per TMEM lane and
// store its logits.  mbarrier waits are bounded and report
// NVFP4_ERR_TIMEOUT through the status word.
#include "common.cuh"
#include "internal.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {

namespace {

using namespace tc;

constexpr int RM = 128;          // tokens per CTA (MMA M)
constexpr int RK = 64;           // k per stage: 128 bytes of bf16, one swizzle row
constexpr int kREGran = 32;      // expert blocks are multiples of this
constexpr int kRMaxE = 512;      // router rows
constexpr int kRMaxEB = 256;     // experts per CTA (one MMA, N <= 256)
constexpr int kRMaxStages = 8;
constexpr int kRThreads = 256;   // warps: 0 MMA, 1 TMA, 4-7 epilogue
constexpr int kRSmemBudget = 200 * 1024;

struct RouterArgs {
    CUtensorMap tmap_x, tmap_w;
    int T, K, E, EB, e_blocks, ksplit, stages, tmem_cols;
    float* logits;
    int32_t* status;
};

// kind::f16 instruction descriptor with bf16 A and B (formats 1), f32 D.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__global__ void __launch_bounds__(kRThreads, 1) router_kernel(const __grid_constant__ RouterArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bar_full[kRMaxStages], bar_done[kRMaxStages], bar_acc;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    grid_dep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.stages;
    const int a_bytes = RM * RK * 2;
    const int stage_bytes = a_bytes + a.EB * RK * 2;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_done[s]), 1);
        }
        mbar_init(smem_u32(&bar_acc), 1);
        s_abort = 0;
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&s_tmem), (uint32_t)a.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;
    // CTAs of one cluster (k slices) are adjacent, then the expert blocks of
    // one token tile (x stays in L2)
    const int KS = a.ksplit;
    const int ks = blockIdx.x % KS, tile = blockIdx.x / KS;
    const int nk = a.K / RK / KS;             // k-stages of this CTA
    const int kc0 = ks * nk;
    const int t0 = (tile / a.e_blocks) * RM;
    const int e0 = (tile % a.e_blocks) * a.EB;
    float* part = reinterpret_cast<float*>(smem + S * stage_bytes);  // [RM][EB + 1] when KS > 1

    if (warp == 0) {
        // ---------------- MMA: warp-uniform loop, one elected lane issues ----------------
        int s = 0;
        uint32_t par = 0;
        for (int kc = 0; kc < nk; ++kc) {
            if (!warp_wait(smem_u32(&bar_full[s]), par, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * stage_bytes), sb = sa + a_bytes;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < RK / 16; ++kk)
                    mma_f16(tmem, sdesc_sw128(sa) + 2 * kk, sdesc_sw128(sb) + 2 * kk, idesc_bf16_f32(RM, a.EB),
                            (kc | kk) != 0);
                mma_commit(smem_u32(&bar_done[s]));
            }
            __syncwarp();
            if (++s == S) {
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
                const int s = kc % S;
                if (kc >= S &&
                    !mbar_wait(smem_u32(&bar_done[s]), (uint32_t)(((kc - S) / S) & 1), abort_flag, a.status))
                    break;
                const uint32_t bar = smem_u32(&bar_full[s]);
                const uint32_t dst = smem_u32(smem + s * stage_bytes);
                mbar_arrive_expect_tx(bar, (uint32_t)stage_bytes);
                tma_load_2d(dst, &a.tmap_x, (kc0 + kc) * (RK * 2), t0, bar);
                tma_load_2d(dst + a_bytes, &a.tmap_w, (kc0 + kc) * (RK * 2), e0, bar);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------- epilogue: one token per TMEM lane ----------------
        const int q = warp - 4;
        const int row = t0 + q * 32 + lane;
        if (warp_wait(smem_u32(&bar_acc), 0, abort_flag, a.status, 64)) {
            tc_fence_after();
            const bool vec = (a.E & 3) == 0;
            for (int c0 = 0; c0 < a.EB; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c0, r);
                tmem_ld_wait();
                if (KS > 1) {  // partial tile for the cluster's reduction
#pragma unroll
                    for (int j = 0; j < 32; ++j) part[(q * 32 + lane) * (a.EB + 1) + c0 + j] = __uint_as_float(r[j]);
                } else if (row < a.T) {
                    float* dst = a.logits + (size_t)row * a.E + e0 + c0;
                    const int n = min(32, a.E - (e0 + c0));
                    if (vec && n == 32) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4*>(dst + j) =
                                make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                            __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < n) dst[j] = __uint_as_float(r[j]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (KS > 1) {
        // every CTA of the cluster gets here (no early exit); the partials
        // are then summed in rank order, each CTA taking RM / KS rows
        cluster_barrier();
        const int rows = RM / KS;
        const uint32_t part_local = smem_u32(part);
        for (int i = threadIdx.x; i < rows * a.EB; i += kRThreads) {
            const int rr = ks * rows + i / a.EB, c = i % a.EB;
            const uint32_t off = part_local + (uint32_t)((rr * (a.EB + 1) + c) * 4);
            float sum = 0.0f;
            for (int q = 0; q < KS; ++q) sum += ld_dsmem(dsmem_addr(off, (uint32_t)q));
            const int row = t0 + rr, e = e0 + c;
            if (row < a.T && e < a.E) a.logits[(size_t)row * a.E + e] = sum;
        }
        cluster_barrier();  // no CTA leaves while another still reads its partial
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
    }
    grid_dep_launch();
}

}  // namespace

}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status moe_router_logits(const uint16_t* x_bf16, int T, int d, const uint16_t* w_router_bf16,
                                          int E, float* logits, int32_t* d_status, cudaStream_t stream) {
    if (T < 0 || d < 1 || E < 1) return NVFP4_ERR_INVALID_ARG;
    if (d % RK != 0 || E > kRMaxE) return NVFP4_ERR_SHAPE;
    if (T == 0) return NVFP4_OK;
    if (!x_bf16 || !w_router_bf16 || !logits) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(w_router_bf16) || !aligned16(logits) || (d_status && !aligned16(d_status)))
        return NVFP4_ERR_ALIGN;
    RouterArgs a{};
    a.T = T;
    a.K = d;
    a.E = E;
    const int nb = (E + kREGran - 1) / kREGran;  // 32-expert blocks
    const int m_tiles = (T + RM - 1) / RM;
    // blocks per CTA: the largest divisor of nb (<= 8) that still gives half
    // the SMs a CTA (N=32 MMAs are issue-bound, so fewer wider CTAs win)
    int c = 1;
    for (int cand = 1; cand <= nb && cand * kREGran <= kRMaxEB; ++cand)
        if (nb % cand == 0 && (long long)m_tiles * (nb / cand) * 2 >= num_sms()) c = cand;
    a.EB = c * kREGran;
    a.e_blocks = nb / c;
    // split K over a cluster while the grid is under half the SMs
    const int nk_all = d / RK;
    int ksplit = 1;
    while (ksplit < 8 && (long long)m_tiles * a.e_blocks * ksplit * 2 <= num_sms() && nk_all % (ksplit * 2) == 0)
        ksplit *= 2;
    a.ksplit = ksplit;
    int cols = 32;
    while (cols < a.EB) cols *= 2;
    a.tmem_cols = cols;
    const int stage_bytes = RM * RK * 2 + a.EB * RK * 2;
    const int part_bytes = ksplit > 1 ? RM * (a.EB + 1) * 4 : 0;
    a.stages = std::max(2, std::min(kRMaxStages, (kRSmemBudget - part_bytes) / stage_bytes));
    a.logits = logits;
    a.status = d_status;
    // bf16 rows as bytes: boxes of 128 bytes (64 values) x rows, 128-byte swizzle
    if (!encode_tmap_u8(&a.tmap_x, x_bf16, (unsigned long long)d * 2, (unsigned long long)T, RK * 2, RM, true) ||
        !encode_tmap_u8(&a.tmap_w, w_router_bf16, (unsigned long long)d * 2, (unsigned long long)E, RK * 2,
                        (unsigned)a.EB, true))
        return NVFP4_ERR_CUDA;
    const size_t smem = 1024 + (size_t)a.stages * stage_bytes + part_bytes;
    static bool init = false;
    if (!init) {
        cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmemBudget + 1024);
        init = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(m_tiles * a.e_blocks * ksplit);
    cfg.blockDim = dim3(kRThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (ksplit > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = ksplit;
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
    NVFP4_LAUNCH("router", stream, cudaLaunchKernelEx(&cfg, router_kernel, a));
    return last_launch_status();
}
