// route.cu -- router logits -> top-k experts -> expert-contiguous rows.
//
// TensorFold issue #308 "GLM-5.3-Flash on CUDA: read nvidia/GLM-5.3-Flash-NVFP4
// (ModelOpt NVFP4) as stored, W4A16", "The checkpoint": the router is BF16
// (its fp32 logits are this file's input); "What the branch does": the routed
// experts run through one grouped kernel, which needs each expert's rows
// contiguous.  Router function (softmax, top-k with ties to the lower id,
// weights renormalised over the k chosen) is the plain reading.
//
// Top-k: one warp per token, logits in registers, k rounds of a warp arg-max.
// Weights: exp(l - l_max) / sum over the k, in fp64, rounded once to fp32.
// Permutation (stable: expert, token, slot): a per-expert histogram, a
// warp-scan exclusive prefix sum, and a scatter in which each row's position
// is its expert's base + the count of equal experts before it -- within a warp
// by __match_any_sync, across warps by per-warp counts in shared memory.  No
// atomic decides an order, so the result is deterministic.
#include <climits>

#include "common.cuh"
#include "internal.cuh"

namespace nvfp4 {

namespace {

constexpr int kSmallMaxRows = 8192;
constexpr int kChunkRows = 1024;   // rows per block in the multi-block path (one scatter round)

template <int MAXL>
__device__ void warp_topk(const float* __restrict__ lg, int E, int k, int32_t* __restrict__ ids,
                          float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    float v[MAXL];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < MAXL; ++i) {
        const int e = lane + 32 * i;
        float x = e < E ? lg[e] : -INFINITY;
        v[i] = (x != x) ? -INFINITY : x;  // NaN never ranks above a number
        if (e >= E) taken |= 1u << i;
    }
    float my_v = 0.0f;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < MAXL; ++i) {
            const int e = lane + 32 * i;
            if (!((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) {
            my_v = bv;
            my_id = bi;
        }
    }
    // the selected logits, in slot order; softmax_weights turns them into
    // the routing weights
    if (lane < k) {
        ids[lane] = my_id;
        w[lane] = my_v;
    }
}

// Routing weights of tokens [t0, t1) from their selected logits in w (slot 0
// holds the largest): fp64 exp(l_j - l_max), summed over the k in slot order,
// divided, rounded once to fp32.  Non-finite top logits: +inf entries share
// the weight equally; all -inf: 1/k each.  Each warp takes floor(32 / k)
// tokens at once (fp64 is slow on this part: a full warp of exponentials
// instead of k lanes per token), so the calling block passes its warp index
// and warp count.
__device__ void softmax_weights(float* w, int t0, int t1, int k, int warp, int n_warps) {
    const int lane = threadIdx.x & 31;
    const int tpw = 32 / k;  // tokens per warp pass
    const int tl = lane / k, j = lane % k;
    for (int tb = t0 + warp * tpw; tb < t1; tb += n_warps * tpw) {  // warp-uniform trip count
        const int t = tb + tl;
        const bool live = tl < tpw && t < t1;
        double ex = 0.0;
        float v = 0.0f;
        if (live) {
            v = w[(size_t)t * k + j];
            const float m = w[(size_t)t * k];
            if (m == INFINITY) ex = v == INFINITY ? 1.0 : 0.0;
            else if (m == -INFINITY) ex = 1.0;
            else ex = exp((double)v - (double)m);
        }
        double sum = 0.0;
        for (int jj = 0; jj < k; ++jj) sum += __shfl_sync(0xffffffffu, ex, (tl < tpw ? tl : 0) * k + jj);
        if (live) w[(size_t)t * k + j] = (float)(ex / sum);
    }
}

__device__ void topk_dispatch(const float* lg, int E, int k, int32_t* ids, float* w) {
    if (E <= 64) warp_topk<2>(lg, E, k, ids, w);
    else if (E <= 128) warp_topk<4>(lg, E, k, ids, w);
    else if (E <= 320) warp_topk<10>(lg, E, k, ids, w);
    else if (E <= 512) warp_topk<16>(lg, E, k, ids, w);
    else warp_topk<32>(lg, E, k, ids, w);
}

// Exclusive scan of four ints per thread over the block in one pass
// (blockDim multiple of 32): returns the prefix, `total` the block sums.
__device__ int4 block_exclusive_scan4(int4 v, int4* tmp, int4& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int4 x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int4 y = make_int4(__shfl_up_sync(0xffffffffu, x.x, o), __shfl_up_sync(0xffffffffu, x.y, o),
                                 __shfl_up_sync(0xffffffffu, x.z, o), __shfl_up_sync(0xffffffffu, x.w, o));
        if (lane >= o) {
            x.x += y.x;
            x.y += y.y;
            x.z += y.z;
            x.w += y.w;
        }
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int4 t = lane < nw ? tmp[lane] : make_int4(0, 0, 0, 0);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int4 y = make_int4(__shfl_up_sync(0xffffffffu, t.x, o), __shfl_up_sync(0xffffffffu, t.y, o),
                                     __shfl_up_sync(0xffffffffu, t.z, o), __shfl_up_sync(0xffffffffu, t.w, o));
            if (lane >= o) {
                t.x += y.x;
                t.y += y.y;
                t.z += y.z;
                t.w += y.w;
            }
        }
        tmp[lane] = t;
    }
    __syncthreads();
    const int4 before = warp > 0 ? tmp[warp - 1] : make_int4(0, 0, 0, 0);
    total = tmp[nw - 1];
    __syncthreads();
    return make_int4(before.x + x.x - v.x, before.y + x.y - v.y, before.z + x.z - v.z, before.w + x.w - v.w);
}

// offsets / active list / gemv tile prefix from per-expert counts c (thread e
// holds expert e; blockDim >= E).
__device__ void write_group_meta(int c, int E, const RouteArrays& ra, int4* tmp, int& off_out) {
    const int e = threadIdx.x;
    const int cc = e < E ? c : 0;
    const int flag = cc > 0 ? 1 : 0;
    // one pass: offsets, active-list index, decode tiles, tensor-core tiles
    int4 tot;
    const int4 pre = block_exclusive_scan4(
        make_int4(cc, flag, flag ? (cc + kGemvTokTile - 1) / kGemvTokTile : 0,
                  flag ? (cc + kTcTokTile - 1) / kTcTokTile : 0),
        tmp, tot);
    if (e < E) ra.offsets[e] = pre.x;
    if (e == 0) ra.offsets[E] = tot.x;
    if (flag) {
        ra.active[pre.y] = e;
        ra.tile_start[pre.y] = pre.z;
        if (ra.tile_start_tc) ra.tile_start_tc[pre.y] = pre.w;
    }
    if (e == 0) {
        *ra.n_active = tot.y;
        ra.tile_start[tot.y] = tot.z;
        if (ra.tile_start_tc) ra.tile_start_tc[tot.y] = tot.w;
    }
    off_out = pre.x;
}

// Scatter rows [row0, row1) in rounds of blockDim rows; run[e] holds the next
// free position of expert e (shared), wh is [32][E] per-warp round counts.
__device__ void scatter_rows(int row0, int row1, int E, const int32_t* __restrict__ ids, int* run,
                             uint8_t* wh, const RouteArrays& ra) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int base = row0; base < row1; base += blockDim.x) {
        const int r = base + threadIdx.x;
        const int e = r < row1 ? ids[r] : -1;
        const unsigned mask = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(mask & ((1u << lane) - 1u));
        if (e >= 0 && rank == 0) wh[warp * E + e] = (uint8_t)__popc(mask);
        __syncthreads();
        if (e >= 0) {
            int pos = run[e] + rank;
            for (int w2 = 0; w2 < warp; ++w2) pos += wh[w2 * E + e];
            ra.row_to_slot[pos] = r;
            ra.slot_to_row[r] = pos;
        }
        __syncthreads();
        const int nwu = min(nw, (row1 - base + 31) / 32);  // warps that held rows this round
        for (int e2 = threadIdx.x; e2 < E; e2 += blockDim.x) {
            int s = 0;
            for (int w2 = 0; w2 < nwu; ++w2) {
                s += wh[w2 * E + e2];
                wh[w2 * E + e2] = 0;
            }
            run[e2] += s;
        }
        __syncthreads();
    }
}

// ids given by the caller: report and clamp out-of-range ids (so no later
// kernel indexes out of bounds).
__device__ void validate_ids(int32_t* ids, int R, int E, int32_t* status) {
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < R; r += gridDim.x * blockDim.x) {
        int e = ids[r];
        if (e < 0 || e >= E) {
            ids[r] = 0;
            if (status) atomicExch(status, (int)NVFP4_ERR_DEVICE_INPUT);
        }
    }
}

// Permutation of R <= kSmallMaxRows rows in one CTA (ids already written by
// topk_kernel, or given by the caller and validated here).  With logits (a
// few tokens) the CTA also runs the top-k itself, one warp per token, so that
// a decode step routes in one launch.  Up to 16 tokens; at 64 tokens the
// separate multi-CTA top-k plus this permutation was measured 9 us faster per
// layer on GB300 (one CTA's 32 warps then take two tokens each).
constexpr int kFusedTopkMaxTokens = 16;

__global__ void __launch_bounds__(1024) route_perm_small_kernel(int T, int E, int k, int given_ids, RouteArrays ra,
                                                                int32_t* status, const float* logits) {
    __shared__ int run[kMaxExperts];
    __shared__ uint8_t wh[32 * kMaxExperts];
    __shared__ int4 tmp32[32];
    grid_dep_wait();
    const int R = T * k;
    if (logits) {
        for (int t = threadIdx.x >> 5; t < T; t += blockDim.x >> 5)
            topk_dispatch(logits + (size_t)t * E, E, k, ra.ids + (size_t)t * k, ra.w + (size_t)t * k);
        __syncthreads();  // the block reads these ids and logits below
        softmax_weights(ra.w, 0, T, k, threadIdx.x >> 5, blockDim.x >> 5);
    }
    if (given_ids) validate_ids(ra.ids, R, E, status);
    for (int i = threadIdx.x; i < E; i += blockDim.x) run[i] = 0;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wh[i] = 0;
    for (int i = threadIdx.x; i < ra.n_clear; i += blockDim.x) ra.clear[i] = 0;
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x) atomicAdd(&run[ra.ids[r]], 1);
    __syncthreads();
    const int c = threadIdx.x < E ? run[threadIdx.x] : 0;
    int off;
    write_group_meta(c, E, ra, tmp32, off);
    if (threadIdx.x < E) run[threadIdx.x] = off;
    __syncthreads();
    scatter_rows(0, R, E, ra.ids, run, wh, ra);
    grid_dep_launch();
}

// One warp per token.
__global__ void topk_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* ids, float* w) {
    grid_dep_wait();
    const int nw = blockDim.x >> 5;
    const int t0 = blockIdx.x * nw, t = t0 + (threadIdx.x >> 5);
    if (t < T) topk_dispatch(logits + (size_t)t * E, E, k, ids + (size_t)t * k, w + (size_t)t * k);
    __syncthreads();  // the block's selected logits are written
    softmax_weights(w, t0, min(T, t0 + nw), k, threadIdx.x >> 5, nw);
    grid_dep_launch();
}

__global__ void validate_ids_kernel(int32_t* ids, int R, int E, int32_t* status) {
    grid_dep_wait();
    validate_ids(ids, R, E, status);
}

__global__ void __launch_bounds__(1024) perm_count_kernel(const int32_t* __restrict__ ids, int R, int E,
                                                          int32_t* counts) {
    __shared__ int hist[kMaxExperts];
    grid_dep_wait();
    for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const int r0 = blockIdx.x * kChunkRows, r1 = min(R, r0 + kChunkRows);
    for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) atomicAdd(&hist[ids[r]], 1);
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) counts[(size_t)blockIdx.x * E + i] = hist[i];
}

__global__ void __launch_bounds__(1024) perm_scan_kernel(int nb, int E, int32_t* counts, RouteArrays ra) {
    __shared__ int4 tmp32[32];
    grid_dep_wait();
    const int e = threadIdx.x;
    int run = 0;
    if (e < E) {
        for (int b0 = 0; b0 < nb; b0 += 8) {  // eight chunks' loads in flight
            int c[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) c[j] = b0 + j < nb ? counts[(size_t)(b0 + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (b0 + j < nb) {
                    counts[(size_t)(b0 + j) * E + e] = run;
                    run += c[j];
                }
        }
    }
    int off;
    write_group_meta(run, E, ra, tmp32, off);
    if (e < E)
        for (int b = 0; b < nb; ++b) counts[(size_t)b * E + e] += off;
    for (int i = threadIdx.x; i < ra.n_clear; i += blockDim.x) ra.clear[i] = 0;
}

__global__ void __launch_bounds__(1024) perm_scatter_kernel(int R, int E, const int32_t* __restrict__ counts,
                                                            RouteArrays ra) {
    __shared__ int run[kMaxExperts];
    __shared__ uint8_t wh[32 * kMaxExperts];
    grid_dep_wait();
    for (int i = threadIdx.x; i < E; i += blockDim.x) run[i] = counts[(size_t)blockIdx.x * E + i];
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wh[i] = 0;
    __syncthreads();
    const int r0 = blockIdx.x * kChunkRows, r1 = min(R, r0 + kChunkRows);
    scatter_rows(r0, r1, E, ra.ids, run, wh, ra);
}

}  // namespace

size_t route_scratch_words(int T, int E, int top_k) {
    size_t R = (size_t)T * top_k;
    size_t nb = (R + kChunkRows - 1) / kChunkRows;
    return nb * (size_t)E;
}

void launch_route(const float* logits, int T, int E, int k, RouteArrays ra, int32_t* d_status, cudaStream_t s) {
    const int R = T * k;
    const bool fused = logits && T <= kFusedTopkMaxTokens && R <= kSmallMaxRows;
    if (logits && !fused) {
        // one warp per token, 8 tokens per CTA: the top-k work spreads over SMs
        NVFP4_LAUNCH("route_topk", s,
                     launch_pdl(topk_kernel, dim3((T + 7) / 8), dim3(256), 0, s, logits, T, E, k, ra.ids, ra.w));
    }
    if (R <= kSmallMaxRows) {
        NVFP4_LAUNCH(fused ? "route" : "route_perm", s,
                     launch_pdl(route_perm_small_kernel, dim3(1), dim3(1024), 0, s, T, E, k, logits ? 0 : 1, ra,
                                d_status, fused ? logits : (const float*)nullptr));
        return;
    }
    if (!logits) {
        NVFP4_LAUNCH("route_validate", s,
                     launch_pdl(validate_ids_kernel, dim3((R + 255) / 256), dim3(256), 0, s, ra.ids, R, E, d_status));
    }
    const int nb = (R + kChunkRows - 1) / kChunkRows;
    NVFP4_LAUNCH("route_count", s,
                 launch_pdl(perm_count_kernel, dim3(nb), dim3(1024), 0, s, (const int32_t*)ra.ids, R, E, ra.counts));
    NVFP4_LAUNCH("route_scan", s, launch_pdl(perm_scan_kernel, dim3(1), dim3(1024), 0, s, nb, E, ra.counts, ra));
    NVFP4_LAUNCH("route_scatter", s,
                 launch_pdl(perm_scatter_kernel, dim3(nb), dim3(1024), 0, s, R, E, (const int32_t*)ra.counts, ra));
}

// Route workspace layout (shared with the MoE workspace's routing block).
struct RouteWs {
    int32_t *active, *n_active, *tile_start, *counts;
};
static RouteWs carve_route_ws(Carver& c, int T, int E, int k) {
    RouteWs r;
    r.active = c.take<int32_t>(E);
    r.n_active = c.take<int32_t>(4);
    r.tile_start = c.take<int32_t>(E + 1);
    r.counts = c.take<int32_t>(route_scratch_words(T, E, k) + 1);
    return r;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" size_t moe_route_permute_workspace_size(int T, int E, int top_k) {
    if (T < 0 || E < 1 || top_k < 1) return 0;
    Carver c(nullptr);
    carve_route_ws(c, T, E, top_k);
    return align_up(c.off, 256);
}

extern "C" nvfp4_status moe_route_permute(const float* logits, int T, int E, int top_k, int32_t* topk_ids,
                                          float* topk_w, int32_t* expert_offsets, int32_t* row_to_slot,
                                          int32_t* slot_to_row, void* ws, size_t ws_bytes,
                                          cudaStream_t stream) {
    if (T < 0) return NVFP4_ERR_INVALID_ARG;
    if (E < 1 || E > kMaxExperts || top_k < 1 || top_k > kMaxTopK || top_k > E) return NVFP4_ERR_SHAPE;
    if ((size_t)T * top_k > (size_t)INT_MAX / 2) return NVFP4_ERR_SHAPE;
    // T == 0: nothing is read; the offsets are still written (all zero)
    if ((T > 0 && (!logits || !topk_ids || !topk_w || !row_to_slot || !slot_to_row)) || !expert_offsets || !ws)
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_w) || !aligned16(expert_offsets) ||
        !aligned16(row_to_slot) || !aligned16(slot_to_row) || !aligned16(ws))
        return NVFP4_ERR_ALIGN;
    if (ws_bytes < moe_route_permute_workspace_size(T, E, top_k)) return NVFP4_ERR_WORKSPACE;
    Carver c(ws);
    RouteWs rw = carve_route_ws(c, T, E, top_k);
    RouteArrays ra{topk_ids, topk_w, expert_offsets, row_to_slot, slot_to_row,
                   rw.active, rw.n_active, rw.tile_start, nullptr, rw.counts, nullptr, 0};
    if (T == 0) {
        launch_zero(expert_offsets, sizeof(int32_t) * (E + 1), stream);
        return last_launch_status();
    }
    launch_route(logits, T, E, top_k, ra, nullptr, stream);
    return last_launch_status();
}
