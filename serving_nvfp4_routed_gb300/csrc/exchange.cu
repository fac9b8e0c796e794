// exchange.cu -- the two ends of an expert-parallel routed layer: the gather
// of each routed row into the permutation's expert-contiguous order (what a
// rank sends to the ranks that own the experts) and the weighted top-k
// combine of the rows that come back.
//
// W4A4 model card "GLM-5.3-Flash-NVFP4-W4A4-Experts", "Validation" (the
// routed experts run tensor- and expert-parallel over four GPUs) and
// TensorFold issue #308 "GLM-5.3-Flash on CUDA: read nvidia/GLM-5.3-Flash-
// NVFP4 (ModelOpt NVFP4) as stored, W4A16", "What the branch does" (the
// grouped kernel takes the routed rows expert by expert).
#include <climits>

#include "common.cuh"
#include "internal.cuh"

namespace nvfp4 {

namespace {

constexpr int kGatherWarps = 8;

// One warp per routed row r: rows_out[r] = x[row_to_slot[r] / k] (16-byte
// copies) and, if asked, expert_of_row[r] = e with offsets[e] <= r < offsets[e+1].
__global__ void __launch_bounds__(kGatherWarps * 32) gather_rows_kernel(
    const uint16_t* __restrict__ x, int d, const int32_t* __restrict__ row_to_slot, int k, int R,
    const int32_t* __restrict__ offsets, int E, uint16_t* __restrict__ rows_out, int32_t* __restrict__ expert_of_row) {
    grid_dep_wait();
    const int lane = threadIdx.x & 31;
    for (int r = blockIdx.x * kGatherWarps + (threadIdx.x >> 5); r < R; r += gridDim.x * kGatherWarps) {
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(row_to_slot[r] / k) * d);
        uint4* dst = reinterpret_cast<uint4*>(rows_out + (size_t)r * d);
        for (int q = lane; q < d / 8; q += 32) dst[q] = __ldg(src + q);
        if (expert_of_row && lane == 0) {
            int lo = 0, hi = E;  // largest lo with offsets[lo] <= r
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (offsets[mid] <= r) lo = mid; else hi = mid;
            }
            expert_of_row[r] = lo;
        }
    }
    grid_dep_launch();
}

}  // namespace

}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status moe_gather_rows(const uint16_t* x_bf16, int T, int d, const int32_t* row_to_slot, int top_k,
                                        const int32_t* expert_offsets, int E, uint16_t* rows_out,
                                        int32_t* expert_of_row, cudaStream_t stream) {
    if (T < 0 || d < 1 || top_k < 1) return NVFP4_ERR_INVALID_ARG;
    if (d % 8 != 0 || (size_t)T * top_k > (size_t)INT_MAX / 2) return NVFP4_ERR_SHAPE;
    if (expert_of_row && (E < 1 || E > kMaxExperts)) return NVFP4_ERR_SHAPE;
    if (T == 0) return NVFP4_OK;
    if (!x_bf16 || !row_to_slot || !rows_out || (expert_of_row && !expert_offsets)) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(x_bf16) || !aligned16(rows_out) || !aligned16(row_to_slot) ||
        (expert_of_row && (!aligned16(expert_of_row) || !aligned16(expert_offsets))))
        return NVFP4_ERR_ALIGN;
    const int R = T * top_k;
    const int grid = std::min((R + kGatherWarps - 1) / kGatherWarps, num_sms() * 8);
    NVFP4_LAUNCH("gather_rows", stream,
                 launch_pdl(gather_rows_kernel, dim3(grid), dim3(kGatherWarps * 32), 0, stream, x_bf16, d, row_to_slot,
                            top_k, R, expert_offsets, E, rows_out, expert_of_row));
    return last_launch_status();
}

extern "C" nvfp4_status moe_combine_rows(const uint16_t* y_bf16, const int32_t* slot_to_row, const float* topk_w, int T,
                                         int top_k, int d, uint16_t* out_bf16, cudaStream_t stream) {
    if (T < 0 || d < 1 || top_k < 1) return NVFP4_ERR_INVALID_ARG;
    if (d % 8 != 0 || (size_t)T * top_k > (size_t)INT_MAX / 2) return NVFP4_ERR_SHAPE;
    if (T == 0) return NVFP4_OK;
    if (!y_bf16 || !slot_to_row || !topk_w || !out_bf16) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(y_bf16) || !aligned16(slot_to_row) || !aligned16(topk_w) || !aligned16(out_bf16))
        return NVFP4_ERR_ALIGN;
    launch_sum_rows(y_bf16, slot_to_row, topk_w, T, top_k, d, out_bf16, stream);
    return last_launch_status();
}
