// internal.cuh -- declarations shared between the library's .cu files (the kernel
// families add their own: gemv.cuh, decode.cuh, tc.cuh).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace nvfp4 {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kGemvTokTile = 8;   // rows per work item of the decode-shaped kernel
constexpr int kTcTokTile = 128;   // rows per work unit of the tensor-core kernel

// Routing outputs plus the grouping metadata the expert kernels walk.
struct RouteArrays {
    int32_t* ids;          // [T*k]
    float* w;              // [T*k]
    int32_t* offsets;      // [E+1]
    int32_t* row_to_slot;  // [R]
    int32_t* slot_to_row;  // [R]
    int32_t* active;       // [E]   experts with rows, ascending
    int32_t* n_active;     // [1]
    int32_t* tile_start;   // [E+1] prefix over active experts of ceil(rows / kGemvTokTile)
    int32_t* tile_start_tc;  // [E+1] prefix over active experts of ceil(rows / kTcTokTile)
    int32_t* counts;       // [n_blocks * E] scratch for the multi-block path
    int32_t* clear;        // [n_clear] zeroed by the route launch (work and completion counters)
    int n_clear;
};

size_t route_scratch_words(int T, int E, int top_k);
// logits != nullptr: top-k + permutation.  logits == nullptr: ids/w are
// given; validates them (status) and builds the permutation.
void launch_route(const float* logits, int T, int E, int top_k, RouteArrays ra, int32_t* d_status,
                  cudaStream_t s);

void launch_zero(void* p, size_t bytes, cudaStream_t s);
// The weight recipe (quant.cu): argument checks, then the amax pass and the
// block pass with `amax` ([batch] floats, cleared first) as scratch.  The
// amax pass runs one grid row per tensor, so batch is limited to the grid's
// y extent.
constexpr int kMaxRecipeBatch = 65535;
nvfp4_status check_weight_recipe(const uint16_t* w, int batch, int N, int K, const uint8_t* codes,
                                 const uint8_t* scales, const float* weight_scale_2);
nvfp4_status launch_weight_recipe(const uint16_t* w, int batch, int N, int K, float* amax, uint8_t* codes,
                                  uint8_t* scales, float* weight_scale_2, cudaStream_t stream);
void launch_quantize_act(const uint16_t* x, int M, int K, const int32_t* row_to_slot, int top_k,
                         const float* input_scale, const int32_t* offsets, int E, uint8_t* codes,
                         uint8_t* scales, cudaStream_t s);

// Operand form of the routed rows: bf16, or NVFP4 codes + scales.
enum BMode { B_BF16 = 0, B_NVFP4 = 1 };

// 2-D uint8 tensor map over [rows, inner_bytes] (row pitch = inner_bytes).
bool encode_tmap_u8(CUtensorMap* map, const void* base, unsigned long long inner_bytes, unsigned long long rows,
                    unsigned box_inner, unsigned box_rows, bool swizzle128);

// out[t] = bf16(sum over slots j in order of w[t*k + j] * y[slot_to_row[t*k + j]]),
// y rows of d bf16 values, the sum in fp32.
void launch_sum_rows(const uint16_t* y, const int32_t* slot_to_row, const float* topk_w, int T, int k, int d,
                     uint16_t* out, cudaStream_t s);
}  // namespace nvfp4
