// gemv.cuh -- arguments and launchers of the decode-shaped grouped GEMM (moe_gemv.cu).
#pragma once

#include "internal.cuh"

namespace nvfp4 {

// ---- decode-shaped grouped GEMM (mma.sync, weights streamed from HBM) ----
enum OutMode { OUT_H = 0, OUT_HQ = 1, OUT_COMBINE = 2, OUT_BF16 = 3 };

struct GemvArgs {
    int K, N, top_k;
    int E;                          // experts: the routing arrays' length
    int nproj;                      // 2: gate+up (SwiGLU epilogue), 1: single projection
    int ksplit;                     // warps of a CTA splitting K (1, 2, 4 or 8)
    int fb_group;                   // feature blocks per work item (they share the staged rows)
    const int32_t* offsets;         // [E+1]
    const int32_t* active;          // [E]
    const int32_t* n_active;        // [1]
    const int32_t* tile_start;      // [E+1]
    const int32_t* row_to_slot;     // [R] (nullptr: row == token, top_k ignored)
    const uint8_t* a_codes[2];      // [E, N, K/2]
    const uint8_t* a_scales[2];     // [E, N, K/16]
    const float* a_ws2[2];          // [E]
    // B_BF16: bf16 rows (row index = token when b_by_token, else the permuted
    // row); each CTA takes a row's max |v| while staging it
    const uint16_t* b_bf16;
    int b_by_token;
    // B_NVFP4: quantised permuted rows and the expert's input scale
    const uint8_t* b_codes;
    const uint8_t* b_scales;
    const float* b_gs;              // [E]
    // epilogue
    uint16_t* h_out;                // OUT_H: [R, N] bf16
    uint8_t* hq_out;                // OUT_HQ: [R, N/2]
    uint8_t* hs_out;                // OUT_HQ: [R, N/16]
    const float* hq_gs;             // OUT_HQ: [E] next input scale
    float* y_rows;                  // OUT_COMBINE: [R, N] w * y per routed row (fp32)
    const int32_t* slot_to_row;     // OUT_COMBINE: [R]
    const float* topk_w;            // OUT_COMBINE: [T*k]
    int* tok_done;                  // OUT_COMBINE: [T, item groups] completed slots (zeroed before)
    uint16_t* out_bf16;             // OUT_COMBINE: [T, N] final bf16 rows
    uint16_t* y_out;                // OUT_BF16: [R, N]
    int* work_counter;              // zeroed before the launch
    // L2 prefetch of the weight tiles ahead of the loads (gate/up, K not
    // split over warps): one TMA tensor prefetch per projection, codes and
    // scales, of the CTA's feature rows (boxes of 128 / 16 bytes x 128 rows),
    // pf_dist chunks ahead (0: off)
    CUtensorMap pf_codes[2], pf_scales[2];
    int pf_dist;
};

// ksplit chosen from the expected number of work items
int gemv_pick_ksplit(int expected_tiles, int N, int nproj);
int gemv_pick_group(int expected_tiles, int N, int ksplit, int nproj);
// Work-item groups along N of a launch with these picks (one completion
// counter per token and group in OUT_COMBINE).
int gemv_item_groups(int N, int ksplit, int fb_group);
size_t gemv_smem_bytes(int K);
bool gemv_supported_k(int K);
void launch_gemv(int bmode, int outmode, const GemvArgs& a, int max_work, cudaStream_t s);

}  // namespace nvfp4
