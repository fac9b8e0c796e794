// decode.cuh -- arguments and launchers of the one-launch decode-shaped layer (moe_decode.cu).
#pragma once

#include "internal.cuh"

namespace nvfp4 {

// ---- decode-shaped layer in one persistent launch (moe_decode.cu) ----
struct DecodeArgs {
    // stored weights as TMA tiles: codes / scales of gate and up [E*F rows],
    // boxes of 128 rows x 256 K; down [E*d rows], boxes of 256 rows x 256 K
    CUtensorMap tm_gate_c, tm_up_c, tm_gate_s, tm_up_s, tm_down_c, tm_down_s;
    int d, F, top_k;
    int gbu, gbd;                   // 128-feature blocks per gate/up item, 256-output blocks per down item
    int chu, chd;                   // consecutive gate/up / down items a CTA takes per grab
    int slot_bytes;                 // set by the launcher
    const int32_t* offsets;         // [E+1]
    const int32_t* active;          // [E]
    const int32_t* n_active;        // [1]
    const int32_t* tile_start;      // [E+1] prefix of ceil(rows / kGemvTokTile)
    const int32_t* row_to_slot;     // [R]
    const int32_t* slot_to_row;     // [R]
    const float* topk_w;            // [R]
    const float *gate_ws2, *up_ws2, *down_ws2;  // [E]
    const uint16_t* x;              // B_BF16: x [T, d] bf16
    const uint8_t *xq, *xs;         // B_NVFP4: permuted NVFP4 rows [R, d/2], [R, d/16]
    const float *is13, *is2;        // B_NVFP4: static input scales [E]
    uint16_t* h;                    // B_BF16: h [R, F] bf16
    uint8_t *hq, *hs;               // B_NVFP4: h requantised [R, F/2], [R, F/16]
    float* yrows;                   // [R, d] w * y per routed row
    uint16_t* out;                  // [T, d] bf16
    int* counters;                  // [2] gate/up and down item counters (zeroed before the launch)
    int* tile_ready;                // [row tiles] gate/up items done (zeroed)
    int* tok_done;                  // [T, d / 256] contributions per (token, output group) (zeroed)
    int32_t* status;                // NVFP4_ERR_TIMEOUT if a bounded wait expired
};
// d and F multiples of 256 and the shared-memory ring fits.
bool decode_supported(int d, int F);
// Output groups of the finest split (sizes the tok_done counters).
int decode_groups_d(int d);
// Encodes the weight tensor maps.
bool decode_set_maps(DecodeArgs* a, const nvfp4_moe_weights* w);
// Item sizes and grab lengths for about `expected_tiles` row tiles (sets
// gbu, gbd, chu, chd; d and F already set).
void decode_pick_work(int expected_tiles, DecodeArgs* a);
void launch_decode(int bmode, const DecodeArgs& a, cudaStream_t s);

}  // namespace nvfp4
