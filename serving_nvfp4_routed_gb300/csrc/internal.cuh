// internal.cuh -- host-side launchers shared between the library's .cu files.
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

// ---- decode-shaped grouped GEMM (mma.sync, weights streamed from HBM) ----
enum BMode { B_BF16 = 0, B_NVFP4 = 1 };
enum OutMode { OUT_H = 0, OUT_HQ = 1, OUT_COMBINE = 2, OUT_BF16 = 3 };

struct GemvArgs {
    int K, N, top_k;
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

// ---- prompt-shaped grouped GEMM (tcgen05, accumulators in TMEM) ----
enum TcOut { TC_OUT_H = 0, TC_OUT_BF16 = 2 };

struct TcArgs {
    int K, N, top_k;
    const int32_t* offsets;      // [E+1]
    const int32_t* active;       // [E]
    const int32_t* n_active;     // [1]
    const int32_t* tile_start;   // [E+1] prefix of ceil(rows / kTcTokTile) over active experts
    const int32_t* row_to_slot;  // [R] (nullptr: row == token)
    const uint8_t* a_codes[2];   // [E, N, K/2]
    const uint8_t* a_scales[2];  // [E, N, K/16]
    const float* a_ws2[2];       // [E]
    const uint16_t* b_f16;       // f16 rows, value = f16 * 2^b_exp[row]
    const int32_t* b_exp;
    int b_by_token;              // B row = token of the permuted row (x) or the row itself (h)
    uint16_t* h_out;             // TC_OUT_H: [R, N] bf16 SwiGLU
    uint16_t* y_out;             // TC_OUT_BF16: [R, N]
    int32_t* status;             // optional: NVFP4_ERR_TIMEOUT if a bounded wait expired
};

// ---- prompt-shaped grouped GEMMs with the routed rows as M (tcgen05) ----
// SWIGLU: h = bf16(silu(bf16 G) * bf16 U); SWIGLU_Q: h requantised to NVFP4
// (codes + e4m3 block scales under hq_gs); BF16: plain bf16 rows; ROWS: bf16
// rows y by routed row, summed per token with the routing weights afterwards
// (launch_sum_rows).
// The f16 kernel (tcm) takes SWIGLU, ROWS and BF16; the block-scaled FP4
// kernel (tcq) SWIGLU_Q and ROWS.
enum TcmEpi { TCM_SWIGLU = 0, TCM_BF16 = 2, TCM_SWIGLU_Q = 3, TCM_ROWS = 4 };

struct TcmArgs {
    CUtensorMap tmap_x;          // tcm: f16 rows [R, K] (expert order), box 64 x 128, 128-byte swizzle
    CUtensorMap tmap_ac;         // tcq: NVFP4 rows, codes [R, K/2]
    CUtensorMap tmap_as;         //   and e4m3 scales [R, K/16]
    CUtensorMap tmap_wc[2];      // weight codes [E*N, K/2] uint8, box 32 x 128
    CUtensorMap tmap_ws[2];      // weight scales [E*N, K/16] uint8, box 16 x 128
    int K, N, top_k;             // N: features of one projection (gate/up: F, down: d)
    const int32_t* offsets;      // [E+1]
    const int32_t* active;       // [E]
    const int32_t* n_active;     // [1]
    const int32_t* tile_start;   // [E+1] prefix of ceil(rows / 128) over active experts
    const uint8_t* a_codes[2];   // weights [E, N, K/2] (SwiGLU: gate, up)
    const uint8_t* a_scales[2];  // [E, N, K/16]
    const float* a_ws2[2];       // [E]
    const int32_t* x_exp;        // [R] value of an f16 row = f16 * 2^x_exp[row]
    const float* x_gs;           // NVFP4 rows: [E] global scale of the rows of expert e
    uint16_t* h_out;             // TCM_SWIGLU: [R, N] bf16
    const int32_t* row_to_slot;  // TCM_ROWS: [R]
    const float* topk_w;         // TCM_ROWS: [T*k]
    uint16_t* y_out;             // TCM_BF16: [R, N]
    uint16_t* y_rows;            // TCM_ROWS: [R, N] bf16 y by routed row (the weights are applied by sum_rows)
    uint8_t* hq_out;             // TCM_SWIGLU_Q: [R, N/2] codes
    uint8_t* hs_out;             //   [R, N/16] e4m3 block scales
    const float* hq_gs;          //   [E] global scale they are taken under
    int32_t* status;             // NVFP4_ERR_TIMEOUT if a bounded wait expired
};
bool make_tmap_rows_f16(CUtensorMap* map, const void* base, int rows, int K);
// 2-D uint8 tensor map over [rows, inner_bytes] (row pitch = inner_bytes).
bool encode_tmap_u8(CUtensorMap* map, const void* base, unsigned long long inner_bytes, unsigned long long rows,
                    unsigned box_inner, unsigned box_rows, bool swizzle128);
bool tcm_supported(int epi, int N, int K);
// Fills tmap_wc / tmap_ws from a_codes / a_scales (rows = E * N, K = a->K).
bool tcm_set_weights(TcmArgs* a, long long rows);
// A rows are f16 (tmap_x, x_exp).
void launch_tcm(int epi, const TcmArgs& a, int max_units, cudaStream_t s);

// ---- W4A4 prompt-shaped grouped GEMM on the block-scaled FP4 tensor cores ----
// Same arguments as TcmArgs (NVFP4 rows: a_codes / x_gs); epi TCM_SWIGLU_Q
// or TCM_ROWS.  Needs K % 256 == 0 and N % 16 (SwiGLU) / N % 32.
bool tcq_supported(int epi, int N, int K);
// Encodes the tensor maps this kernel uses (rows_w = E * N, rows_x = R).
bool tcq_set_maps(TcmArgs* a, const uint8_t* x_codes, const uint8_t* x_scales, long long rows_x, long long rows_w);
// max_tiles bounds the 128-row tiles over all experts; the unit count
// follows from the kernel's column slice.
void launch_tcq(int epi, const TcmArgs& a, int max_tiles, cudaStream_t s);
// out[t] = bf16(sum over slots j in order of w[t*k + j] * y[slot_to_row[t*k + j]]),
// y rows of d bf16 values, the sum in fp32.
void launch_sum_rows(const uint16_t* y, const int32_t* slot_to_row, const float* topk_w, int T, int k, int d,
                     uint16_t* out, cudaStream_t s);

size_t tc_smem_bytes(int nproj);
void launch_tc_gemm(int outmode, int nproj, const TcArgs& a, int max_units, cudaStream_t s,
                    bool routed_down = false);
// dst row r = f16(src row (map ? map[r] / map_div : r) * 2^-s), exps[r] = s;
// optionally zeroes row r of zero_rows (length zero_len) for r < zero_count.
void launch_rows_to_f16(const uint16_t* src, int rows, int K, uint16_t* dst, int32_t* exps, float* zero_rows,
                        int zero_len, cudaStream_t s, const int32_t* map = nullptr, int map_div = 1,
                        int zero_count = -1);
}  // namespace nvfp4
