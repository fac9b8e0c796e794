// tc.cuh -- arguments and launchers of the prompt-shaped tensor-core GEMMs (moe_tc.cu, moe_tcm.cu, moe_tcq.cu).
#pragma once

#include "internal.cuh"

namespace nvfp4 {

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
// f16 rows [rows, K] as the f16 kernel's A operand (boxes of 128 rows x 64 values, 128-byte swizzle).
bool make_tmap_rows_f16(CUtensorMap* map, const void* base, int rows, int K);
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

size_t tc_smem_bytes(int nproj);
void launch_tc_gemm(int outmode, int nproj, const TcArgs& a, int max_units, cudaStream_t s,
                    bool routed_down = false);
// dst row r = f16(src row (map ? map[r] / map_div : r) * 2^-s), exps[r] = s;
// optionally zeroes row r of zero_rows (length zero_len) for r < zero_count.
void launch_rows_to_f16(const uint16_t* src, int rows, int K, uint16_t* dst, int32_t* exps, float* zero_rows,
                        int zero_len, cudaStream_t s, const int32_t* map = nullptr, int map_div = 1,
                        int zero_count = -1);

}  // namespace nvfp4
