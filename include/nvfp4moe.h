/*
 * nvfp4moe.h -- C ABI of libnvfp4moe: the routed-expert MoE layer over a
 * ModelOpt NVFP4 checkpoint as stored, on one GB300 (sm_103a).
 *
 * The format (TensorFold issue #308, "GLM-5.3-Flash on CUDA: read
 * nvidia/GLM-5.3-Flash-NVFP4 (ModelOpt NVFP4) as stored, W4A16", section "The
 * checkpoint"): a weight tensor [N, K] is stored as
 *   codes  uint8 [N, K/2]   two e2m1 codes per byte, EVEN k in the LOW nibble
 *   scales uint8 [N, K/16]  one e4m3 scale per 16 consecutive k ("fn": bias 7,
 *                           max 448, 0x7F NaN), row-major as stored
 *   weight_scale_2 float    one fp32 tensor scale
 * and the weight value is  e2m1(q) * e4m3(s) * weight_scale_2.
 * A static fp32 input_scale per linear is stored for W4A4.
 *
 * Conventions for every call below
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; the
 *     library never allocates, frees or keeps a pointer after returning.
 *     Tensors are row-major and contiguous.  bf16 tensors are passed as
 *     uint16_t bit patterns.
 *   - Every pointer must be 16-byte aligned (NVFP4_ERR_ALIGN otherwise).
 *   - Calls are asynchronous on the caller's CUDA stream (0 = legacy default
 *     stream) and return before the work is done.  The return value reports
 *     host-side validation and launch errors only.
 *   - Host validation happens before any launch: bad shapes, NULL pointers,
 *     misalignment and a too-small workspace are rejected and nothing is
 *     enqueued.  Problems only the device can see (a user-supplied expert id
 *     out of range) are written to the optional int32 status word d_status
 *     as an nvfp4_status value; kernels never trap.
 *   - K (the reduction length of a GEMM) must be a multiple of 64 (the
 *     decode-shaped kernel streams K in 64-wide chunks: 4 lanes x 16 values,
 *     one e4m3 scale each); N (output features) a multiple of 16; row
 *     counts M or T may be 0 (no-op).
 *   - Activations and weights must be finite (their NaN/Inf behaviour is
 *     unspecified); non-finite router logits follow moe_route_permute.
 *   - Workspace contents are scratch owned by the call until it completes on
 *     the stream; two calls that overlap on the GPU must not share one.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* cudaStream_t;

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1, /* NULL pointer, negative size, bad enum       */
    NVFP4_ERR_SHAPE = 2,       /* K % 64, N % 16, top_k > E, E > 1024, ...     */
    NVFP4_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned             */
    NVFP4_ERR_WORKSPACE = 4,   /* ws_bytes smaller than the size query's       */
    NVFP4_ERR_UNSUPPORTED = 5, /* no device / not sm_100-family                */
    NVFP4_ERR_CUDA = 6,        /* a CUDA launch failed (cudaGetLastError)      */
    NVFP4_ERR_TIMEOUT = 7,     /* a bounded device wait gave up (d_status)     */
    NVFP4_ERR_DEVICE_INPUT = 8 /* device saw an out-of-range id (d_status)     */
} nvfp4_status;

/* One stacked NVFP4 tensor bank: codes [E, N, K/2], scales [E, N, K/16],
 * weight_scale_2 [E] (E = 1 for a single tensor). */
typedef struct {
    const uint8_t* codes;
    const uint8_t* scales;
    const float* weight_scale_2;
} nvfp4_w;

/* The routed experts of one layer (model card "GLM-5.3-Flash-NVFP4-W4A4-
 * Experts", "Quantization boundary": gate_proj, up_proj, down_proj per
 * expert).  gate/up: N = F, K = d; down: N = d, K = F. */
typedef struct {
    nvfp4_w gate, up, down;
    int E, d, F;
} nvfp4_moe_weights;

/* ------------------------------------------------------------------------
 * nvfp4_quantize_weights -- ModelOpt's NVFP4 recipe, applied to each of
 * `batch` bf16 tensors [N, K] (TensorFold #308, "What the branch does": BF16
 * experts packed to NVFP4 by ModelOpt's recipe at load, one projection at a
 * time).  Per tensor b:
 *   weight_scale_2[b] = amax / 2688                      (fp32, 2688 = 6*448)
 *   per 16-block: s = e4m3_rn_sat((block_amax / 6) / weight_scale_2[b])
 *   per element:  q = e2m1_rn_sat(w / (e4m3(s) * weight_scale_2[b]))
 * (IEEE fp32 round-to-nearest division and product in exactly this order; a
 * block whose scale rounds to 0 gets all-zero codes.)
 *   w       [batch, N, K] bf16     codes [batch, N, K/2]   scales [batch, N, K/16]
 *   weight_scale_2 [batch] fp32
 *   ws      scratch of at least nvfp4_quantize_weights_workspace_size() bytes
 * K must be a multiple of 16 and batch at most 65535 (NVFP4_ERR_SHAPE
 * otherwise).  Two device passes (global amax, then codes).
 * --------------------------------------------------------------------- */
nvfp4_status nvfp4_quantize_weights(const uint16_t* w_bf16, int batch, int N, int K,
                                    uint8_t* codes, uint8_t* scales, float* weight_scale_2,
                                    void* ws, size_t ws_bytes, cudaStream_t stream);
size_t nvfp4_quantize_weights_workspace_size(int batch, int N, int K);

/* ------------------------------------------------------------------------
 * nvfp4_quantize_weights_noalloc -- the same recipe and outputs as
 * nvfp4_quantize_weights, for callers that cannot allocate device memory
 * (the pages have no counterpart: a convenience of this library).
 * Such callers include code that may not call cudaMalloc because another
 * component owns the device's memory (a pool planned ahead), plain C
 * loaders with no allocator of their own, and loops that must not call
 * cudaMalloc because it can implicitly synchronise the device.  Instead of
 * a caller workspace it uses a fixed scratch array (one float per tensor,
 * at most nvfp4_quantize_weights_noalloc_max_batch() = 4096 tensors per
 * call, 16 KB of device memory on every GPU that loads the library, held
 * until the process exits) and allocates nothing.
 *   - batch above the maximum: NVFP4_ERR_SHAPE, nothing enqueued.
 *   - Every call looks up the array's device address in the current
 *     context (cudaGetSymbolAddress, with the caller's device current;
 *     nothing is cached, so calls after cudaDeviceReset are served too).
 *     The first call of a process on a device may load the library's
 *     device code: make it before any stream capture.
 *   - All calls on a device share the one array: calls that can overlap on
 *     the GPU (other streams, other host threads) race; order them.
 *   - The scratch is cleared on each call; outputs as for
 *     nvfp4_quantize_weights.
 * --------------------------------------------------------------------- */
nvfp4_status nvfp4_quantize_weights_noalloc(const uint16_t* w_bf16, int batch, int N, int K,
                                            uint8_t* codes, uint8_t* scales, float* weight_scale_2,
                                            cudaStream_t stream);
int nvfp4_quantize_weights_noalloc_max_batch(void);

/* ------------------------------------------------------------------------
 * nvfp4_quantize_act -- static-scale NVFP4 quantisation of activation rows
 * (TensorFold #308 "The checkpoint": input_scale stored for static
 * activations; W4A4 model card: calibrated static activation scales).
 * Output row r (0 <= r < M) quantises source row
 *     src(r) = row_to_slot ? row_to_slot[r] / top_k : r
 * of x [*, K] with tensor scale
 *     gs(r) = expert_offsets ? input_scale[e] where offsets[e] <= r < offsets[e+1]
 *                            : input_scale[0]
 * using the same block rule as the weight recipe with gs in place of
 * weight_scale_2 (block scales above 448 saturate to 448, codes to +-6).
 *   codes [M, K/2], scales [M, K/16].  K % 16 == 0.  E <= 1024.
 * --------------------------------------------------------------------- */
nvfp4_status nvfp4_quantize_act(const uint16_t* x_bf16, int M, int K,
                                const int32_t* row_to_slot, int top_k,
                                const float* input_scale, const int32_t* expert_offsets, int E,
                                uint8_t* codes, uint8_t* scales, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_router_logits -- the BF16 router GEMM in front of routing
 * (TensorFold #308 "The checkpoint": the router is BF16, not NVFP4):
 *   logits[t, e] = sum_k x[t, k] * w_router[e, k]     (fp32)
 *   x_bf16 [T, d], w_router_bf16 [E, d], logits [T, E], all row-major,
 *   device pointers owned by the caller, 16-byte aligned.
 * Every bf16 product is exact in fp32; the k-sum is fp32 (tensor cores),
 * so |logits - exact| <= d * 2^-24 * sum_k |x[t,k] w[e,k]|.
 * d % 64 == 0, 1 <= E <= 512; T == 0 is a no-op.  d_status (nullable)
 * receives NVFP4_ERR_TIMEOUT if a bounded wait expired.  Asynchronous on
 * the stream; returns NVFP4_ERR_* for bad arguments before any launch.
 * --------------------------------------------------------------------- */
nvfp4_status moe_router_logits(const uint16_t* x_bf16, int T, int d, const uint16_t* w_router_bf16,
                               int E, float* logits, int32_t* d_status, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_shared_expert -- the BF16 shared-expert MLP after the routed layer
 * (TensorFold #308 "The checkpoint": the shared expert is BF16, next to the
 * NVFP4 routed experts).  For every token t:
 *   G = bf16(x Wg^T)   U = bf16(x Wu^T)   h = bf16(silu(G) * U)
 *   out[t] = bf16(out[t] + h Wd^T)          (fp32 sums; out holds the
 *                                            routed layer's bf16 result)
 *   x_bf16 [T, d], w_gate_bf16 / w_up_bf16 [Fs, d], w_down_bf16 [d, Fs],
 *   out_bf16 [T, d] read and written; row-major device pointers owned by
 *   the caller, 16-byte aligned.  d % 256 == 0, Fs % 128 == 0.
 *   ws: at least moe_shared_expert_workspace_size(T, Fs) bytes (h).
 * Tensor cores (tcgen05, bf16 operands by TMA).  T == 0 is a no-op;
 * d_status (nullable) receives NVFP4_ERR_TIMEOUT if a bounded wait expired.
 * --------------------------------------------------------------------- */
nvfp4_status moe_shared_expert(const uint16_t* x_bf16, int T, int d, const uint16_t* w_gate_bf16,
                               const uint16_t* w_up_bf16, const uint16_t* w_down_bf16, int Fs,
                               uint16_t* out_bf16, void* ws, size_t ws_bytes, int32_t* d_status,
                               cudaStream_t stream);
size_t moe_shared_expert_workspace_size(int T, int Fs);

/* ------------------------------------------------------------------------
 * moe_route_permute -- the BF16 router's logits to expert-contiguous rows
 * (TensorFold #308: router BF16, routed experts through one grouped
 * kernel).  Per token t: softmax over the E logits, the top_k experts in
 * descending order (ties -> lower expert id), and their weights
 * renormalised over the chosen top_k (exp, sum and division in fp64, one
 * rounding to fp32).  NaN logits rank as -inf; a token whose top logit is
 * +inf gives its +inf entries equal weights (the rest 0), one whose chosen
 * logits are all -inf gets 1/top_k each:
 *   topk_ids [T, top_k] int32, topk_w [T, top_k] fp32.
 * Then a stable permutation of the R = T*top_k (token, slot) pairs by
 * expert (order: expert, token, slot):
 *   expert_offsets [E+1]: first row of each expert, offsets[E] = R
 *   row_to_slot [R]: row -> t*top_k + slot;  slot_to_row [R]: the inverse.
 * Per-expert histogram, warp-scan prefix sum and scatter; the result is
 * deterministic (no atomics decide an order).  E <= 1024, top_k <= 32.
 *   ws: at least moe_route_permute_workspace_size(T, E, top_k) bytes.
 * --------------------------------------------------------------------- */
nvfp4_status moe_route_permute(const float* logits, int T, int E, int top_k,
                               int32_t* topk_ids, float* topk_w, int32_t* expert_offsets,
                               int32_t* row_to_slot, int32_t* slot_to_row,
                               void* ws, size_t ws_bytes, cudaStream_t stream);
size_t moe_route_permute_workspace_size(int T, int E, int top_k);

/* ------------------------------------------------------------------------
 * nvfp4_moe_w4a16 / nvfp4_moe_w4a4 -- the routed-expert layer.
 * TensorFold #308 "What the branch does": routed experts run through a
 * grouped NVFP4 expert kernel over bf16 rows (W4A16) with weight_scale_2 as
 * the per-expert multiplier; the checkpoint's own FP4 x FP4 math (W4A4)
 * quantises the activations with the stored static input_scale.  Per token
 * t and slot j with e = topk_ids[t, j]:
 *   G = bf16(ws2_g[e] * x W_g[e]^T)   U = bf16(ws2_u[e] * x W_u[e]^T)
 *   h = bf16(silu(G) * U)
 *   Y = ws2_d[e] * h W_d[e]^T         (fp32)
 *   out[t] = bf16(sum_j topk_w[t, j] * Y_j)
 * W4A4: x is first quantised per (t, e) with input_scale_w13[e]; h with
 * input_scale_w2[e]; the GEMMs multiply FP4 x FP4 with fp32 accumulation.
 *   x [T, d] bf16, logits [T, E] fp32, out [T, d] bf16.
 *   logits == NULL: the routing arrays already in the workspace (written by
 *   an earlier call or by moe_route_permute into the views that
 *   nvfp4_moe_workspace_views returns) are used; out-of-range expert ids
 *   are then reported through d_status (NVFP4_ERR_DEVICE_INPUT).
 *   ws: at least nvfp4_moe_workspace_size(T, E, top_k, d, F, mode) bytes
 *   (mode 0 = W4A16, 1 = W4A4); d_status: optional device int32.
 * Shapes: d % 64 == 0, F % 64 == 0, E <= 1024, 1 <= top_k <= min(E, 32).
 * --------------------------------------------------------------------- */
nvfp4_status nvfp4_moe_w4a16(const uint16_t* x_bf16, int T, const float* logits, int top_k,
                             const nvfp4_moe_weights* w, uint16_t* out_bf16,
                             void* ws, size_t ws_bytes, int32_t* d_status, cudaStream_t stream);
nvfp4_status nvfp4_moe_w4a4(const uint16_t* x_bf16, int T, const float* logits, int top_k,
                            const nvfp4_moe_weights* w, const float* input_scale_w13,
                            const float* input_scale_w2, uint16_t* out_bf16,
                            void* ws, size_t ws_bytes, int32_t* d_status, cudaStream_t stream);
size_t nvfp4_moe_workspace_size(int T, int E, int top_k, int d, int F, int mode);

/* Device pointers to the routing arrays inside an nvfp4_moe workspace (the
 * same arrays moe_route_permute produces), so that a caller can read them
 * back or fill them.  Any output pointer may be NULL. */
nvfp4_status nvfp4_moe_workspace_views(void* ws, int T, int E, int top_k, int d, int F, int mode,
                                       int32_t** topk_ids, float** topk_w,
                                       int32_t** expert_offsets, int32_t** row_to_slot,
                                       int32_t** slot_to_row);

/* Device pointers to the per-row intermediates inside an nvfp4_moe
 * workspace, as the last call that used it left them, rows in the permuted
 * (expert-contiguous) order of row_to_slot (R = T * top_k rows):
 *   mode 0 (W4A16): h_bf16 [R, F] = bf16(silu(G) * U);
 *   mode 1 (W4A4):  xq [R, d/2], xs [R, d/16] (the NVFP4 x rows under
 *                   input_scale_w13) and hq [R, F/2], hs [R, F/16] (h
 *                   requantised under input_scale_w2).
 * Pointers of the other mode are set to NULL; any output pointer may be
 * NULL.  The pages have no counterpart: an inspection helper (the parity
 * tests read the intermediates through it). */
nvfp4_status nvfp4_moe_workspace_intermediates(void* ws, int T, int E, int top_k, int d, int F, int mode,
                                               uint16_t** h_bf16, uint8_t** xq, uint8_t** xs,
                                               uint8_t** hq, uint8_t** hs);

/* ------------------------------------------------------------------------
 * moe_gather_rows / moe_combine_rows -- the two ends of an expert-parallel
 * routed layer (W4A4 model card "GLM-5.3-Flash-NVFP4-W4A4-Experts",
 * "Validation": the routed experts run expert-parallel over several GPUs;
 * TensorFold #308 "What the branch does": the grouped kernel takes the
 * routed rows expert by expert).  With the permutation of
 * moe_route_permute (R = T * top_k rows, expert-contiguous):
 *   moe_gather_rows:  rows_out[r] = x[row_to_slot[r] / top_k]   [R, d] bf16
 *                     expert_of_row[r] = e, offsets[e] <= r < offsets[e+1]
 *                     (nullable; then expert_offsets and E are unused)
 *     -- the rows a rank sends, in order, to the ranks owning the experts;
 *   moe_combine_rows: out[t] = bf16(sum_j topk_w[t, j] * y[slot_to_row[t*k + j]])
 *                     (fp32, j in slot order), y bf16 [R, d] in the same
 *                     row order -- the combine of the rows that come back.
 * d % 8 == 0; device pointers owned by the caller, 16-byte aligned; T == 0
 * is a no-op; asynchronous on the stream.
 * --------------------------------------------------------------------- */
nvfp4_status moe_gather_rows(const uint16_t* x_bf16, int T, int d, const int32_t* row_to_slot, int top_k,
                             const int32_t* expert_offsets, int E, uint16_t* rows_out, int32_t* expert_of_row,
                             cudaStream_t stream);
nvfp4_status moe_combine_rows(const uint16_t* y_bf16, const int32_t* slot_to_row, const float* topk_w, int T,
                              int top_k, int d, uint16_t* out_bf16, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * nvfp4_set_kernel_choice -- which kernels the later nvfp4_moe_* and
 * nvfp4_linear calls of this process run (the pages have no counterpart):
 *   0 = by shape (the default: the prompt-shaped tensor-core kernels once
 *       the experts average 32 or more routed rows, else the decode-shaped
 *       streaming kernels);
 *   1 = the decode-shaped kernels for every shape;
 *   2 = the prompt-shaped kernels wherever the shapes allow them;
 *   3 = as 1, with the decode-shaped layer as two launches (gate/up, then
 *       down + combine);
 *   4 = as 1, with the decode-shaped layer as one persistent launch where
 *       its shape allows it (d and F multiples of 256).
 * Choices 0 and 1 take whichever decode-shaped form is faster for the
 * shape.  For tests and measurements that cover every kernel at one size.
 * Takes effect for calls made after it returns; returns
 * NVFP4_ERR_INVALID_ARG for any other value.
 * --------------------------------------------------------------------- */
nvfp4_status nvfp4_set_kernel_choice(int choice);

/* ------------------------------------------------------------------------
 * nvfp4_linear -- dense NVFP4 linear over bf16 rows (TensorFold #308: the
 * dense MLP runs on Fp4Linear, gate and up apart since their tensor scales
 * differ).
 *   w_up == NULL:  out [M, N] = bf16(ws2 * x W^T)
 *   w_up != NULL:  out [M, N] = bf16(silu(bf16(ws2 * x W^T)) * bf16(ws2_up * x W_up^T))
 * x [M, K] bf16, w / w_up single tensors [N, K] (E = 1).  K % 64 == 0,
 * N % 16 == 0.  ws: at least nvfp4_linear_workspace_size(M, K, N) bytes.
 * --------------------------------------------------------------------- */
nvfp4_status nvfp4_linear(const uint16_t* x_bf16, int M, int K, const nvfp4_w* w, int N,
                          const nvfp4_w* w_up, uint16_t* out_bf16,
                          void* ws, size_t ws_bytes, cudaStream_t stream);
size_t nvfp4_linear_workspace_size(int M, int K, int N);

/* ------------------------------------------------------------------------
 * Helpers.
 * nvfp4_status_string: a static, human-readable name of a status.
 * nvfp4_launch_count: number of kernels this library has launched in this
 *   process (all devices, all streams), for accounting.
 * nvfp4_profile_enable(1): from now on, every launch is bracketed by CUDA
 *   events on its stream; nvfp4_profile_collect synchronises on those events,
 *   writes per-kernel-name totals (name, launches, milliseconds) for up to
 *   `max` names, resets the totals and returns the number of names.
 *   names must hold max * 64 chars.  Timing adds event records between
 *   launches; turn it off (0) for headline measurements.
 * --------------------------------------------------------------------- */
const char* nvfp4_status_string(nvfp4_status s);
uint64_t nvfp4_launch_count(void);

/* ------------------------------------------------------------------------
 * nvfp4_selftest_bounded_wait: exercises the failure detection every
 * kernel of the library relies on (the pages have no counterpart).  One CTA
 * waits on an mbarrier that nothing arrives on; the bounded wait gives up
 * after about 2 s of SM clock, stores NVFP4_ERR_TIMEOUT in *d_status and the
 * kernel returns normally (no trap, no fault; the context stays usable).
 * d_status: device int32, 16-byte aligned, caller-owned.  Asynchronous on
 * `stream`; returns NVFP4_ERR_INVALID_ARG / NVFP4_ERR_ALIGN on a bad pointer.
 * --------------------------------------------------------------------- */
nvfp4_status nvfp4_selftest_bounded_wait(int32_t* d_status, cudaStream_t stream);
void nvfp4_profile_enable(int on);
int nvfp4_profile_collect(int max, char* names, int* launches, double* ms);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4MOE_H */
