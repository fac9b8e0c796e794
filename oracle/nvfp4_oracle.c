/*
 * nvfp4_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * A plain, slow, obviously-correct CPU restatement of what the NVFP4
 * routed-expert MoE layer computes.  Only the test suite, the smoke check in
 * __graft_entry__.py and the cpu_baseline leg of bench.py may load it.  It
 * shares no code, header, table or helper with the CUDA library: every
 * codec below is written from the format definitions, every sum is an fp64
 * loop, and nothing is blocked, fused or reordered.
 *
 * Sources (web pages, cited by title and section):
 *   [TF308]  TensorFold issue #308, "GLM-5.3-Flash on CUDA: read
 *            nvidia/GLM-5.3-Flash-NVFP4 (ModelOpt NVFP4) as stored, W4A16".
 *            "The checkpoint": routed experts and dense MLP are ModelOpt
 *            NVFP4 -- e2m1 codes, an e4m3 scale per 16 inputs, an fp32
 *            weight_scale_2 per tensor, a stored static input_scale; the
 *            router is BF16.
 *            "What the branch does": grouped expert kernel over bf16 rows
 *            (W4A16) with weight_scale_2 as the per-expert multiplier; dense
 *            MLP with gate and up apart (different tensor scales); FP4 x FP4
 *            as the checkpoint's own math (W4A4); BF16 experts packed to
 *            NVFP4 by ModelOpt's recipe one projection at a time.
 *   [W4A4]   Model card "GLM-5.3-Flash-NVFP4-W4A4-Experts", "Quantization
 *            boundary": e2m1 weights, group size 16, gate/up/down per
 *            expert, calibrated static activation scales (W4A4).
 *
 * The pages give the format and the data flow but no formula for the router
 * or the activation; the readings taken here (softmax over the experts,
 * top-k with ties to the lower id, weights renormalised over the chosen k;
 * SwiGLU = silu(gate) * up; the ModelOpt recipe global = amax / (6*448),
 * block scale = e4m3(block_amax / 6 / global), codes by round-to-nearest-even)
 * are the plainest ones and are listed with the rest in the design notes.
 *
 * Beside the layer: the BF16 router GEMM (orc_router_logits: fp64 sums of
 * exact bf16 products, and their |.| sums for the fp32 error bound) and the
 * BF16 shared-expert MLP (orc_shared_expert: the same SwiGLU rounding points,
 * added to the routed output and rounded once).
 *
 * Rounding points (the same places the kernels round):
 *   G = bf16(ws2_g * sum x*w_g)   U = bf16(ws2_u * sum x*w_u)       (R1)
 *   h = bf16(silu(G) * U)                                            (R2)
 *   Y = ws2_d * sum h*w_d   (unrounded; with the R3 switch, bf16(Y) (R3))
 *   out[t] = bf16(sum_j w_j * Y_j)                                   (R4)
 * R3 is the rounding point of the kernels that keep each routed row's Y in
 * bf16 for the slot-ordered combine (the prompt-shaped path); without it Y
 * stays unrounded, as in the decode-shaped path.
 * All sums here are fp64.  Scale arithmetic that decides a code (block
 * scale, element / scale) is done in fp32 in the order the recipe states,
 * because that is the precision in which the codes are defined.
 *
 * The layer groups its (token, slot) pairs by expert and dequantises each
 * touched expert's three projections once (exact in fp32); every pair is
 * then evaluated on its own with plain fp64 loops.  Besides the bf16
 * outputs it can return each output's value before its final rounding and
 * the sum of |terms| behind it (the scale of the error bound of an fp32
 * evaluation), and the gate / up values before their rounding, which the
 * parity tests use to tell a legitimate rounding flip from an error.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* bf16                                                                */
/* ------------------------------------------------------------------ */

/* bf16 bits -> float: bf16 is the upper half of an IEEE binary32. */
static float bf16_bits_to_float(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a double to the nearest bf16 value (8 significant bits), ties to
 * even, by scaling the significand and calling nearbyint (default rounding
 * mode = to nearest, ties to even).  Subnormal bf16 keeps fewer bits. */
double orc_round_bf16(double v) {
    if (v == 0.0 || !isfinite(v)) return v;
    int e;
    double m = frexp(v, &e);          /* v = m * 2^e, 0.5 <= |m| < 1 */
    int bits = 8;                     /* significant bits of bf16 */
    int unbiased = e - 1;             /* v = 1.xxx * 2^unbiased     */
    if (unbiased < -126) bits -= (-126 - unbiased);
    if (bits < 0) return copysign(0.0, v);
    double r = nearbyint(ldexp(m, bits));
    return ldexp(r, e - bits);
}

/* ------------------------------------------------------------------ */
/* e2m1 (FP4): sign bit 3, magnitudes {0,.5,1,1.5,2,3,4,6} for codes 0..7 */
/* ------------------------------------------------------------------ */
static const double E2M1_MAGNITUDE[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_decode(int code) {
    double m = E2M1_MAGNITUDE[code & 7];
    return (code & 8) ? -m : m;
}

/* Nearest e2m1 magnitude to |v| by brute force over the eight values; an
 * exact tie goes to the even code (round-to-nearest-even); |v| > 6
 * saturates to 6 (the format has no infinity).  The sign bit is kept,
 * so a tiny negative value gives code 8 (-0). */
int orc_e2m1_encode(float v) {
    double a = fabs((double)v);
    if (a > 6.0) a = 6.0; /* saturate first: for huge |v| the fp64 distances below would tie */
    int best = 0;
    double bestd = fabs(a - E2M1_MAGNITUDE[0]);
    for (int c = 1; c < 8; ++c) {
        double d = fabs(a - E2M1_MAGNITUDE[c]);
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return best | (signbit(v) ? 8 : 0);
}

/* ------------------------------------------------------------------ */
/* e4m3 (FP8, "fn" variant): bias 7, no infinities, 0x7F/0xFF are NaN   */
/* ------------------------------------------------------------------ */
double orc_e4m3_decode(int b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? m * ldexp(1.0, -9) : (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return s ? -v : v;
}

/* Nearest non-negative finite e4m3 value by brute force over bytes
 * 0..126; ties go to the even byte (even mantissa); values above 448
 * saturate to 448 (0x7E). */
int orc_e4m3_encode_nonneg(float v) {
    double a = (double)v;
    if (a > 448.0) a = 448.0; /* saturate first, as for e2m1 */
    int best = 0;
    double bestd = fabs(a - orc_e4m3_decode(0));
    for (int b = 1; b <= 126; ++b) {
        double d = fabs(a - orc_e4m3_decode(b));
        if (d < bestd || (d == bestd && (b & 1) == 0)) {
            best = b;
            bestd = d;
        }
    }
    return best;
}

/* ------------------------------------------------------------------ */
/* NVFP4 block quantisation of one row of K values with a given fp32     */
/* tensor scale gs (weight_scale_2 for weights, input_scale for          */
/* activations).  ModelOpt recipe, per 16-block j:                       */
/*   bam = max |v|;  sf = (bam / 6) / gs  (two fp32 divisions);           */
/*   s = e4m3(sf);  S = dec(s);                                          */
/*   q_i = e2m1(v_i / (S * gs))  (fp32 product, then fp32 division).     */
/* A block with S == 0 (all zero, or sf below half the smallest e4m3    */
/* subnormal) gets scale byte 0 and all codes 0.  Codes are packed two  */
/* per byte, even index in the low nibble.                               */
/* ------------------------------------------------------------------ */
static void quantize_row(const float* v, int64_t K, float gs, uint8_t* codes, uint8_t* scales) {
    for (int64_t j = 0; j < K / 16; ++j) {
        float bam = 0.0f;
        for (int i = 0; i < 16; ++i) bam = fmaxf(bam, fabsf(v[16 * j + i]));
        int s = 0;
        float S = 0.0f;
        if (gs > 0.0f) {
            float sf = (bam / 6.0f) / gs;
            s = orc_e4m3_encode_nonneg(sf);
            S = (float)orc_e4m3_decode(s);
        }
        scales[j] = (uint8_t)s;
        for (int i = 0; i < 16; i += 2) {
            int q0 = 0, q1 = 0;
            if (S != 0.0f) {
                float denom = S * gs;
                q0 = orc_e2m1_encode(v[16 * j + i] / denom);
                q1 = orc_e2m1_encode(v[16 * j + i + 1] / denom);
            }
            codes[(16 * j + i) / 2] = (uint8_t)(q0 | (q1 << 4));
        }
    }
}

/* ModelOpt NVFP4 weight recipe for one [N, K] bf16 tensor:
 * weight_scale_2 = amax / 2688 (2688 = 6 * 448, fp32 division), then
 * quantize_row with gs = weight_scale_2. */
void orc_quantize_tensor(const uint16_t* w, int64_t N, int64_t K, uint8_t* codes,
                         uint8_t* scales, float* weight_scale_2) {
    float amax = 0.0f;
    for (int64_t i = 0; i < N * K; ++i) amax = fmaxf(amax, fabsf(bf16_bits_to_float(w[i])));
    float ws2 = amax / 2688.0f;
    *weight_scale_2 = ws2;
#pragma omp parallel
    {
        float* row = (float*)malloc(sizeof(float) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t k = 0; k < K; ++k) row[k] = bf16_bits_to_float(w[n * K + k]);
            quantize_row(row, K, ws2, codes + n * (K / 2), scales + n * (K / 16));
        }
        free(row);
    }
}

/* Static-scale activation quantisation: row r of the bf16 [M, K] matrix is
 * quantised with its own tensor scale gs[r] (the input_scale of the expert
 * the row is routed to). */
void orc_quantize_rows(const uint16_t* x, int64_t M, int64_t K, const float* gs,
                       uint8_t* codes, uint8_t* scales) {
#pragma omp parallel
    {
        float* row = (float*)malloc(sizeof(float) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < M; ++r) {
            for (int64_t k = 0; k < K; ++k) row[k] = bf16_bits_to_float(x[r * K + k]);
            quantize_row(row, K, gs[r], codes + r * (K / 2), scales + r * (K / 16));
        }
        free(row);
    }
}

/* Dequantised weight element n, k of one [N, K] tensor, WITHOUT the tensor
 * scale: dec(q) * dec(s).  The product is exact in fp32 and in fp64. */
static double deq(const uint8_t* codes, const uint8_t* scales, int64_t K, int64_t n, int64_t k) {
    int byte = codes[(n * K + k) / 2];
    int q = (k & 1) ? (byte >> 4) : (byte & 15);
    return orc_e2m1_decode(q) * orc_e4m3_decode(scales[n * (K / 16) + k / 16]);
}

void orc_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t N, int64_t K,
                    double* out) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) out[n * K + k] = deq(codes, scales, K, n, k);
}

/* ------------------------------------------------------------------ */
/* Router GEMM ([TF308] "The checkpoint": the router is BF16):          */
/*   logits[t][e] = sum_k x[t][k] * w[e][k]                             */
/* as an fp64 loop in k order (every bf16 product is exact in fp64),    */
/* and abs_sum[t][e] = sum_k |x[t][k] * w[e][k]|, the scale of the      */
/* error bound of any fp32 evaluation of the same sum.                  */
/* ------------------------------------------------------------------ */
void orc_router_logits(const uint16_t* x, int64_t T, int64_t d, const uint16_t* w, int64_t E,
                       double* logits, double* abs_sum) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t e = 0; e < E; ++e) {
            double s = 0.0, a = 0.0;
            for (int64_t k = 0; k < d; ++k) {
                const double p = (double)bf16_bits_to_float(x[t * d + k]) * (double)bf16_bits_to_float(w[e * d + k]);
                s += p;
                a += fabs(p);
            }
            logits[t * E + e] = s;
            abs_sum[t * E + e] = a;
        }
}

/* ------------------------------------------------------------------ */
/* Routing: softmax over E logits, top-k descending (ties -> lower      */
/* expert id), weights renormalised over the k chosen:                  */
/*   w_j = exp(l_j - l_max) / sum_{i in top-k} exp(l_i - l_max)         */
/* (the softmax normaliser cancels).  fp64, stored as fp32.             */
/* Non-finite logits (the pages never meet them; the reading taken):    */
/* NaN ranks as -inf; if the top logit is +inf the +inf entries among   */
/* the k share the weight equally and the rest get 0; if every chosen   */
/* logit is -inf the k weights are 1/k.                                 */
/* Then a stable counting sort of the T*k (token, slot) pairs by expert  */
/* (order: expert, then token, then slot):                               */
/*   offsets[e] = number of pairs routed to experts < e;                 */
/*   row_to_slot[row] = t*k + slot;  slot_to_row[t*k + slot] = row.      */
/* ------------------------------------------------------------------ */
static double rank_key(float v) { return isnan(v) ? -INFINITY : (double)v; }

void orc_route(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w,
               int32_t* offsets, int32_t* row_to_slot, int32_t* slot_to_row) {
    char* chosen = (char*)malloc((size_t)E);
    double* num = (double*)malloc(sizeof(double) * (size_t)k);
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        memset(chosen, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (chosen[e]) continue;
                if (best < 0 || rank_key(l[e]) > rank_key(l[best])) best = e;
            }
            chosen[best] = 1;
            ids[t * k + j] = best;
        }
        const double lmax = rank_key(l[ids[t * k]]);
        double den = 0.0;
        for (int j = 0; j < k; ++j) {
            const double lj = rank_key(l[ids[t * k + j]]);
            if (lmax == INFINITY) num[j] = (lj == INFINITY) ? 1.0 : 0.0;
            else if (lmax == -INFINITY) num[j] = 1.0;
            else num[j] = exp(lj - lmax);
            den += num[j];
        }
        for (int j = 0; j < k; ++j) w[t * k + j] = (float)(num[j] / den);
    }
    free(num);
    free(chosen);

    int64_t R = T * k;
    int64_t* count = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    for (int64_t i = 0; i < R; ++i) count[ids[i]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + (int32_t)count[e];
    int64_t* fill = (int64_t*)malloc(sizeof(int64_t) * (size_t)E);
    for (int e = 0; e < E; ++e) fill[e] = offsets[e];
    for (int64_t i = 0; i < R; ++i) {
        int64_t row = fill[ids[i]]++;
        row_to_slot[row] = (int32_t)i;
        slot_to_row[i] = (int32_t)row;
    }
    free(fill);
    free(count);
}

/* ------------------------------------------------------------------ */
/* The layer.                                                            */
/* ------------------------------------------------------------------ */
static double silu(double g) { return g / (1.0 + exp(-g)); }

/* Dequantised weights of one [N, K] tensor without the tensor scale,
 * dec(q) * dec(s) per element, as float: exact, since the product of an
 * e2m1 value and an e4m3 value has at most 6 significant bits and lies in
 * [2^-10, 2688]. */
static void dequant_f32(const uint8_t* codes, const uint8_t* scales, int64_t N, int64_t K, float* out) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) out[n * K + k] = (float)deq(codes, scales, K, n, k);
}

/* One linear over one input vector a[K] (fp64) and dequantised weights
 * W [N, K]: out[n] = sum_k a[k] * W[n, k], an fp64 sum in k order (every
 * product is exact in fp64).  abs_out, if not NULL, receives
 * sum_k |a[k] * W[n, k]| (the scale of the error bound of any fp32
 * evaluation of the same sum). */
static void matvec(const double* a, const float* W, int64_t N, int64_t K, double* out, double* abs_out) {
    for (int64_t n = 0; n < N; ++n) {
        const float* wr = W + n * K;
        double s = 0.0, sa = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double p = a[k] * (double)wr[k];
            s += p;
            sa += fabs(p);
        }
        out[n] = s;
        if (abs_out) abs_out[n] = sa;
    }
}

/* Quantise a float vector with tensor scale gs and return it dequantised
 * (dec(q) * dec(s), no tensor scale) in fp64; the codes and scales are
 * also written to c / s when those are not NULL. */
static void quant_dequant(const float* v, int64_t K, float gs, double* out, uint8_t* c_out, uint8_t* s_out) {
    uint8_t* c = (uint8_t*)malloc((size_t)(K / 2));
    uint8_t* s = (uint8_t*)malloc((size_t)(K / 16));
    quantize_row(v, K, gs, c, s);
    for (int64_t k = 0; k < K; ++k) out[k] = deq(c, s, K, 0, k);
    if (c_out) memcpy(c_out, c, (size_t)(K / 2));
    if (s_out) memcpy(s_out, s, (size_t)(K / 16));
    free(c);
    free(s);
}

/* Optional outputs of orc_moe_layer_ex (any pointer may be NULL); n is the
 * number of listed tokens:
 *   out_pre [n, d]    sum_j w_j * Y_j before the final bf16 rounding
 *   out_abs [n, d]    sum_j |w_j| * scale_j * sum_f |h_f * W_d[.,f]|: the
 *                     scale of the error bound of an fp32 evaluation
 *   g_pre, u_pre [n, k, F]  the gate / up values before their bf16 rounding
 *   g_abs, u_abs [n, k, F]  their sums of |terms| times the same scales
 *   h  [n, k, F]      h (bf16 values)
 *   xq, xs [n, k, d/2], [n, k, d/16]  W4A4: the pair's NVFP4 x row
 *   hq, hs [n, k, F/2], [n, k, F/16]  W4A4: the pair's NVFP4 h row
 *   y_pre, y_abs [n, k, d]  each pair's Y before the R3 rounding and its
 *                     scale * sum_f |h_f * W_d| */
typedef struct {
    double* out_pre;
    double* out_abs;
    double* g_pre;
    double* u_pre;
    double* g_abs;
    double* u_abs;
    float* h;
    uint8_t* xq;
    uint8_t* xs;
    uint8_t* hq;
    uint8_t* hs;
    double* y_pre;
    double* y_abs;
} orc_layer_extras;

/*
 * Routed-expert MoE layer for the tokens listed in `tokens` (n_tokens of
 * them), given routing ids/w [T, k].  mode 0 = W4A16 (bf16 activations),
 * mode 1 = W4A4 (activations quantised to NVFP4 with the static per-expert
 * input_scale: is13[e] before gate/up, is2[e] before down).
 * Weight banks are stacked over experts: gate/up codes [E, F, d/2], scales
 * [E, F, d/16], ws2 [E]; down codes [E, d, F/2], scales [E, d, F/16].
 * out[i, :] receives bf16(sum_j w_j * Y_j) for token tokens[i] (as float);
 * round_y != 0 rounds each Y_j to bf16 first (R3).
 * The (token, slot) pairs are grouped by expert so that each touched
 * expert's three projections are dequantised once; every pair is then
 * evaluated on its own, with the same fp64 sums in the same order.
 */
void orc_moe_layer_ex(int mode, const uint16_t* x, int64_t T, int64_t d, int64_t F, int E, int k,
                      const int32_t* ids, const float* w,
                      const uint8_t* gq, const uint8_t* gs, const float* g_ws2,
                      const uint8_t* uq, const uint8_t* us, const float* u_ws2,
                      const uint8_t* dq, const uint8_t* ds, const float* d_ws2,
                      const float* is13, const float* is2, int round_y,
                      const int32_t* tokens, int64_t n_tokens, float* out, const orc_layer_extras* ex) {
    (void)T;
    const int64_t n_pairs = n_tokens * k;
    /* Y_j of every (token, slot) pair (and the |term| sums), then the
     * weighted sum over the slots in slot order. */
    double* Y = (double*)malloc(sizeof(double) * (size_t)(n_pairs * d));
    double* Ya = (double*)malloc(sizeof(double) * (size_t)(n_pairs * d));
    /* pairs grouped by expert (counting sort, pair order kept) */
    int64_t* cnt = (int64_t*)calloc((size_t)E + 1, sizeof(int64_t));
    int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_pairs > 0 ? n_pairs : 1));
    for (int64_t p = 0; p < n_pairs; ++p) cnt[ids[(int64_t)tokens[p / k] * k + p % k] + 1]++;
    for (int e = 0; e < E; ++e) cnt[e + 1] += cnt[e];
    {
        int64_t* fill = (int64_t*)malloc(sizeof(int64_t) * (size_t)E);
        for (int e = 0; e < E; ++e) fill[e] = cnt[e];
        for (int64_t p = 0; p < n_pairs; ++p) order[fill[ids[(int64_t)tokens[p / k] * k + p % k]]++] = p;
        free(fill);
    }
#pragma omp parallel
    {
        float* Wg = (float*)malloc(sizeof(float) * (size_t)(F * d));
        float* Wu = (float*)malloc(sizeof(float) * (size_t)(F * d));
        float* Wd = (float*)malloc(sizeof(float) * (size_t)(d * F));
        float* xrow = (float*)malloc(sizeof(float) * (size_t)d);
        double* xa = (double*)malloc(sizeof(double) * (size_t)d);
        double* sg = (double*)malloc(sizeof(double) * (size_t)F);
        double* su = (double*)malloc(sizeof(double) * (size_t)F);
        double* ag = (double*)malloc(sizeof(double) * (size_t)F);
        double* au = (double*)malloc(sizeof(double) * (size_t)F);
        float* h = (float*)malloc(sizeof(float) * (size_t)F);
        double* ha = (double*)malloc(sizeof(double) * (size_t)F);
        double* y = (double*)malloc(sizeof(double) * (size_t)d);
        double* ya = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int e = 0; e < E; ++e) {
            if (cnt[e + 1] == cnt[e]) continue;
            dequant_f32(gq + (int64_t)e * F * (d / 2), gs + (int64_t)e * F * (d / 16), F, d, Wg);
            dequant_f32(uq + (int64_t)e * F * (d / 2), us + (int64_t)e * F * (d / 16), F, d, Wu);
            dequant_f32(dq + (int64_t)e * d * (F / 2), ds + (int64_t)e * d * (F / 16), d, F, Wd);
            for (int64_t q = cnt[e]; q < cnt[e + 1]; ++q) {
                const int64_t pair = order[q];
                const int64_t i = pair / k;
                const int64_t t = tokens[i];
                for (int64_t n = 0; n < d; ++n) xrow[n] = bf16_bits_to_float(x[t * d + n]);
                double xscale = 1.0;
                if (mode == 1) {
                    quant_dequant(xrow, d, is13[e], xa, ex && ex->xq ? ex->xq + pair * (d / 2) : NULL,
                                  ex && ex->xs ? ex->xs + pair * (d / 16) : NULL);
                    xscale = (double)is13[e];
                } else {
                    for (int64_t n = 0; n < d; ++n) xa[n] = (double)xrow[n];
                }
                matvec(xa, Wg, F, d, sg, ag);
                matvec(xa, Wu, F, d, su, au);
                for (int64_t f = 0; f < F; ++f) {
                    const double gp = sg[f] * xscale * (double)g_ws2[e];
                    const double up = su[f] * xscale * (double)u_ws2[e];
                    const double G = orc_round_bf16(gp);
                    const double U = orc_round_bf16(up);
                    h[f] = (float)orc_round_bf16(silu(G) * U);
                    if (ex) {
                        const int64_t o = pair * F + f;
                        if (ex->g_pre) ex->g_pre[o] = gp;
                        if (ex->u_pre) ex->u_pre[o] = up;
                        if (ex->g_abs) ex->g_abs[o] = ag[f] * xscale * (double)g_ws2[e];
                        if (ex->u_abs) ex->u_abs[o] = au[f] * xscale * (double)u_ws2[e];
                        if (ex->h) ex->h[o] = h[f];
                    }
                }
                double hscale = 1.0;
                if (mode == 1) {
                    quant_dequant(h, F, is2[e], ha, ex && ex->hq ? ex->hq + pair * (F / 2) : NULL,
                                  ex && ex->hs ? ex->hs + pair * (F / 16) : NULL);
                    hscale = (double)is2[e];
                } else {
                    for (int64_t f = 0; f < F; ++f) ha[f] = (double)h[f];
                }
                matvec(ha, Wd, d, F, y, ya);
                for (int64_t n = 0; n < d; ++n) {
                    const double yv = y[n] * hscale * (double)d_ws2[e];
                    Y[pair * d + n] = round_y ? orc_round_bf16(yv) : yv;
                    Ya[pair * d + n] = ya[n] * hscale * (double)d_ws2[e];
                    if (ex && ex->y_pre) ex->y_pre[pair * d + n] = yv;
                    if (ex && ex->y_abs) ex->y_abs[pair * d + n] = Ya[pair * d + n];
                }
            }
        }
        free(Wg); free(Wu); free(Wd); free(xrow); free(xa); free(sg); free(su); free(ag); free(au);
        free(h); free(ha); free(y); free(ya);
    }
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t t = tokens[i];
        for (int64_t n = 0; n < d; ++n) {
            double acc = 0.0, aabs = 0.0;
            for (int j = 0; j < k; ++j) {
                acc += (double)w[t * k + j] * Y[(i * k + j) * d + n];
                aabs += fabs((double)w[t * k + j]) * Ya[(i * k + j) * d + n];
            }
            out[i * d + n] = (float)orc_round_bf16(acc);
            if (ex && ex->out_pre) ex->out_pre[i * d + n] = acc;
            if (ex && ex->out_abs) ex->out_abs[i * d + n] = aabs;
        }
    }
    free(order);
    free(cnt);
    free(Y);
    free(Ya);
}

/* The layer's plain form: out only, plus h [n_tokens, k, F] if h_out is
 * not NULL. */
void orc_moe_layer(int mode, const uint16_t* x, int64_t T, int64_t d, int64_t F, int E, int k,
                   const int32_t* ids, const float* w,
                   const uint8_t* gq, const uint8_t* gs, const float* g_ws2,
                   const uint8_t* uq, const uint8_t* us, const float* u_ws2,
                   const uint8_t* dq, const uint8_t* ds, const float* d_ws2,
                   const float* is13, const float* is2,
                   const int32_t* tokens, int64_t n_tokens, float* out, float* h_out) {
    orc_layer_extras ex;
    memset(&ex, 0, sizeof ex);
    ex.h = h_out;
    orc_moe_layer_ex(mode, x, T, d, F, E, k, ids, w, gq, gs, g_ws2, uq, us, u_ws2, dq, ds, d_ws2, is13, is2, 0,
                     tokens, n_tokens, out, &ex);
}

/*
 * BF16 shared-expert MLP after the weighted combine (the pages name the
 * shared expert as BF16 next to the NVFP4 routed experts; the math is the
 * plainest reading, with the routed layer's rounding points):
 *   G = bf16(sum x*wg)   U = bf16(sum x*wu)   h = bf16(silu(G) * U)
 *   out = bf16(routed + sum h*wd)
 * x [T, d], wg, wu [Fs, d], wd [d, Fs], routed/out [T, d] (bf16 bits);
 * fp64 sums in k order.  Optional outputs (NULL to skip): out_pre [T, d]
 * (routed + y before the final rounding), out_abs [T, d] (|routed| +
 * sum |h wd|), g_pre / u_pre / g_abs / u_abs [T, Fs] (the gate / up sums
 * before rounding and their sums of |terms|), h_out [T, Fs].
 */
void orc_shared_expert_ex(const uint16_t* x, int64_t T, int64_t d, const uint16_t* wg, const uint16_t* wu,
                          const uint16_t* wd, int64_t Fs, const uint16_t* routed, float* out, double* out_pre,
                          double* out_abs, double* g_pre, double* u_pre, double* g_abs, double* u_abs,
                          float* h_out) {
#pragma omp parallel
    {
        double* h = (double*)malloc(sizeof(double) * (size_t)Fs);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t f = 0; f < Fs; ++f) {
                double g = 0.0, u = 0.0, ga = 0.0, ua = 0.0;
                for (int64_t k = 0; k < d; ++k) {
                    const double xv = bf16_bits_to_float(x[t * d + k]);
                    const double pg = xv * bf16_bits_to_float(wg[f * d + k]);
                    const double pu = xv * bf16_bits_to_float(wu[f * d + k]);
                    g += pg;
                    u += pu;
                    ga += fabs(pg);
                    ua += fabs(pu);
                }
                const double G = orc_round_bf16(g), U = orc_round_bf16(u);
                h[f] = orc_round_bf16(silu(G) * U);
                if (g_pre) g_pre[t * Fs + f] = g;
                if (u_pre) u_pre[t * Fs + f] = u;
                if (g_abs) g_abs[t * Fs + f] = ga;
                if (u_abs) u_abs[t * Fs + f] = ua;
                if (h_out) h_out[t * Fs + f] = (float)h[f];
            }
            for (int64_t n = 0; n < d; ++n) {
                double y = 0.0, ya = 0.0;
                for (int64_t f = 0; f < Fs; ++f) {
                    const double p = h[f] * bf16_bits_to_float(wd[n * Fs + f]);
                    y += p;
                    ya += fabs(p);
                }
                const double r = (double)bf16_bits_to_float(routed[t * d + n]);
                out[t * d + n] = (float)orc_round_bf16(r + y);
                if (out_pre) out_pre[t * d + n] = r + y;
                if (out_abs) out_abs[t * d + n] = fabs(r) + ya;
            }
        }
        free(h);
    }
}

/* The shared expert's plain form (out only). */
void orc_shared_expert(const uint16_t* x, int64_t T, int64_t d, const uint16_t* wg, const uint16_t* wu,
                       const uint16_t* wd, int64_t Fs, const uint16_t* routed, float* out) {
    orc_shared_expert_ex(x, T, d, wg, wu, wd, Fs, routed, out, NULL, NULL, NULL, NULL, NULL, NULL, NULL);
}

/*
 * Dense NVFP4 linear over the bf16 rows x [M, K] (the dense MLP runs on it,
 * gate and up apart because their tensor scales differ).
 * Without w_up:  out = bf16(ws2 * sum x*w)                     [M, N]
 * With w_up:     out = bf16(silu(bf16(ws2*sum x*w)) * bf16(ws2u*sum x*wu))
 * Optional outputs (NULL to skip), all [M, N] fp64: pre = the value before
 * the final bf16 rounding; g_pre / u_pre = the gate / up values before
 * their rounding, g_abs / u_abs their sums of |terms| times the tensor
 * scale (without w_up only g_pre / g_abs are written, g_pre = pre).
 */
void orc_linear_ex(const uint16_t* x, int64_t M, int64_t K,
                   const uint8_t* wq, const uint8_t* ws, float ws2, int64_t N,
                   const uint8_t* uq, const uint8_t* us, float us2, float* out,
                   double* pre, double* g_pre, double* u_pre, double* g_abs, double* u_abs) {
    float* Wg = (float*)malloc(sizeof(float) * (size_t)(N * K));
    float* Wu = uq ? (float*)malloc(sizeof(float) * (size_t)(N * K)) : NULL;
    dequant_f32(wq, ws, N, K, Wg);
    if (uq) dequant_f32(uq, us, N, K, Wu);
#pragma omp parallel
    {
        double* xa = (double*)malloc(sizeof(double) * (size_t)K);
        double* sg = (double*)malloc(sizeof(double) * (size_t)N);
        double* su = (double*)malloc(sizeof(double) * (size_t)N);
        double* ag = (double*)malloc(sizeof(double) * (size_t)N);
        double* au = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 1)
        for (int64_t m = 0; m < M; ++m) {
            for (int64_t kk = 0; kk < K; ++kk) xa[kk] = (double)bf16_bits_to_float(x[m * K + kk]);
            matvec(xa, Wg, N, K, sg, ag);
            if (uq) {
                matvec(xa, Wu, N, K, su, au);
                for (int64_t n = 0; n < N; ++n) {
                    const double gp = sg[n] * (double)ws2, up = su[n] * (double)us2;
                    double G = orc_round_bf16(gp);
                    double U = orc_round_bf16(up);
                    const double hp = silu(G) * U;
                    out[m * N + n] = (float)orc_round_bf16(hp);
                    if (pre) pre[m * N + n] = hp;
                    if (g_pre) g_pre[m * N + n] = gp;
                    if (u_pre) u_pre[m * N + n] = up;
                    if (g_abs) g_abs[m * N + n] = ag[n] * (double)ws2;
                    if (u_abs) u_abs[m * N + n] = au[n] * (double)us2;
                }
            } else {
                for (int64_t n = 0; n < N; ++n) {
                    const double gp = sg[n] * (double)ws2;
                    out[m * N + n] = (float)orc_round_bf16(gp);
                    if (pre) pre[m * N + n] = gp;
                    if (g_pre) g_pre[m * N + n] = gp;
                    if (g_abs) g_abs[m * N + n] = ag[n] * (double)ws2;
                }
            }
        }
        free(xa); free(sg); free(su); free(ag); free(au);
    }
    free(Wg);
    free(Wu);
}

void orc_linear(const uint16_t* x, int64_t M, int64_t K,
                const uint8_t* wq, const uint8_t* ws, float ws2, int64_t N,
                const uint8_t* uq, const uint8_t* us, float us2, float* out) {
    orc_linear_ex(x, M, K, wq, ws, ws2, N, uq, us, us2, out, NULL, NULL, NULL, NULL, NULL);
}

int orc_num_threads(void) {
#ifdef _OPENMP
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
#else
    return 1;
#endif
}
