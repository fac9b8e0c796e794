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
 *   Y = ws2_d * sum h*w_d   (unrounded)
 *   out[t] = bf16(sum_j w_j * Y_j)                                   (R4)
 * All sums here are fp64.  Scale arithmetic that decides a code (block
 * scale, element / scale) is done in fp32 in the order the recipe states,
 * because that is the precision in which the codes are defined.
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
/* Then a stable counting sort of the T*k (token, slot) pairs by expert  */
/* (order: expert, then token, then slot):                               */
/*   offsets[e] = number of pairs routed to experts < e;                 */
/*   row_to_slot[row] = t*k + slot;  slot_to_row[t*k + slot] = row.      */
/* ------------------------------------------------------------------ */
void orc_route(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w,
               int32_t* offsets, int32_t* row_to_slot, int32_t* slot_to_row) {
    char* chosen = (char*)malloc((size_t)E);
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        memset(chosen, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (chosen[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;
            }
            chosen[best] = 1;
            ids[t * k + j] = best;
        }
        double lmax = (double)l[ids[t * k]];
        double den = 0.0;
        for (int j = 0; j < k; ++j) den += exp((double)l[ids[t * k + j]] - lmax);
        for (int j = 0; j < k; ++j)
            w[t * k + j] = (float)(exp((double)l[ids[t * k + j]] - lmax) / den);
    }
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

/* One NVFP4 linear over one input vector a[K] (already dequantised, fp64):
 * out[n] = sum_k a[k] * dec(q[n,k]) * dec(s[n,k/16]) for n < N. */
static void nvfp4_matvec(const double* a, const uint8_t* codes, const uint8_t* scales,
                         int64_t N, int64_t K, double* out) {
    for (int64_t n = 0; n < N; ++n) {
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += a[k] * deq(codes, scales, K, n, k);
        out[n] = s;
    }
}

/* Quantise a float vector with tensor scale gs and return it dequantised
 * (dec(q) * dec(s), no tensor scale) in fp64. */
static void quant_dequant(const float* v, int64_t K, float gs, double* out) {
    uint8_t* c = (uint8_t*)malloc((size_t)(K / 2));
    uint8_t* s = (uint8_t*)malloc((size_t)(K / 16));
    quantize_row(v, K, gs, c, s);
    for (int64_t k = 0; k < K; ++k) out[k] = deq(c, s, K, 0, k);
    free(c);
    free(s);
}

/*
 * Routed-expert MoE layer for the tokens listed in `tokens` (n_tokens of
 * them), given routing ids/w [T, k].  mode 0 = W4A16 (bf16 activations),
 * mode 1 = W4A4 (activations quantised to NVFP4 with the static per-expert
 * input_scale: is13[e] before gate/up, is2[e] before down).
 * Weight banks are stacked over experts: gate/up codes [E, F, d/2], scales
 * [E, F, d/16], ws2 [E]; down codes [E, d, F/2], scales [E, d, F/16].
 * out[i, :] receives bf16(sum_j w_j * Y_j) for token tokens[i] (as float).
 * h_out, if not NULL, receives h [n_tokens, k, F] (the bf16 values).
 */
void orc_moe_layer(int mode, const uint16_t* x, int64_t T, int64_t d, int64_t F, int E, int k,
                   const int32_t* ids, const float* w,
                   const uint8_t* gq, const uint8_t* gs, const float* g_ws2,
                   const uint8_t* uq, const uint8_t* us, const float* u_ws2,
                   const uint8_t* dq, const uint8_t* ds, const float* d_ws2,
                   const float* is13, const float* is2,
                   const int32_t* tokens, int64_t n_tokens, float* out, float* h_out) {
    (void)T;
    (void)E;
    /* Y_j of every (token, slot) pair, then the weighted sum over the slots
     * in slot order.  Pairs are independent, so they are spread over the
     * threads; the sum itself is sequential. */
    double* Y = (double*)malloc(sizeof(double) * (size_t)(n_tokens * k * d));
#pragma omp parallel
    {
        float* xrow = (float*)malloc(sizeof(float) * (size_t)d);
        double* xa = (double*)malloc(sizeof(double) * (size_t)d);
        double* sg = (double*)malloc(sizeof(double) * (size_t)F);
        double* su = (double*)malloc(sizeof(double) * (size_t)F);
        float* h = (float*)malloc(sizeof(float) * (size_t)F);
        double* ha = (double*)malloc(sizeof(double) * (size_t)F);
        double* y = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t pair = 0; pair < n_tokens * k; ++pair) {
            int64_t i = pair / k;
            int j = (int)(pair % k);
            int64_t t = tokens[i];
            int e = ids[t * k + j];
            for (int64_t n = 0; n < d; ++n) xrow[n] = bf16_bits_to_float(x[t * d + n]);
            double xscale = 1.0;
            if (mode == 1) {
                quant_dequant(xrow, d, is13[e], xa);
                xscale = (double)is13[e];
            } else {
                for (int64_t n = 0; n < d; ++n) xa[n] = (double)xrow[n];
            }
            nvfp4_matvec(xa, gq + (int64_t)e * F * (d / 2), gs + (int64_t)e * F * (d / 16), F, d, sg);
            nvfp4_matvec(xa, uq + (int64_t)e * F * (d / 2), us + (int64_t)e * F * (d / 16), F, d, su);
            for (int64_t f = 0; f < F; ++f) {
                double G = orc_round_bf16(sg[f] * xscale * (double)g_ws2[e]);
                double U = orc_round_bf16(su[f] * xscale * (double)u_ws2[e]);
                h[f] = (float)orc_round_bf16(silu(G) * U);
            }
            if (h_out)
                for (int64_t f = 0; f < F; ++f) h_out[(i * k + j) * F + f] = h[f];
            double hscale = 1.0;
            if (mode == 1) {
                quant_dequant(h, F, is2[e], ha);
                hscale = (double)is2[e];
            } else {
                for (int64_t f = 0; f < F; ++f) ha[f] = (double)h[f];
            }
            nvfp4_matvec(ha, dq + (int64_t)e * d * (F / 2), ds + (int64_t)e * d * (F / 16), d, F, y);
            for (int64_t n = 0; n < d; ++n) Y[pair * d + n] = y[n] * hscale * (double)d_ws2[e];
        }
        free(xrow); free(xa); free(sg); free(su); free(h); free(ha); free(y);
    }
    for (int64_t i = 0; i < n_tokens; ++i) {
        int64_t t = tokens[i];
        for (int64_t n = 0; n < d; ++n) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j) acc += (double)w[t * k + j] * Y[(i * k + j) * d + n];
            out[i * d + n] = (float)orc_round_bf16(acc);
        }
    }
    free(Y);
}

/*
 * BF16 shared-expert MLP after the weighted combine (the pages name the
 * shared expert as BF16 next to the NVFP4 routed experts; the math is the
 * plainest reading, with the routed layer's rounding points):
 *   G = bf16(sum x*wg)   U = bf16(sum x*wu)   h = bf16(silu(G) * U)
 *   out = bf16(routed + sum h*wd)
 * x [T, d], wg, wu [Fs, d], wd [d, Fs], routed/out [T, d] (bf16 bits);
 * fp64 sums in k order.
 */
void orc_shared_expert(const uint16_t* x, int64_t T, int64_t d, const uint16_t* wg, const uint16_t* wu,
                       const uint16_t* wd, int64_t Fs, const uint16_t* routed, float* out) {
#pragma omp parallel
    {
        double* h = (double*)malloc(sizeof(double) * (size_t)Fs);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t f = 0; f < Fs; ++f) {
                double g = 0.0, u = 0.0;
                for (int64_t k = 0; k < d; ++k) {
                    const double xv = bf16_bits_to_float(x[t * d + k]);
                    g += xv * bf16_bits_to_float(wg[f * d + k]);
                    u += xv * bf16_bits_to_float(wu[f * d + k]);
                }
                const double G = orc_round_bf16(g), U = orc_round_bf16(u);
                h[f] = orc_round_bf16(silu(G) * U);
            }
            for (int64_t n = 0; n < d; ++n) {
                double y = 0.0;
                for (int64_t f = 0; f < Fs; ++f) y += h[f] * bf16_bits_to_float(wd[n * Fs + f]);
                out[t * d + n] = (float)orc_round_bf16((double)bf16_bits_to_float(routed[t * d + n]) + y);
            }
        }
        free(h);
    }
}

/*
 * Dense NVFP4 linear over the bf16 rows x [M, K] (the dense MLP runs on it,
 * gate and up apart because their tensor scales differ).
 * Without w_up:  out = bf16(ws2 * sum x*w)                     [M, N]
 * With w_up:     out = bf16(silu(bf16(ws2*sum x*w)) * bf16(ws2u*sum x*wu))
 */
void orc_linear(const uint16_t* x, int64_t M, int64_t K,
                const uint8_t* wq, const uint8_t* ws, float ws2, int64_t N,
                const uint8_t* uq, const uint8_t* us, float us2, float* out) {
#pragma omp parallel
    {
        double* xa = (double*)malloc(sizeof(double) * (size_t)K);
        double* sg = (double*)malloc(sizeof(double) * (size_t)N);
        double* su = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 1)
        for (int64_t m = 0; m < M; ++m) {
            for (int64_t kk = 0; kk < K; ++kk) xa[kk] = (double)bf16_bits_to_float(x[m * K + kk]);
            nvfp4_matvec(xa, wq, ws, N, K, sg);
            if (uq) {
                nvfp4_matvec(xa, uq, us, N, K, su);
                for (int64_t n = 0; n < N; ++n) {
                    double G = orc_round_bf16(sg[n] * (double)ws2);
                    double U = orc_round_bf16(su[n] * (double)us2);
                    out[m * N + n] = (float)orc_round_bf16(silu(G) * U);
                }
            } else {
                for (int64_t n = 0; n < N; ++n) out[m * N + n] = (float)orc_round_bf16(sg[n] * (double)ws2);
            }
        }
        free(xa); free(sg); free(su);
    }
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
