// moe.cu -- the routed-expert layer (W4A16 and W4A4) and the dense NVFP4
// linear: host validation, workspace layout and the launch sequence.
//
// TensorFold issue #308 "GLM-5.3-Flash on CUDA: read nvidia/GLM-5.3-Flash-NVFP4
// (ModelOpt NVFP4) as stored, W4A16": "What the branch does" (grouped routed
// experts over bf16 rows with weight_scale_2 per expert; dense MLP with gate
// and up apart; FP4 x FP4 as the checkpoint's own math) and "The checkpoint"
// (static input_scale).  Launch sequence of one layer call:
//   route + permutation (also clears the counters)
//   [W4A4: static-scale act-quant of the permuted rows]
//   gate/up + SwiGLU (h per routed row; W4A4: h requantised to NVFP4)
//   down + weighted top-k combine:
//     decode-shaped kernels: w * y per routed row in fp32; the CTA that
//       completes a token's last slot in a group of outputs sums the
//       token's k rows there in slot order and writes them as bf16;
//     prompt-shaped kernels: y written per routed row in bf16, then each
//       token's k rows weighted and summed in slot order.
//   Both are deterministic (the same bits on every run).
#include <climits>
#include <cstring>

#include "common.cuh"
#include "internal.cuh"
#include "gemv.cuh"
#include "decode.cuh"
#include "tc.cuh"

namespace nvfp4 {

namespace {

constexpr int kCounters = 8;
// Decode-shaped gate/up: chunks (256 of K) between a CTA's L2 prefetch of
// its weight tiles and its loads of them (measured on GB300 at T=64: 0 ->
// 538 µs per layer, 2 -> 529 µs, 4 -> 541 µs, 8 -> 633 µs).
constexpr int kGemvPrefetch = 2;

struct MoeWs {
    RouteArrays ra;
    uint16_t* h;      // [R, F]     W4A16
    uint8_t* xq;      // [R, d/2]   W4A4
    uint8_t* xs;      // [R, d/16]  W4A4
    uint8_t* hq;      // [R, F/2]   W4A4
    uint8_t* hs;      // [R, F/16]  W4A4
    float* yrows;     // [R, d]: w * y fp32 rows (decode kernel) or bf16 y rows (prompt paths)
    int* clear;       // zeroed by the route launch (decode-shaped paths): work counters, then
                      // per-tile and per-(token, output group) completion counters
    int* tile_ready;  // [max tiles]
    int* tok_done;    // [T, d / 16]
    // prompt-shaped (tensor-core) path, W4A16
    uint16_t* xp;     // [R, d]  f16 x * 2^-s, rows in expert order
    int32_t* xp_exp;  // [R]
    uint16_t* hh;     // [R, F]  f16 h * 2^-s
    int32_t* h_exp;   // [R]
};

bool tc_possible(int mode, int d, int F) { return mode == 0 && d % 128 == 0 && F % 128 == 0; }

// nvfp4_set_kernel_choice: -1 by shape, 0 decode-shaped, 1 prompt-shaped.
int forced_path() {
    const int c = kernel_choice();
    return c == 0 ? -1 : (c == 2 ? 1 : 0);
}

// Decode-shaped layers: the persistent one-launch kernel or the two GEMV launches.
bool use_fused_decode(int d, int F) {
    if (!decode_supported(d, F)) return false;
    const int c = kernel_choice();
    if (c == 3) return false;
    if (c == 4) return true;
    return false;
}

// Tensor cores once the experts average 32 or more routed rows.
bool use_tc(int mode, int T, int E, int k, int d, int F) {
    if (!tc_possible(mode, d, F)) return false;
    const int f = forced_path();
    if (f >= 0) return f == 1;
    const long long R = (long long)T * k;
    return R >= 32LL * std::min<long long>(E, R);
}

// W4A4 on the block-scaled FP4 tensor cores (K a multiple of 256 on both projections).
bool use_tc_w4a4(int T, int E, int k, int d, int F) {
    if (!tcq_supported(TCM_SWIGLU_Q, F, d) || !tcq_supported(TCM_ROWS, d, F)) return false;
    const int f = forced_path();
    if (f >= 0) return f == 1;
    const long long R = (long long)T * k;
    return R >= 32LL * std::min<long long>(E, R);
}

MoeWs carve_moe(void* base, int T, int E, int k, int d, int F, int mode, size_t* bytes) {
    Carver c(base);
    const size_t R = (size_t)T * k;
    MoeWs w{};
    w.ra.ids = c.take<int32_t>(R + 1);
    w.ra.w = c.take<float>(R + 1);
    w.ra.offsets = c.take<int32_t>(E + 1);
    w.ra.row_to_slot = c.take<int32_t>(R + 1);
    w.ra.slot_to_row = c.take<int32_t>(R + 1);
    w.ra.active = c.take<int32_t>(E);
    w.ra.n_active = c.take<int32_t>(4);
    w.ra.tile_start = c.take<int32_t>(E + 1);
    w.ra.tile_start_tc = c.take<int32_t>(E + 1);
    w.ra.counts = c.take<int32_t>(route_scratch_words(T, E, k) + 1);
    const size_t max_tiles = R / kGemvTokTile + std::min<size_t>(E, R) + 1;
    const size_t n_clear = kCounters + max_tiles + (size_t)T * std::max(decode_groups_d(d), d / 16);
    w.clear = c.take<int>(n_clear);
    w.ra.clear = w.clear;
    w.ra.n_clear = (int)n_clear;
    w.tile_ready = w.clear + kCounters;
    w.tok_done = w.tile_ready + max_tiles;
    w.yrows = c.take<float>(R * d);
    if (mode == 0) {
        w.h = c.take<uint16_t>(R * F);
        if (tc_possible(mode, d, F)) {
            w.xp = c.take<uint16_t>(R * d);
            w.xp_exp = c.take<int32_t>(R + 1);
            w.hh = c.take<uint16_t>(R * F);
            w.h_exp = c.take<int32_t>(R + 1);
        }
    } else {
        w.xq = c.take<uint8_t>(R * (d / 2));
        w.xs = c.take<uint8_t>(R * (d / 16));
        w.hq = c.take<uint8_t>(R * (F / 2));
        w.hs = c.take<uint8_t>(R * (F / 16));
    }
    if (bytes) *bytes = align_up(c.off, 256);
    return w;
}

bool w_ok(const nvfp4_w& w) { return w.codes && w.scales && w.weight_scale_2; }
bool w_aligned(const nvfp4_w& w) {
    return aligned16(w.codes) && aligned16(w.scales) && aligned16(w.weight_scale_2);
}

nvfp4_status check_moe(const uint16_t* x, int T, int top_k, const nvfp4_moe_weights* w, const void* out,
                       const void* ws, size_t ws_bytes, int mode) {
    if (!w) return NVFP4_ERR_INVALID_ARG;
    if (T < 0 || w->E < 1 || w->d < 1 || w->F < 1) return NVFP4_ERR_INVALID_ARG;
    if (w->E > kMaxExperts || top_k < 1 || top_k > kMaxTopK || top_k > w->E) return NVFP4_ERR_SHAPE;
    if (w->d % 64 != 0 || w->F % 64 != 0 || !gemv_supported_k(w->d) || !gemv_supported_k(w->F))
        return NVFP4_ERR_SHAPE;
    if ((size_t)T * top_k > (size_t)INT_MAX / 2) return NVFP4_ERR_SHAPE;
    if (T == 0) return NVFP4_OK;
    if (!x || !out || !ws || !w_ok(w->gate) || !w_ok(w->up) || !w_ok(w->down)) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || !aligned16(ws) || !w_aligned(w->gate) || !w_aligned(w->up) ||
        !w_aligned(w->down))
        return NVFP4_ERR_ALIGN;
    if (ws_bytes < nvfp4_moe_workspace_size(T, w->E, top_k, w->d, w->F, mode)) return NVFP4_ERR_WORKSPACE;
    return NVFP4_OK;
}

GemvArgs base_args(const MoeWs& ws, int top_k, int E) {
    GemvArgs a{};
    a.top_k = top_k;
    a.E = E;
    a.offsets = ws.ra.offsets;
    a.active = ws.ra.active;
    a.n_active = ws.ra.n_active;
    a.tile_start = ws.ra.tile_start;
    a.row_to_slot = ws.ra.row_to_slot;
    a.topk_w = ws.ra.w;
    return a;
}

int gemv_max_work(int R, int E, int N) {
    long long tiles = (long long)(R + kGemvTokTile - 1) / kGemvTokTile + std::min(E, R);
    long long w = tiles * (N / 16);
    return (int)std::min<long long>(w, INT_MAX / 2);
}

int expected_tiles(int R, int E) { return std::max(std::min(E, R), R / kGemvTokTile); }

nvfp4_status run_moe(int mode, const uint16_t* x, int T, const float* logits, int top_k,
                     const nvfp4_moe_weights* w, const float* is13, const float* is2, uint16_t* out, void* wsp,
                     size_t ws_bytes, int32_t* d_status, cudaStream_t s) {
    nvfp4_status st = check_moe(x, T, top_k, w, out, wsp, ws_bytes, mode);
    if (st != NVFP4_OK || T == 0) return st;
    if (mode == 1) {
        if (!is13 || !is2) return NVFP4_ERR_INVALID_ARG;
        if (!aligned16(is13) || !aligned16(is2)) return NVFP4_ERR_ALIGN;
    }
    if (d_status && !aligned16(d_status)) return NVFP4_ERR_ALIGN;
    const int E = w->E, d = w->d, F = w->F, R = T * top_k;
    MoeWs ws = carve_moe(wsp, T, E, top_k, d, F, mode, nullptr);
    const bool prompt = mode == 1 ? use_tc_w4a4(T, E, top_k, d, F) : use_tc(mode, T, E, top_k, d, F);
    const bool fused = !prompt && use_fused_decode(d, F);
    const int tiles = expected_tiles(R, E);
    // the decode-shaped down launch: K split and feature blocks per item
    const int ks_d = gemv_pick_ksplit(tiles, d, 1);
    const int grp_d = gemv_pick_group(tiles, d, ks_d, 1);
    {   // counters the chosen path uses (the prompt-shaped kernels use none)
        const size_t max_tiles = (size_t)R / kGemvTokTile + std::min(E, R) + 1;
        const int groups = fused ? decode_groups_d(d) : gemv_item_groups(d, ks_d, grp_d);
        ws.ra.n_clear = prompt ? 0 : (int)(kCounters + max_tiles + (size_t)T * groups);
    }

    launch_route(logits, T, E, top_k, ws.ra, d_status, s);
    if (mode == 1)
        launch_quantize_act(x, R, d, ws.ra.row_to_slot, top_k, is13, ws.ra.offsets, E, ws.xq, ws.xs, s);

    if (mode == 1 && prompt) {
        const int max_tiles = R / kTcTokTile + std::min(E, R) + 1;
        // gate/up + SwiGLU, h requantised under the down projection's input scale
        TcmArgs g{};
        g.K = d;
        g.N = F;
        g.top_k = top_k;
        g.offsets = ws.ra.offsets;
        g.active = ws.ra.active;
        g.n_active = ws.ra.n_active;
        g.tile_start = ws.ra.tile_start_tc;
        g.a_codes[0] = w->gate.codes;  g.a_scales[0] = w->gate.scales;  g.a_ws2[0] = w->gate.weight_scale_2;
        g.a_codes[1] = w->up.codes;    g.a_scales[1] = w->up.scales;    g.a_ws2[1] = w->up.weight_scale_2;
        g.x_gs = is13;
        g.hq_out = ws.hq;
        g.hs_out = ws.hs;
        g.hq_gs = is2;
        g.status = d_status;
        if (!tcq_set_maps(&g, ws.xq, ws.xs, R, (long long)E * F)) return NVFP4_ERR_CUDA;
        launch_tcq(TCM_SWIGLU_Q, g, max_tiles, s);
        // down: w * y rows by routed row, then each token's slots summed in slot order
        TcmArgs u = g;
        u.K = F;
        u.N = d;
        u.a_codes[0] = w->down.codes;  u.a_scales[0] = w->down.scales;  u.a_ws2[0] = w->down.weight_scale_2;
        u.a_codes[1] = u.a_codes[0];   u.a_scales[1] = u.a_scales[0];   u.a_ws2[1] = u.a_ws2[0];
        u.x_gs = is2;
        u.hq_out = nullptr;
        u.hs_out = nullptr;
        u.row_to_slot = ws.ra.row_to_slot;
        u.topk_w = ws.ra.w;
        u.y_rows = reinterpret_cast<uint16_t*>(ws.yrows);
        if (!tcq_set_maps(&u, ws.hq, ws.hs, R, (long long)E * d)) return NVFP4_ERR_CUDA;
        launch_tcq(TCM_ROWS, u, max_tiles, s);
        launch_sum_rows(u.y_rows, ws.ra.slot_to_row, ws.ra.w, T, top_k, d, out, s);
        return last_launch_status();
    }

    if (prompt) {
        // the down projection writes w * y rows (summed per token in slot order
        // afterwards) when the prompt-shaped kernel takes its shape (K = F a
        // multiple of 256), else the weights-as-M kernel adds into a zeroed
        // fp32 accumulator
        const bool rows = tcm_supported(TCM_ROWS, d, F);
        // x -> f16 rows in expert order (and zero the combine accumulator)
        launch_rows_to_f16(x, R, d, ws.xp, ws.xp_exp, nullptr, d, s, ws.ra.row_to_slot, top_k, T);
        const int max_tiles = R / kTcTokTile + std::min(E, R) + 1;
        // gate/up + SwiGLU -> h (bf16)
        TcmArgs g{};
        g.K = d;
        g.N = F;
        g.top_k = top_k;
        g.offsets = ws.ra.offsets;
        g.active = ws.ra.active;
        g.n_active = ws.ra.n_active;
        g.tile_start = ws.ra.tile_start_tc;
        g.a_codes[0] = w->gate.codes;  g.a_scales[0] = w->gate.scales;  g.a_ws2[0] = w->gate.weight_scale_2;
        g.a_codes[1] = w->up.codes;    g.a_scales[1] = w->up.scales;    g.a_ws2[1] = w->up.weight_scale_2;
        g.x_exp = ws.xp_exp;
        g.h_out = ws.h;
        g.status = d_status;
        if (tcm_supported(TCM_SWIGLU, F, d)) {
            if (!make_tmap_rows_f16(&g.tmap_x, ws.xp, R, d) || !tcm_set_weights(&g, (long long)E * F))
                return NVFP4_ERR_CUDA;
            launch_tcm(TCM_SWIGLU, g, max_tiles * (F / 128), s);
        } else {
            TcArgs t{};
            t.top_k = top_k;
            t.offsets = ws.ra.offsets;
            t.active = ws.ra.active;
            t.n_active = ws.ra.n_active;
            t.tile_start = ws.ra.tile_start_tc;
            t.row_to_slot = nullptr;
            t.status = d_status;
            t.K = d;
            t.N = F;
            for (int p = 0; p < 2; ++p) {
                t.a_codes[p] = g.a_codes[p];  t.a_scales[p] = g.a_scales[p];  t.a_ws2[p] = g.a_ws2[p];
            }
            t.b_f16 = ws.xp;
            t.b_exp = ws.xp_exp;
            t.b_by_token = 0;
            t.h_out = ws.h;
            launch_tc_gemm(TC_OUT_H, 2, t, max_tiles * (F / 128), s);
        }
        // h -> f16 rows
        launch_rows_to_f16(ws.h, R, F, ws.hh, ws.h_exp, nullptr, 0, s);
        // down + weighted combine
        if (rows) {
            TcmArgs u = g;
            u.K = F;
            u.N = d;
            u.a_codes[0] = w->down.codes;  u.a_scales[0] = w->down.scales;  u.a_ws2[0] = w->down.weight_scale_2;
            u.a_codes[1] = u.a_codes[0];   u.a_scales[1] = u.a_scales[0];   u.a_ws2[1] = u.a_ws2[0];
            u.x_exp = ws.h_exp;
            u.h_out = nullptr;
            u.y_rows = reinterpret_cast<uint16_t*>(ws.yrows);
            if (!make_tmap_rows_f16(&u.tmap_x, ws.hh, R, F) || !tcm_set_weights(&u, (long long)E * d))
                return NVFP4_ERR_CUDA;
            launch_tcm(TCM_ROWS, u, max_tiles * (d / 256), s);
            launch_sum_rows(u.y_rows, ws.ra.slot_to_row, ws.ra.w, T, top_k, d, out, s);
            return last_launch_status();
        } else {
            TcArgs u{};
            u.top_k = top_k;
            u.offsets = ws.ra.offsets;
            u.active = ws.ra.active;
            u.n_active = ws.ra.n_active;
            u.tile_start = ws.ra.tile_start_tc;
            u.row_to_slot = ws.ra.row_to_slot;
            u.status = d_status;
            u.K = F;
            u.N = d;
            u.a_codes[0] = w->down.codes;  u.a_scales[0] = w->down.scales;  u.a_ws2[0] = w->down.weight_scale_2;
            u.a_codes[1] = u.a_codes[0];   u.a_scales[1] = u.a_scales[0];   u.a_ws2[1] = u.a_ws2[0];
            u.b_f16 = ws.hh;
            u.b_exp = ws.h_exp;
            u.b_by_token = 0;
            // y in bf16 by routed row, then each token's rows in slot order
            u.y_out = reinterpret_cast<uint16_t*>(ws.yrows);
            launch_tc_gemm(TC_OUT_BF16, 1, u, max_tiles * (d / 128), s, true);
            launch_sum_rows(u.y_out, ws.ra.slot_to_row, ws.ra.w, T, top_k, d, out, s);
        }
        return last_launch_status();
    }

    if (fused) {
        // one persistent launch: gate/up + SwiGLU, then down + the slot-ordered combine
        DecodeArgs da{};
        da.d = d;
        da.F = F;
        da.top_k = top_k;
        decode_pick_work(tiles, &da);
        if (!decode_set_maps(&da, w)) return NVFP4_ERR_CUDA;
        da.offsets = ws.ra.offsets;
        da.active = ws.ra.active;
        da.n_active = ws.ra.n_active;
        da.tile_start = ws.ra.tile_start;
        da.row_to_slot = ws.ra.row_to_slot;
        da.slot_to_row = ws.ra.slot_to_row;
        da.topk_w = ws.ra.w;
        da.gate_ws2 = w->gate.weight_scale_2;
        da.up_ws2 = w->up.weight_scale_2;
        da.down_ws2 = w->down.weight_scale_2;
        da.x = x;
        da.xq = ws.xq;
        da.xs = ws.xs;
        da.is13 = is13;
        da.is2 = is2;
        da.h = ws.h;
        da.hq = ws.hq;
        da.hs = ws.hs;
        da.yrows = ws.yrows;
        da.out = out;
        da.counters = ws.clear + 2;
        da.tile_ready = ws.tile_ready;
        da.tok_done = ws.tok_done;
        da.status = d_status;
        launch_decode(mode == 0 ? B_BF16 : B_NVFP4, da, s);
        return last_launch_status();
    }
    GemvArgs a = base_args(ws, top_k, E);
    // gate/up + SwiGLU (also zeroes the fp32 combine accumulator)
    a.K = d;
    a.N = F;
    a.nproj = 2;
    a.ksplit = gemv_pick_ksplit(tiles, F, 2);
    a.fb_group = gemv_pick_group(tiles, F, a.ksplit, 2);
    a.a_codes[0] = w->gate.codes;  a.a_scales[0] = w->gate.scales;  a.a_ws2[0] = w->gate.weight_scale_2;
    a.a_codes[1] = w->up.codes;    a.a_scales[1] = w->up.scales;    a.a_ws2[1] = w->up.weight_scale_2;
    a.work_counter = ws.clear + 0;
    if (d % 256 == 0 && a.ksplit == 1) {
        // L2 prefetch of the CTA's feature rows (16 x 8 / ksplit of them),
        // kGemvPrefetch of each warp's chunks ahead (measured slower when K
        // is split over warps: the few-token shapes)
        const unsigned long long rows = (unsigned long long)E * F;
        const unsigned fb_rows = 16u * (8u / (unsigned)a.ksplit);
        bool ok = true;
        for (int p = 0; p < 2 && ok; ++p)
            ok = encode_tmap_u8(&a.pf_codes[p], a.a_codes[p], d / 2, rows, 128, fb_rows, false) &&
                 encode_tmap_u8(&a.pf_scales[p], a.a_scales[p], d / 16, rows, 16, fb_rows, false);
        a.pf_dist = ok ? kGemvPrefetch : 0;
    }
    if (mode == 0) {
        a.b_bf16 = x;
        a.b_by_token = 1;
        a.h_out = ws.h;
        launch_gemv(B_BF16, OUT_H, a, gemv_max_work(R, E, F), s);
    } else {
        a.b_codes = ws.xq;
        a.b_scales = ws.xs;
        a.b_gs = is13;
        a.hq_out = ws.hq;
        a.hs_out = ws.hs;
        a.hq_gs = is2;
        launch_gemv(B_NVFP4, OUT_HQ, a, gemv_max_work(R, E, F), s);
    }
    // down + weighted combine; the last contribution to a token writes its bf16 row
    GemvArgs b = base_args(ws, top_k, E);
    b.K = F;
    b.N = d;
    b.nproj = 1;
    b.ksplit = ks_d;
    b.fb_group = grp_d;
    b.a_codes[0] = w->down.codes;  b.a_scales[0] = w->down.scales;  b.a_ws2[0] = w->down.weight_scale_2;
    b.a_codes[1] = w->down.codes;  b.a_scales[1] = w->down.scales;  b.a_ws2[1] = w->down.weight_scale_2;
    b.work_counter = ws.clear + 1;
    // (no L2 prefetch here: measured slower on the down projection, whose
    // shared-memory ring already keeps three batches in flight)
    b.y_rows = ws.yrows;
    b.slot_to_row = ws.ra.slot_to_row;
    b.tok_done = ws.tok_done;
    b.out_bf16 = out;
    if (mode == 0) {
        b.b_bf16 = ws.h;
        b.b_by_token = 0;
        launch_gemv(B_BF16, OUT_COMBINE, b, gemv_max_work(R, E, d), s);
    } else {
        b.b_codes = ws.hq;
        b.b_scales = ws.hs;
        b.b_gs = is2;
        launch_gemv(B_NVFP4, OUT_COMBINE, b, gemv_max_work(R, E, d), s);
    }
    return last_launch_status();
}

// ---- dense linear ----
struct LinWs {
    int32_t* meta;     // offsets[2], active[1], n_active[1], tile_start[2], tile_start_tc[2]
    int* counters;
    uint16_t* xh;      // [M, K] (tensor-core path)
    int32_t* x_exp;    // [M]
};

bool lin_tc_possible(int N) { return N % 128 == 0; }

bool use_tc_linear(int M, int N) {
    if (!lin_tc_possible(N)) return false;
    const int f = forced_path();
    if (f >= 0) return f == 1;
    return M >= 128;
}

LinWs carve_lin(void* base, int M, int K, int N, size_t* bytes) {
    Carver c(base);
    LinWs l{};
    l.meta = c.take<int32_t>(8);
    l.counters = c.take<int>(kCounters);
    if (lin_tc_possible(N)) {
        l.xh = c.take<uint16_t>((size_t)M * K);
        l.x_exp = c.take<int32_t>(M + 1);
    }
    if (bytes) *bytes = align_up(c.off, 256);
    return l;
}

__global__ void linear_prep_kernel(int M, int32_t* meta, int* counters) {
    grid_dep_wait();
    if (threadIdx.x == 0) {
        meta[0] = 0;                                      // offsets[0]
        meta[1] = M;                                      // offsets[1]
        meta[2] = 0;                                      // active[0] = expert 0
        meta[3] = 1;                                      // n_active
        meta[4] = 0;                                      // tile_start[0]
        meta[5] = (M + kGemvTokTile - 1) / kGemvTokTile;  // tile_start[1]
        meta[6] = 0;                                      // tile_start_tc[0]
        meta[7] = (M + kTcTokTile - 1) / kTcTokTile;      // tile_start_tc[1]
    }
    if (threadIdx.x < kCounters) counters[threadIdx.x] = 0;
}

}  // namespace

}  // namespace nvfp4

using namespace nvfp4;

extern "C" size_t nvfp4_moe_workspace_size(int T, int E, int top_k, int d, int F, int mode) {
    if (T < 0 || E < 1 || top_k < 1 || d < 1 || F < 1 || (mode != 0 && mode != 1)) return 0;
    size_t b = 0;
    carve_moe(nullptr, T, E, top_k, d, F, mode, &b);
    return b;
}

extern "C" nvfp4_status nvfp4_moe_workspace_views(void* ws, int T, int E, int top_k, int d, int F, int mode,
                                                  int32_t** topk_ids, float** topk_w, int32_t** expert_offsets,
                                                  int32_t** row_to_slot, int32_t** slot_to_row) {
    if (!ws || T < 0 || E < 1 || top_k < 1 || d < 1 || F < 1 || (mode != 0 && mode != 1))
        return NVFP4_ERR_INVALID_ARG;
    MoeWs w = carve_moe(ws, T, E, top_k, d, F, mode, nullptr);
    if (topk_ids) *topk_ids = w.ra.ids;
    if (topk_w) *topk_w = w.ra.w;
    if (expert_offsets) *expert_offsets = w.ra.offsets;
    if (row_to_slot) *row_to_slot = w.ra.row_to_slot;
    if (slot_to_row) *slot_to_row = w.ra.slot_to_row;
    return NVFP4_OK;
}

extern "C" nvfp4_status nvfp4_moe_workspace_intermediates(void* ws, int T, int E, int top_k, int d, int F,
                                                          int mode, uint16_t** h_bf16, uint8_t** xq, uint8_t** xs,
                                                          uint8_t** hq, uint8_t** hs) {
    if (!ws || T < 0 || E < 1 || top_k < 1 || d < 1 || F < 1 || (mode != 0 && mode != 1))
        return NVFP4_ERR_INVALID_ARG;
    MoeWs w = carve_moe(ws, T, E, top_k, d, F, mode, nullptr);
    if (h_bf16) *h_bf16 = w.h;
    if (xq) *xq = w.xq;
    if (xs) *xs = w.xs;
    if (hq) *hq = w.hq;
    if (hs) *hs = w.hs;
    return NVFP4_OK;
}

extern "C" nvfp4_status nvfp4_moe_w4a16(const uint16_t* x, int T, const float* logits, int top_k,
                                        const nvfp4_moe_weights* w, uint16_t* out, void* ws, size_t ws_bytes,
                                        int32_t* d_status, cudaStream_t stream) {
    return run_moe(0, x, T, logits, top_k, w, nullptr, nullptr, out, ws, ws_bytes, d_status, stream);
}

extern "C" nvfp4_status nvfp4_moe_w4a4(const uint16_t* x, int T, const float* logits, int top_k,
                                       const nvfp4_moe_weights* w, const float* is13, const float* is2,
                                       uint16_t* out, void* ws, size_t ws_bytes, int32_t* d_status,
                                       cudaStream_t stream) {
    return run_moe(1, x, T, logits, top_k, w, is13, is2, out, ws, ws_bytes, d_status, stream);
}

extern "C" size_t nvfp4_linear_workspace_size(int M, int K, int N) {
    if (M < 0 || K < 0 || N < 0) return 0;
    size_t b = 0;
    carve_lin(nullptr, M, K, N, &b);
    return b;
}

extern "C" nvfp4_status nvfp4_linear(const uint16_t* x, int M, int K, const nvfp4_w* w, int N,
                                     const nvfp4_w* w_up, uint16_t* out, void* ws, size_t ws_bytes,
                                     cudaStream_t stream) {
    if (M < 0 || K < 1 || N < 1 || !w) return NVFP4_ERR_INVALID_ARG;
    if (K % 64 != 0 || N % 16 != 0 || !gemv_supported_k(K)) return NVFP4_ERR_SHAPE;
    if (M == 0) return NVFP4_OK;
    if (!x || !out || !ws || !w_ok(*w) || (w_up && !w_ok(*w_up))) return NVFP4_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || !aligned16(ws) || !w_aligned(*w) || (w_up && !w_aligned(*w_up)))
        return NVFP4_ERR_ALIGN;
    if (ws_bytes < nvfp4_linear_workspace_size(M, K, N)) return NVFP4_ERR_WORKSPACE;
    LinWs l = carve_lin(ws, M, K, N, nullptr);
    NVFP4_LAUNCH("linear_prep", stream, launch_pdl(linear_prep_kernel, dim3(1), dim3(32), 0, stream, M, l.meta,
                                                   l.counters));
    if (use_tc_linear(M, N)) {
        launch_rows_to_f16(x, M, K, l.xh, l.x_exp, nullptr, 0, stream);
        TcArgs t{};
        t.K = K;
        t.N = N;
        t.top_k = 1;
        t.offsets = l.meta + 0;
        t.active = l.meta + 2;
        t.n_active = l.meta + 3;
        t.tile_start = l.meta + 6;
        t.row_to_slot = nullptr;
        t.a_codes[0] = w->codes;  t.a_scales[0] = w->scales;  t.a_ws2[0] = w->weight_scale_2;
        t.a_codes[1] = w->codes;  t.a_scales[1] = w->scales;  t.a_ws2[1] = w->weight_scale_2;
        t.b_f16 = l.xh;
        t.b_exp = l.x_exp;
        t.b_by_token = 1;
        const int max_units = ((M + kTcTokTile - 1) / kTcTokTile) * (N / 128);
        TcmArgs g{};
        const bool tcm = tcm_supported(w_up ? TCM_SWIGLU : TCM_BF16, N, K);
        if (tcm) {
            if (!make_tmap_rows_f16(&g.tmap_x, l.xh, M, K)) return NVFP4_ERR_CUDA;
            g.K = K;
            g.N = N;
            g.top_k = 1;
            g.offsets = t.offsets;
            g.active = t.active;
            g.n_active = t.n_active;
            g.tile_start = t.tile_start;
            g.a_codes[0] = w->codes;  g.a_scales[0] = w->scales;  g.a_ws2[0] = w->weight_scale_2;
            g.a_codes[1] = w->codes;  g.a_scales[1] = w->scales;  g.a_ws2[1] = w->weight_scale_2;
            g.x_exp = l.x_exp;
        }
        if (tcm && w_up) {
            g.a_codes[1] = w_up->codes;  g.a_scales[1] = w_up->scales;  g.a_ws2[1] = w_up->weight_scale_2;
            g.h_out = out;
            if (!tcm_set_weights(&g, N)) return NVFP4_ERR_CUDA;
            launch_tcm(TCM_SWIGLU, g, max_units, stream);
        } else if (tcm) {
            g.y_out = out;
            if (!tcm_set_weights(&g, N)) return NVFP4_ERR_CUDA;
            launch_tcm(TCM_BF16, g, (max_units + 1) / 2, stream);
        } else if (w_up) {
            t.a_codes[1] = w_up->codes;  t.a_scales[1] = w_up->scales;  t.a_ws2[1] = w_up->weight_scale_2;
            t.h_out = out;
            launch_tc_gemm(TC_OUT_H, 2, t, max_units, stream);
        } else {
            t.y_out = out;
            launch_tc_gemm(TC_OUT_BF16, 1, t, max_units, stream);
        }
        return last_launch_status();
    }
    GemvArgs a{};
    a.K = K;
    a.N = N;
    a.top_k = 1;
    a.E = 1;
    a.offsets = l.meta + 0;
    a.active = l.meta + 2;
    a.n_active = l.meta + 3;
    a.tile_start = l.meta + 4;
    a.row_to_slot = nullptr;
    a.a_codes[0] = w->codes;  a.a_scales[0] = w->scales;  a.a_ws2[0] = w->weight_scale_2;
    a.a_codes[1] = w->codes;  a.a_scales[1] = w->scales;  a.a_ws2[1] = w->weight_scale_2;
    a.b_bf16 = x;
    a.b_by_token = 1;
    a.work_counter = l.counters;
    const int tiles = (M + kGemvTokTile - 1) / kGemvTokTile;
    const int max_work = gemv_max_work(M, 1, N);
    if (w_up) {
        a.nproj = 2;
        a.ksplit = gemv_pick_ksplit(tiles, N, 2);
        a.fb_group = gemv_pick_group(tiles, N, a.ksplit, 2);
        a.a_codes[1] = w_up->codes;  a.a_scales[1] = w_up->scales;  a.a_ws2[1] = w_up->weight_scale_2;
        a.h_out = out;
        launch_gemv(B_BF16, OUT_H, a, max_work, stream);
    } else {
        a.nproj = 1;
        a.ksplit = gemv_pick_ksplit(tiles, N, 1);
        a.fb_group = gemv_pick_group(tiles, N, a.ksplit, 1);
        a.y_out = out;
        launch_gemv(B_BF16, OUT_BF16, a, max_work, stream);
    }
    return last_launch_status();
}
