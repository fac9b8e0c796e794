"""Element-by-element parity of one routed-layer call against the oracle,
with the kernel's intermediates checked on the way (no method arithmetic:
the expected values come from the oracle; this file only compares).

For the listed tokens:
  * routing arrays in the workspace equal the oracle's (bit-exact);
  * W4A4: every pair's NVFP4 x row (codes + scales) equals the oracle's;
  * h (W4A16: bf16 h; W4A4: its NVFP4 requantisation) equals the oracle's
    or lies in the interval the error model allows (gpu_util.h_interval);
  * the output satisfies gpu_util.assert_out_close with the bound
        (gamma(F) + (k + 2) 2^-24) * out_abs  +  effect of the h differences,
    where out_abs is the oracle's sum_j |w_j| * scale * sum_f |h_f W_d|;
  * paths that keep each routed row's y in bf16 (round_y, the prompt-shaped
    kernels) round at R3 too: each kernel Y_j lies in
    [bf16(y_j - e_j), bf16(y_j + e_j)] around the oracle's unrounded y_j,
    e_j = gamma(F) * y_abs_j + 2^-23 |y_j| + the effect of the pair's h
    differences, and the bound is sum_j |w_j| D_j + (k + 1) 2^-24
    sum_j |w_j| (|bf16(y_j)| + D_j), D_j the widest distance from bf16(y_j)
    to that interval's ends.
"""
import numpy as np
import torch

import serving_nvfp4_routed_gb300 as lib
from gpu_util import (U32, assert_h_in_interval, assert_out_close, bf16_to_f32, gamma, h_interval,
                      nvfp4_block_feasible, round_bf16, unpack_codes)
from serving_nvfp4_routed_gb300 import synth


def _e4m3(b):
    return torch.from_numpy(np.ascontiguousarray(b, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])


def _deq_rows(codes, scales):
    """dec(code) * dec(scale) of NVFP4 rows [..., K/2], [..., K/16] -> [..., K]
    (format decode only, for the size of a difference)."""
    return E2M1[unpack_codes(codes)] * np.repeat(_e4m3(scales), 16, axis=-1)


def check_layer(orc, mode, x, logits, k, ob, out, ws, tok, is13=None, is2=None, what="", round_y=False):
    """Compare the layer output `out` (GPU, [T, d] bf16, computed with the
    workspace `ws`) for tokens `tok` against the oracle; returns a report."""
    T, d = x.shape
    E = ob["gate"][0].shape[0]
    F = ob["gate"][0].shape[1]
    xb = synth.bf16_bits(x)
    r = orc.route(logits.cpu().numpy(), k)
    v = lib.moe_workspace_views(ws, T, E, k, d, F, mode)
    assert np.array_equal(v["ids"].cpu().numpy(), r["ids"]), f"{what}: routing ids"
    assert np.array_equal(v["slot_to_row"].cpu().numpy(), r["slot_to_row"]), f"{what}: permutation"
    ex = orc.moe_layer_ex(mode, xb, r["ids"], r["w"], ob, tokens=tok, is13=is13, is2=is2, round_y=round_y)
    n = len(tok)
    rows = r["slot_to_row"].reshape(T, k)[tok]  # [n, k] permuted row of each pair
    ids = r["ids"][tok]
    inter = lib.moe_workspace_intermediates(ws, T, E, k, d, F, mode)
    rs_exact = mode == "w4a16"
    h_lo, h_hi = h_interval(ex["g_pre"], ex["u_pre"], ex["g_abs"], ex["u_abs"], d, rs_exact)
    # per pair: the difference between the kernel's h and the oracle's, in
    # the units the down projection multiplies (without the tensor scales)
    delta = np.zeros((n, k, F))
    scale_d = np.ones((n, k))
    if mode == "w4a16":
        hk = bf16_to_f32(inter["h"][torch.from_numpy(rows.reshape(-1)).long().to(inter["h"].device)]).reshape(n, k, F)
        assert_h_in_interval(hk, h_lo, h_hi, f"{what}: h")
        delta = hk.astype(np.float64) - ex["h"]
    else:
        idx = torch.from_numpy(rows.reshape(-1)).long().to(inter["xq"].device)
        xq = inter["xq"][idx].cpu().numpy().reshape(n, k, d // 2)
        xs = inter["xs"][idx].cpu().numpy().reshape(n, k, d // 16)
        assert np.array_equal(xq, ex["xq"]) and np.array_equal(xs, ex["xs"]), f"{what}: NVFP4 x rows"
        hq = inter["hq"][idx].cpu().numpy().reshape(n, k, F // 2)
        hs = inter["hs"][idx].cpu().numpy().reshape(n, k, F // 16)
        qk = unpack_codes(hq).reshape(n, k, F // 16, 16)
        qo = unpack_codes(ex["hq"]).reshape(n, k, F // 16, 16)
        differ = (hs != ex["hs"]) | np.any(qk != qo, axis=-1)
        for (i, j, b) in zip(*np.nonzero(differ)):
            sl = slice(16 * b, 16 * b + 16)
            assert nvfp4_block_feasible(orc, h_lo[i, j, sl], h_hi[i, j, sl], float(is2[ids[i, j]]),
                                        int(hs[i, j, b]), qk[i, j, b]), (
                f"{what}: NVFP4 h block (token {tok[i]}, slot {j}, block {b}) not reachable from the allowed h")
        delta = _deq_rows(hq, hs) - _deq_rows(ex["hq"], ex["hs"])
        scale_d = np.asarray(is2, np.float64)[ids]
    # effect of each pair's h differences on its y, through |W_d|
    h_eff = np.zeros((n, k, d))
    wts = np.abs(r["w"][tok].astype(np.float64))
    dq, dsc, d2 = ob["down"]
    cache = {}
    for i, j in zip(*np.nonzero(np.any(delta != 0, axis=-1))):
        e = int(ids[i, j])
        if e not in cache:
            cache[e] = np.abs(orc.dequantize(dq[e], dsc[e]))
        h_eff[i, j] = float(d2[e]) * scale_d[i, j] * (cache[e] @ np.abs(delta[i, j]))
    if round_y:
        e_y = gamma(F) * ex["y_abs"] + 2 * U32 * np.abs(ex["y_pre"]) + h_eff
        y_r = round_bf16(ex["y_pre"])
        dist = np.maximum(y_r - round_bf16(ex["y_pre"] - e_y), round_bf16(ex["y_pre"] + e_y) - y_r)
        bound = (np.einsum("nk,nkd->nd", wts, dist)
                 + (k + 1) * U32 * np.einsum("nk,nkd->nd", wts, np.abs(y_r) + dist))
    else:
        bound = (gamma(F) + (k + 2) * U32) * ex["out_abs"] + np.einsum("nk,nkd->nd", wts, h_eff)
    got = bf16_to_f32(out)[tok]
    rep = assert_out_close(got, ex["out"], ex["out_pre"], bound, what)
    rep["h_pairs_differing"] = int(np.any(delta != 0, axis=-1).sum())
    return rep


def check_linear_h(orc, x, qg_o, qu_o, h_got, what=""):
    """nvfp4_linear with w_up: the kernel's h rows [M, N] against the oracle
    (qg_o / qu_o: the oracle's (codes, scales, ws2)): every element inside
    the interval of the error model, plus the output tolerance."""
    ex = orc.linear_ex(synth.bf16_bits(x), qg_o[0], qg_o[1], qg_o[2], wup=qu_o)
    K = x.shape[1]
    lo, hi = h_interval(ex["g_pre"], ex["u_pre"], ex["g_abs"], ex["u_abs"], K, True)
    assert_h_in_interval(h_got, lo, hi, what)
    # the output rule: within 2e-2 rms, or a neighbour inside the interval
    bound = np.maximum(np.abs(ex["pre"] - lo), np.abs(ex["pre"] - hi))
    rep = assert_out_close(h_got, ex["out"], ex["pre"], bound, what)
    return ex, rep


def check_linear_y(orc, xbits, q_o, y_got, what=""):
    """nvfp4_linear without w_up: y = bf16(ws2 * x W^T) against the oracle."""
    ex = orc.linear_ex(xbits, q_o[0], q_o[1], q_o[2])
    K = xbits.shape[1]
    bound = gamma(K) * ex["g_abs"] + 2 * U32 * np.abs(ex["pre"])
    return assert_out_close(y_got, ex["out"], ex["pre"], bound, what)
