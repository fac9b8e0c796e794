"""Static activation-scale calibration for W4A4 -- TEST INFRASTRUCTURE.

Model card "GLM-5.3-Flash-NVFP4-W4A4-Experts", "Quantization boundary": the
static activation scales are calibrated, with a 5 % safety margin, at a
percentile of the calibrated amax (p99 by default; p98 / p98.9 for w2 at
some layers).  Reading used here, per expert and per projection:

    input_scale[e] = percentile_p(block amaxes of the rows routed to e) * 1.05 / 2688

where a block amax is max |v| over 16 consecutive inputs, the percentile is
numpy's default (linear interpolation), and 2688 = 6 * 448 puts the scale in
the same role as weight_scale_2 (the block scale of the calibrated amax lands
on the top of the e4m3 range).  w13 (gate/up) rows are the bf16 x rows; w2
(down) rows are the W4A16 h rows of the same tokens.  An expert that no
calibration row reaches takes the percentile over all experts' rows of that
projection (the model card's "across experts" policy).
"""
from __future__ import annotations

import numpy as np

from . import oracle


# the card's converted layers: the base routed-expert layers 3..44
ROUTED_LAYERS = range(3, 45)


def layer_percentiles(layer: int) -> tuple[float, float]:
    """(pct13, pct2) of the card's activation-scale policy for a routed layer
    (model card "GLM-5.3-Flash-NVFP4-W4A4-Experts", the activation-scale
    policy: p99 by default, p98 for w2 at layers 3-8, p98.9 for w2 at layers
    24-44; gate/up always p99)."""
    if layer not in ROUTED_LAYERS:
        raise ValueError(f"layer {layer} is not a converted routed-expert layer (3..44)")
    if layer <= 8:
        return 99.0, 98.0
    if layer >= 24:
        return 99.0, 98.9
    return 99.0, 99.0


def _block_amax(rows: np.ndarray) -> np.ndarray:
    n, K = rows.shape
    return np.abs(rows.reshape(n, K // 16, 16)).max(axis=2).reshape(-1)


def _bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def calibrate(x_bits: np.ndarray, logits: np.ndarray, top_k: int, bank, pct13: float = 99.0,
              pct2: float = 99.0, margin: float = 1.05):
    """Returns (is13 [E] f32, is2 [E] f32) from a calibration draw."""
    r = oracle.route(logits, top_k)
    ids = r["ids"]
    T, d = x_bits.shape
    E = bank["gate"][0].shape[0]
    xf = _bf16_bits_to_f32(np.ascontiguousarray(x_bits, np.uint16))
    _, h = oracle.moe_layer("w4a16", x_bits, ids, r["w"], bank, want_h=True)  # h [T, k, F]
    F = h.shape[2]
    per13 = [[] for _ in range(E)]
    per2 = [[] for _ in range(E)]
    for t in range(T):
        for j in range(top_k):
            e = int(ids[t, j])
            per13[e].append(_block_amax(xf[t:t + 1]))
            per2[e].append(_block_amax(h[t, j:j + 1].astype(np.float32)))
    all13 = np.concatenate([np.concatenate(v) for v in per13 if v])
    all2 = np.concatenate([np.concatenate(v) for v in per2 if v])
    fb13 = np.percentile(all13, pct13)
    fb2 = np.percentile(all2, pct2)
    is13 = np.empty(E, np.float32)
    is2 = np.empty(E, np.float32)
    for e in range(E):
        p13 = np.percentile(np.concatenate(per13[e]), pct13) if per13[e] else fb13
        p2 = np.percentile(np.concatenate(per2[e]), pct2) if per2[e] else fb2
        is13[e] = np.float32(p13 * margin / 2688.0)
        is2[e] = np.float32(p2 * margin / 2688.0)
    return is13, is2
