"""The oracle's pins catch plausible mistakes: each case plants one mistake
in a copy of the oracle's C source (a dropped term, a wrong sign, a
transposed operand, a wrong tie rule or bias, a swapped nibble order),
builds it, and checks that at least one pin fails.  CPU only."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import test_oracle_codecs as codecs
import test_oracle_layer as layer
import test_oracle_recipe as recipe
import test_oracle_route as route
from oracle import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "nvfp4_oracle.c")

MUTATIONS = {
    "e2m1 ties to the odd code": ("(d == bestd && (c & 1) == 0)", "(d == bestd && (c & 1) == 1)"),
    "e4m3 exponent bias 8": ("ldexp(1.0, e - 7)", "ldexp(1.0, e - 8)"),
    "global scale amax/2687": ("amax / 2688.0f", "amax / 2687.0f"),
    "odd index in the low nibble": ("(uint8_t)(q0 | (q1 << 4))", "(uint8_t)(q1 | (q0 << 4))"),
    "gate and up transposed": ("dequant_f32(gq + (int64_t)e * F * (d / 2), gs + (int64_t)e * F * (d / 16), F, d, Wg);",
                               "dequant_f32(uq + (int64_t)e * F * (d / 2), us + (int64_t)e * F * (d / 16), F, d, Wg);"),
    "down weight_scale_2 dropped": ("y[n] * hscale * (double)d_ws2[e]", "y[n] * hscale"),
    "silu sign": ("return g / (1.0 + exp(-g));", "return g / (1.0 + exp(g));"),
    "top-k ties to the higher id": ("if (best < 0 || rank_key(l[e]) > rank_key(l[best])) best = e;",
                                    "if (best < 0 || rank_key(l[e]) >= rank_key(l[best])) best = e;"),
    "renormalised over all experts": ("den += num[j];", "den += num[j] * 1.5;"),
    "block scale without the /6": ("float sf = (bam / 6.0f) / gs;", "float sf = bam / gs;"),
    "permutation not stable": ("int64_t row = fill[ids[i]]++;", "int64_t row = offsets[ids[i] + 1] - 1 - (fill[ids[i]]++ - offsets[ids[i]]);"),
}


def _pins(orc):
    """Run the pins; return the names of those that fail."""
    import torch

    failed = []
    checks = {
        "e2m1 table": lambda: codecs.test_e2m1_decode_matches_format_table(orc),
        "e2m1 ties": lambda: codecs.test_e2m1_encode_ties_and_saturation(orc),
        "e4m3 points": lambda: codecs.test_e4m3_decode_fixed_points(orc),
        "nibble order": lambda: recipe.test_nibble_order(orc),
        "on-grid requant": lambda: recipe.test_requantise_on_grid_is_identity(orc),
        "route ties": lambda: route.test_route_ties_go_to_lower_id(orc),
        "route random": lambda: route.test_route_random(orc),
        "single expert = dense": lambda: layer.test_single_expert_equals_dense_mlp(orc),
        "larger brute force": lambda: layer.test_larger_shape_brute_force(orc),
    }
    for name, fn in checks.items():
        try:
            fn()
        except AssertionError:
            failed.append(name)
    # the recipe's global-scale and brute-force pins, restated on a small tensor
    from serving_nvfp4_routed_gb300 import synth

    w = synth.make_weights(1, 32, 256, seed=11)[0]
    bits = synth.bf16_bits(w)
    _, _, ws2 = orc.quantize_tensor(bits)
    amax = np.abs((bits.astype(np.uint32) << 16).view(np.float32)).max()
    if ws2 != np.float32(amax) / np.float32(2688.0):
        failed.append("global scale")
    return failed


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old}"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so),
                    str(mutated), "-lm"], check=True)
    saved = oracle._lib
    try:
        oracle._lib = oracle.bind(ctypes.CDLL(str(so)))
        failed = _pins(oracle)
    finally:
        oracle._lib = saved
    assert failed, f"no pin caught the planted mistake '{name}'"


def test_unmutated_oracle_passes_all(orc):
    assert _pins(orc) == []
