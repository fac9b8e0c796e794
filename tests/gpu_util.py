"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch

from serving_nvfp4_routed_gb300 import synth

REL_L2 = 5e-3        # layer output tolerance: relative L2 error
MAX_ABS_RMS = 2e-2   # layer output tolerance: max abs error / rms(oracle out)


def bf16_to_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (8 significant bits)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 2.0 ** -133)))
    return np.exp2(np.maximum(e, -126) - 7)


def assert_layer_close(got: np.ndarray, ref: np.ndarray, what=""):
    """rel L2 <= 5e-3, and every element within 2e-2 * rms(ref) of the
    oracle or on a bf16 neighbour of it: the kernels sum in fp32 in another
    order than the oracle's fp64 sum, so a value within ~2^-24 of a bf16
    rounding midpoint can land on the adjacent bf16 value at the final
    rounding; for an element above ~2.6 * rms that one step alone exceeds
    2e-2 * rms."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), what
    rms = np.sqrt(np.mean(ref ** 2))
    assert rms > 0
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    err = np.abs(got - ref)
    allowed = np.maximum(MAX_ABS_RMS * rms, bf16_ulp(ref) * 1.0000001)
    worst = np.argmax(err / allowed)
    assert rel <= REL_L2 and np.all(err <= allowed), (
        f"{what}: rel_l2={rel:.3g} max_abs/rms={err.max() / rms:.3g} worst: got {got.flat[worst]} "
        f"ref {ref.flat[worst]}")
    return rel, err.max() / rms


def oracle_bank(orc, banks: dict, experts=None):
    """Oracle-quantised copy of the bf16 banks (only `experts` filled; the
    rest of the stacked arrays stay zero)."""
    out = {}
    for name, w in banks.items():
        E, N, K = w.shape
        codes = np.zeros((E, N, K // 2), np.uint8)
        scales = np.zeros((E, N, K // 16), np.uint8)
        ws2 = np.zeros(E, np.float32)
        for e in (range(E) if experts is None else experts):
            c, s, g = orc.quantize_tensor(synth.bf16_bits(w[int(e)]))
            codes[e], scales[e], ws2[e] = c, s, g
        out[name] = (codes, scales, ws2)
    return out


def gpu_bank(lib, banks: dict):
    q = {name: lib.nvfp4_quantize_weights(w) for name, w in banks.items()}
    return lib.MoEWeights(q["gate"], q["up"], q["down"])


def assert_bank_equal(gw, ob, experts):
    for name in ("gate", "up", "down"):
        g = getattr(gw, name)
        oc, os_, o2 = ob[name]
        for e in experts:
            e = int(e)
            assert np.array_equal(g.codes[e].cpu().numpy(), oc[e]), (name, e, "codes")
            assert np.array_equal(g.scales[e].cpu().numpy(), os_[e]), (name, e, "scales")
            assert g.weight_scale_2[e].item() == o2[e], (name, e, "ws2")
