"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch

from serving_nvfp4_routed_gb300 import synth

REL_L2 = 5e-3        # layer output tolerance: relative L2 error
MAX_ABS_RMS = 2e-2   # layer output tolerance: max abs error / rms(oracle out)


def bf16_to_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def assert_layer_close(got: np.ndarray, ref: np.ndarray, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), what
    rms = np.sqrt(np.mean(ref ** 2))
    assert rms > 0
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    mabs = np.abs(got - ref).max()
    assert rel <= REL_L2 and mabs <= MAX_ABS_RMS * rms, f"{what}: rel_l2={rel:.3g} max_abs/rms={mabs / rms:.3g}"
    return rel, mabs / rms


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
