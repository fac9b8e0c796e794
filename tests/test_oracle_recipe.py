"""Pins for the oracle's ModelOpt NVFP4 recipe and static activation quant.

Properties the recipe fixes, independent of how the oracle computes them:
  * weight_scale_2 = amax / 2688 exactly (fp32 division);
  * the block holding the tensor's amax gets the top e4m3 scale (0x7E);
  * every block with a normal e4m3 scale has a code of magnitude 6 at its
    largest element (e4m3 rounding keeps bam / (S*ws2) within [5.65, 6.4]);
  * per-element error <= 1.0625 * block_amax / 6 for normal-scale blocks;
  * a tensor already on the NVFP4 grid (power-of-two ws2, every block with a
    +-6 code) re-quantises to the same codes and scales;
  * an all-zero tensor gives ws2 = 0 and all-zero codes and scales;
  * low nibble = even index.
"""
import numpy as np
import pytest
import torch

from serving_nvfp4_routed_gb300 import synth


def _f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _codes_unpacked(codes):
    c = np.asarray(codes)
    out = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = c & 15
    out[..., 1::2] = c >> 4
    return out


E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])


def _e4m3(b):
    return torch.from_numpy(np.asarray(b, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


@pytest.fixture(scope="module")
def tensor(orc):
    w = synth.make_weights(1, 96, 512, seed=11)[0]
    bits = synth.bf16_bits(w)
    codes, scales, ws2 = orc.quantize_tensor(bits)
    return bits, codes, scales, ws2


def test_global_scale(tensor):
    bits, codes, scales, ws2 = tensor
    amax = np.abs(_f32(bits)).max()
    assert ws2 == np.float32(amax) / np.float32(2688.0)


def test_top_block_scale_is_448(tensor):
    bits, codes, scales, ws2 = tensor
    assert scales.max() == 0x7E
    v = np.abs(_f32(bits)).reshape(96, 32, 16).max(-1)
    n, j = np.unravel_index(np.argmax(v), v.shape)
    assert scales[n, j] == 0x7E


def test_normal_blocks_reach_six_and_error_bound(tensor):
    bits, codes, scales, ws2 = tensor
    v = _f32(bits).astype(np.float64).reshape(96, 32, 16)
    q = _codes_unpacked(codes).reshape(96, 32, 16)
    S = _e4m3(scales)
    normal = (scales >> 3) > 0
    assert normal.mean() > 0.99
    bam = np.abs(v).max(-1)
    for n in range(96):
        for j in range(32):
            if not normal[n, j]:
                continue
            i = np.argmax(np.abs(v[n, j]))
            assert (q[n, j, i] & 7) == 7
            deq = E2M1[q[n, j]] * S[n, j] * float(ws2)
            assert np.all(np.abs(deq - v[n, j]) <= 1.0625 * bam[n, j] / 6 + 1e-12)
    # signs of nonzero codes follow the input
    nz = (q & 7) != 0
    assert np.all(((q >> 3) == 1)[nz] == (v < 0)[nz])


def test_requantise_on_grid_is_identity(orc):
    rng = np.random.default_rng(5)
    N, K = 8, 64
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    q.reshape(N, K // 16, 16)[:, :, 3] = rng.choice([7, 15], size=(N, K // 16))
    s = rng.integers(0x30, 0x7E, size=(N, K // 16)).astype(np.uint8)
    s[0, 0] = 0x7E
    q[0, 0:16] = np.where(np.arange(16) == 3, 7, q[0, 0:16])  # +6 * 448 is the amax
    ws2 = np.float32(2.0 ** -12)
    vals = E2M1[q] * np.repeat(_e4m3(s), 16, axis=1) * float(ws2)
    bits = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(bits.to(torch.float64), torch.from_numpy(vals))  # values are bf16-exact
    codes, scales, got_ws2 = orc.quantize_tensor(synth.bf16_bits(bits))
    assert got_ws2 == ws2
    assert np.array_equal(scales, s)
    # -0 inputs come back as +0 codes only where the value is +0; compare values and nonzero codes
    cu = _codes_unpacked(codes)
    assert np.array_equal(E2M1[cu], E2M1[q])
    assert np.array_equal(cu[(q & 7) != 0], q[(q & 7) != 0])


def test_zero_tensor(orc):
    bits = np.zeros((4, 32), np.uint16)
    codes, scales, ws2 = orc.quantize_tensor(bits)
    assert ws2 == 0 and not codes.any() and not scales.any()


def test_nibble_order(orc):
    # x = [6*448*g at index 0, 0 at index 1, ...]: code 7 in the LOW nibble of byte 0
    v = np.zeros((1, 16), np.float32)
    v[0, 0] = 1.0
    v[0, 1] = -0.5
    bits = synth.bf16_bits(torch.from_numpy(v).to(torch.bfloat16))
    codes, scales, ws2 = orc.quantize_tensor(bits)
    assert codes[0, 0] & 15 == 7
    assert codes[0, 0] >> 4 == 13  # -0.5 / (448 * (1/2688)) = -3 -> code 5 | sign bit 8
    assert scales[0, 0] == 0x7E


def test_activation_quant_static_scale(orc):
    """Static input_scale: sf may exceed 448 and saturates to 0x7E, codes to +-6;
    doubling the input scale of a row whose blocks are all normal and unsaturated
    halves every block scale and keeps every code."""
    x = synth.make_x(6, 256, seed=3)
    bits = synth.bf16_bits(x)
    xf = _f32(bits).reshape(6, 256)
    amax = np.abs(xf).max()
    gs = np.full(6, np.float32(amax / 2688.0), np.float32)
    c1, s1 = orc.quantize_rows(bits, gs)
    c2, s2 = orc.quantize_rows(bits, gs * np.float32(2.0))
    ok = ((s1 >> 3) > 1) & (s1 < 0x7E)
    assert ok.mean() > 0.95
    assert np.array_equal(_e4m3(s2)[ok] * 2, _e4m3(s1)[ok])
    cu1 = _codes_unpacked(c1).reshape(6, 16, 16)
    cu2 = _codes_unpacked(c2).reshape(6, 16, 16)
    assert np.array_equal(cu1[ok], cu2[ok])
    # tiny scale: everything saturates
    c3, s3 = orc.quantize_rows(bits, np.full(6, 1e-6, np.float32))
    assert np.all((s3 == 0x7E) | (s3 == 0))
    big = np.abs(xf) > 6 * 448 * 1e-6
    assert np.all((_codes_unpacked(c3).reshape(6, 256) & 7)[big] == 7)
