"""Pins for the oracle's e2m1 / e4m3 / bf16 codecs (CPU only).

Each codec is checked against something other than itself: the format's
fixed value table (tests/golden), the interval form of round-to-nearest-even,
the closed form of e4m3, and torch's own float8_e4m3fn / bfloat16 casts.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def test_e2m1_decode_matches_format_table(orc):
    rows = _rows("e2m1_values.txt")
    assert len(rows) == 16
    for code, val in rows:
        got = orc.e2m1_decode(int(code))
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def _interval_code(a, table):
    for lo, loc, hi, hic, code in table:
        lo, hi = float(lo), float(hi)
        above = a >= lo if loc == "1" else a > lo
        below = a <= hi if hic == "1" else a < hi
        if above and below:
            return int(code)
    raise AssertionError(a)


def test_e2m1_encode_all_bf16_in_range(orc):
    """Every bf16 value in [-8, 8] rounds as the interval table says."""
    table = _rows("e2m1_rounding.txt")
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    sel = np.isfinite(vals) & (np.abs(vals) <= 8.0)
    n = 0
    for v in vals[sel]:
        code = orc.e2m1_encode(float(v))
        want = _interval_code(abs(float(v)), table) | (8 if math.copysign(1.0, v) < 0 else 0)
        assert code == want, (float(v), code, want)
        n += 1
    assert n > 30000


def test_e2m1_encode_ties_and_saturation(orc):
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for v, c in ties.items():
        assert orc.e2m1_encode(v) == c
        assert orc.e2m1_encode(-v) == c | 8
    for v in (6.0, 6.5, 7.0, 1e6, 3.4e38):
        assert orc.e2m1_encode(v) == 7
        assert orc.e2m1_encode(-v) == 15
    assert orc.e2m1_encode(-0.0) == 8
    assert orc.e2m1_encode(-1e-3) == 8


def test_e4m3_decode_fixed_points(orc):
    for b, val in _rows("e4m3_points.txt"):
        got = orc.e4m3_decode(int(b, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val)


def test_e4m3_decode_all_bytes_match_torch(orc):
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        got = orc.e4m3_decode(b)
        if math.isnan(t[b]):
            assert math.isnan(got)
        else:
            assert got == t[b], (b, got, t[b])


def test_e4m3_encode_matches_torch_cast(orc):
    """Nearest-even e4m3 of fp32 values in [0, 448]: the representable values,
    their midpoints, one fp32 ulp either side of each midpoint, and random
    values -- against torch's float32 -> float8_e4m3fn cast."""
    finite = np.array([orc.e4m3_decode(b) for b in range(127)], np.float64)
    mids = (finite[:-1] + finite[1:]) / 2
    pts = [finite, mids]
    m32 = mids.astype(np.float32)
    pts.append(np.nextafter(m32, np.float32(np.inf)).astype(np.float64))
    pts.append(np.nextafter(m32, np.float32(0)).astype(np.float64))
    rng = np.random.default_rng(7)
    pts.append(rng.uniform(0, 448, 20000))
    pts.append(np.exp(rng.uniform(np.log(1e-4), np.log(448), 20000)))
    v = np.concatenate(pts).astype(np.float32)
    v = v[(v >= 0) & (v <= 448)]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, r in zip(v, ref):
        assert orc.e4m3_encode(float(x)) == int(r), (float(x), int(r))


def test_e4m3_encode_saturates(orc):
    for v in (448.0, 450.0, 464.0, 500.0, 1e9):
        assert orc.e4m3_encode(v) == 0x7E
    assert orc.e4m3_encode(0.0) == 0
    # below half the smallest subnormal (2^-10) rounds to zero; exactly half ties to even (0)
    assert orc.e4m3_encode(2.0 ** -10) == 0
    assert orc.e4m3_encode(2.0 ** -10 * 1.01) == 1


def test_round_bf16_matches_torch_on_fp32(orc):
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        rng.standard_normal(2000)]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    for x, r in zip(v, ref):
        assert orc.round_bf16(float(x)) == r


def test_round_bf16_ties_to_even(orc):
    one = 1.0
    ulp = 2.0 ** -7
    assert orc.round_bf16(one + ulp / 2) == one          # tie -> even (1.0)
    assert orc.round_bf16(one + 3 * ulp / 2) == one + 2 * ulp
    assert orc.round_bf16(one + ulp / 2 + 1e-12) == one + ulp
    assert orc.round_bf16(-(one + ulp / 2)) == -one
