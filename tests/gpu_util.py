"""Helpers shared by the GPU parity tests (no method arithmetic here: the
expected values all come from the oracle; this file only decides how far a
kernel result may sit from them).

Tolerance (the layer's, from its statement of the problem): relative L2
error <= 5e-3 and every element within 2e-2 * rms(out) of the oracle.  An
element may miss that only by being a bf16 value that rounding some value
within a derived bound B of the oracle's unrounded value can give.  For
the fp32 sums alone B is far below half a bf16 step: the element is then
the oracle's value or, where the unrounded value lies within B of the
midpoint, its neighbour (the kernel's sums run in another order than the
oracle's fp64 ones and can round either way).

Error model of a kernel dot product over K terms (every product is exact
in fp32): the tensor-core and mma.sync kernels add at most 16 products per
MMA instruction (64 for the FP4 kind) to an fp32 accumulator; each
instruction is taken as one addition of the exact sum of its products with
at most one fp32 ulp (2^-23, which also covers truncation) of error
relative to |acc| + sum |products| <= the sum of all |terms|; up to 16 more
roundings cover split-K partial sums and the epilogue's scale multiplies:

    |kernel - exact| <= gamma(K) * sum|terms|,   gamma(K) = 2^-23 (K/16 + 16).

A layer output also moves when the kernel's h differs from the oracle's
(a gate / up value whose exact value lies near a bf16 midpoint rounds the
other way).  The tests read the kernel's h, check each element against the
interval the model allows, and add the effect of the observed differences
to the output's bound.  In W4A4 such a one-step difference in h can move
the NVFP4 code of h (or its block scale), and its effect on the output can
span several bf16 steps: B then covers it, computed from the differences
the kernel actually made after each has been checked to be one the model
allows.
"""
import numpy as np
import torch

from serving_nvfp4_routed_gb300 import synth

REL_L2 = 5e-3        # layer output tolerance: relative L2 error
MAX_ABS_RMS = 2e-2   # layer output tolerance: max abs error / rms(oracle out)
U32 = 2.0 ** -24     # unit roundoff of fp32
SILU_MIN_G = -1.2784645427610738  # argmin of g / (1 + exp(-g))


def gamma(K: int) -> float:
    """Bound constant of a kernel fp32 dot product over K terms (above)."""
    return 2.0 ** -23 * (K / 16.0 + 16.0)


def bf16_to_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def round_bf16(v) -> np.ndarray:
    """fp64 -> nearest bf16 value (8 significant bits, ties to even), as fp64
    (normal range; zeros kept)."""
    m, e = np.frexp(np.asarray(v, np.float64))
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def bf16_key(v) -> np.ndarray:
    """Monotone integer key of bf16 values (adjacent bf16 values differ by 1;
    -0 and +0 share a key)."""
    b = (np.asarray(v, np.float32).view(np.uint32) >> 16).astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def silu(g):
    g = np.asarray(g, np.float64)
    return g / (1.0 + np.exp(-g))


class Report(dict):
    pass


def assert_out_close(got, ref, pre, bound, what=""):
    """Layer / linear outputs: rel L2 <= 5e-3; every element within
    2e-2 * rms(ref) of the oracle, or a bf16 value that rounding a value
    within ``bound`` of the oracle's unrounded value ``pre`` can give
    (bf16(pre - bound) <= got <= bf16(pre + bound)).  With a bound below
    half a bf16 step that is the oracle's value itself or, where pre lies
    within the bound of the midpoint, its neighbour."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    pre = np.asarray(pre, np.float64)
    bound = np.broadcast_to(np.asarray(bound, np.float64), ref.shape)
    assert got.shape == ref.shape == pre.shape, (got.shape, ref.shape, pre.shape)
    assert np.all(np.isfinite(got)), what
    assert np.array_equal(round_bf16(pre), ref), f"{what}: oracle pre-rounding values do not round to its output"
    rms = np.sqrt(np.mean(ref ** 2))
    assert rms > 0, what
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    err = np.abs(got - ref)
    within = err <= MAX_ABS_RMS * rms
    reach = (got >= round_bf16(pre - bound)) & (got <= round_bf16(pre + bound))
    bad = ~(within | reach)
    steps = np.abs(bf16_key(got) - bf16_key(ref))
    rep = Report(rel_l2=rel, max_abs_rms=float(err.max() / rms), mismatched=int((got != ref).sum()),
                 beyond_tol=int((~within).sum()), max_steps_beyond_tol=int(steps[~within].max()) if (~within).any()
                 else 0, n=int(ref.size))
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(
            f"{what}: {int(bad.sum())} element(s) outside the tolerance; first at {np.unravel_index(i, ref.shape)}: "
            f"got {got.flat[i]!r} ref {ref.flat[i]!r} pre {pre.flat[i]!r} bound {bound.flat[i]:.3e} "
            f"(rms {rms:.4g}; {rep})")
    assert rel <= REL_L2, f"{what}: rel_l2={rel:.3g} ({rep})"
    return rep


def h_interval(g_pre, u_pre, g_abs, u_abs, K, rs_exact: bool):
    """The bf16 values the kernels may produce for h = bf16(silu(G) * U),
    G = bf16(gate sum * scales), U likewise, given the oracle's values before
    rounding and their |term| sums: [h_lo, h_hi] per element.  The kernel's
    G lies in [bf16(g - eG), bf16(g + eG)] with eG = gamma(K) g_abs plus the
    scale multiplies (two roundings; three when the row scale is not a
    power of two); silu(G) * U in fp32 (expf within 2 ulp, the add, the
    division, the product) is within 8 ulp of its exact value."""
    nr = 2 if rs_exact else 3
    eg = gamma(K) * np.asarray(g_abs) + nr * U32 * np.abs(g_pre)
    eu = gamma(K) * np.asarray(u_abs) + nr * U32 * np.abs(u_pre)
    g_lo, g_hi = round_bf16(g_pre - eg), round_bf16(g_pre + eg)
    u_lo, u_hi = round_bf16(u_pre - eu), round_bf16(u_pre + eu)
    s_a, s_b = silu(g_lo), silu(g_hi)
    s_lo = np.minimum(s_a, s_b)
    s_hi = np.maximum(s_a, s_b)
    inside = (g_lo < SILU_MIN_G) & (g_hi > SILU_MIN_G)
    s_lo = np.where(inside, silu(SILU_MIN_G), s_lo)
    c = np.stack([s_lo * u_lo, s_lo * u_hi, s_hi * u_lo, s_hi * u_hi])
    lo, hi = c.min(0), c.max(0)
    return round_bf16(lo - 8 * U32 * np.abs(lo)), round_bf16(hi + 8 * U32 * np.abs(hi))


def assert_h_in_interval(h_got, h_lo, h_hi, what=""):
    h_got = np.asarray(h_got, np.float64)
    bad = (h_got < h_lo) | (h_got > h_hi)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} h value(s) outside the interval the error model allows; "
                             f"first at {np.unravel_index(i, h_got.shape)}: got {h_got.flat[i]!r} allowed "
                             f"[{h_lo.flat[i]!r}, {h_hi.flat[i]!r}]")
    return int((h_lo != h_hi).sum())


def pick_tokens(r, T, k, n=32, seed=0):
    """At least ``n`` tokens of a full-size batch, covering the first and the
    last 128-row tile of the most popular expert, every row of the least
    popular expert that has any (a ragged tile), the first and the last
    routed row, and a seeded random rest."""
    offs = np.asarray(r["offsets"])
    r2s = np.asarray(r["row_to_slot"])
    counts = np.diff(offs)
    top = int(np.argmax(counts))
    rows = list(range(offs[top], min(offs[top] + 3, offs[top + 1])))
    rows += list(range(max(offs[top], offs[top + 1] - 3), offs[top + 1]))
    nz = np.flatnonzero(counts)
    low = int(nz[np.argmin(counts[nz])])
    rows += list(range(offs[low], min(offs[low + 1], offs[low] + 4)))
    rows += [0, int(offs[-1]) - 1]
    tok = set(int(r2s[i]) // k for i in rows)
    rng = np.random.default_rng(seed)
    for t in rng.permutation(T):
        if len(tok) >= n:
            break
        tok.add(int(t))
    return np.array(sorted(tok), np.int32)


class OracleBank:
    """Oracle-quantised copy of bf16 expert banks, filled expert by expert
    on demand and kept (a full-size bank takes minutes to quantise)."""

    def __init__(self, orc, banks: dict):
        self.orc = orc
        self.banks = banks
        self.done = set()
        self.q = {}
        for name, w in banks.items():
            E, N, K = w.shape
            self.q[name] = (np.zeros((E, N, K // 2), np.uint8), np.zeros((E, N, K // 16), np.uint8),
                            np.zeros(E, np.float32))

    def get(self, experts=None):
        E = next(iter(self.banks.values())).shape[0]
        for e in (range(E) if experts is None else experts):
            e = int(e)
            if e in self.done:
                continue
            for name, w in self.banks.items():
                c, s, g = self.orc.quantize_tensor(synth.bf16_bits(w[e]))
                self.q[name][0][e], self.q[name][1][e], self.q[name][2][e] = c, s, g
            self.done.add(e)
        return self.q


def oracle_bank(orc, banks: dict, experts=None):
    """Oracle-quantised copy of the bf16 banks (only `experts` filled; the
    rest of the stacked arrays stay zero)."""
    return OracleBank(orc, banks).get(experts)


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


def kernels_ran(lib, fn):
    """Run fn() with per-launch timing on and return (its result, the set of
    kernel names the library launched)."""
    lib.profile_collect()
    lib.profile_enable(True)
    try:
        res = fn()
        torch.cuda.synchronize()
    finally:
        lib.profile_enable(False)
    return res, set(lib.profile_collect().keys())


def _e2m1(orc, v):
    return orc.e2m1_decode(orc.e2m1_encode(float(v)))


def nvfp4_block_feasible(orc, h_lo, h_hi, gs, s_k, codes_k):
    """Whether the kernel's NVFP4 block (scale byte s_k, codes codes_k) is
    the quantisation (the block rule of the recipe under tensor scale gs) of
    some h with each element in [h_lo_i, h_hi_i]: the scale byte must lie
    between the scale bytes of the smallest and largest achievable block
    maxima (the rule is monotone in the maximum), and given that scale each
    code between the codes of its interval's ends (monotone too)."""
    f32 = np.float32
    amin = np.where((h_lo <= 0) & (h_hi >= 0), 0.0, np.minimum(np.abs(h_lo), np.abs(h_hi)))
    amax = np.maximum(np.abs(h_lo), np.abs(h_hi))

    def sbyte(m):
        return orc.e4m3_encode(float(f32(f32(f32(m) / f32(6.0)) / f32(gs))))

    if gs <= 0:
        return s_k == 0 and not np.any(codes_k)
    if not (sbyte(amin.max()) <= s_k <= sbyte(amax.max())):
        return False
    S = f32(orc.e4m3_decode(int(s_k)))
    if S == 0:
        return not np.any(codes_k)
    den = f32(S * f32(gs))
    for i in range(len(codes_k)):
        lo = _e2m1(orc, f32(f32(h_lo[i]) / den))
        hi = _e2m1(orc, f32(f32(h_hi[i]) / den))
        got = orc.e2m1_decode(int(codes_k[i]))
        if not (lo <= got <= hi):
            return False
    return True


def unpack_codes(packed):
    """[..., K/2] bytes -> [..., K] e2m1 codes (even index in the low nibble)."""
    p = np.asarray(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = p & 15
    out[..., 1::2] = p >> 4
    return out
