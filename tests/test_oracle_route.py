"""Pins for the oracle's routing and permutation (CPU only).

  * top-k ids = brute-force sort on (-logit, expert id) (ties -> lower id);
  * weights = torch.softmax in fp64 over all E, gathered and renormalised;
  * permutation = numpy's stable argsort of the flattened ids;
  * offsets = exclusive cumulative sum of the per-expert counts;
  * -inf logits are never chosen while k finite ones remain.
"""
import numpy as np
import torch

from serving_nvfp4_routed_gb300 import synth


def _check(orc, logits, k):
    r = orc.route(logits, k)
    T, E = logits.shape
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        assert list(r["ids"][t]) == order
    p = torch.softmax(torch.from_numpy(logits.astype(np.float64)), dim=-1).numpy()
    sel = np.take_along_axis(p, r["ids"].astype(np.int64), axis=1)
    want = sel / sel.sum(1, keepdims=True)
    np.testing.assert_allclose(r["w"], want, rtol=2e-7, atol=1e-30)
    flat = r["ids"].reshape(-1)
    perm = np.argsort(flat, kind="stable")
    assert np.array_equal(r["row_to_slot"], perm)
    assert np.array_equal(r["slot_to_row"][perm], np.arange(T * k))
    counts = np.bincount(flat, minlength=E)
    assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(counts)]))
    return r


def test_route_random(orc):
    lg = synth.make_logits(64, 288, seed=1).numpy()
    r = _check(orc, lg, 8)
    s = r["w"].astype(np.float64).sum(1)
    assert np.all(np.abs(s - 1) <= 8 * 2.0 ** -24)


def test_route_tiny(orc):
    _check(orc, synth.make_logits(4, 8, seed=2).numpy(), 2)


def test_route_ties_go_to_lower_id(orc):
    lg = np.zeros((3, 10), np.float32)
    lg[1, [7, 3, 5]] = 1.0
    lg[2, :] = -1.0
    lg[2, 9] = 2.0
    r = _check(orc, lg, 4)
    assert list(r["ids"][0]) == [0, 1, 2, 3]
    assert list(r["ids"][1]) == [3, 5, 7, 0]
    assert list(r["ids"][2]) == [9, 0, 1, 2]
    np.testing.assert_allclose(r["w"][0], 0.25, rtol=0)


def test_route_masked_experts_never_chosen(orc):
    lg = synth.make_logits(512, 288, seed=4, kind="zipf_masked").numpy()
    masked = np.where(np.isinf(lg[0]))[0]
    assert len(masked) == 96
    r = orc.route(lg, 8)
    assert not np.isin(r["ids"], masked).any()
    counts = np.diff(r["offsets"])
    assert np.all(counts[masked] == 0)


def test_route_zipf_skew(orc):
    lg = synth.make_logits(4096, 288, seed=5, kind="zipf").numpy()
    r = orc.route(lg, 8)
    counts = np.sort(np.diff(r["offsets"]))[::-1]
    top3 = counts[:3].sum() / counts.sum()
    assert 0.2 < top3 < 0.35


def test_route_non_finite_logits(orc):
    """The reading for logits the pages never meet: NaN ranks as -inf; a
    +inf top logit gives its +inf entries equal weights and the rest 0; a
    token whose chosen logits are all -inf gets 1/k each.  Weights still sum
    to 1 and no index leaves its range."""
    lg = np.zeros((5, 12), np.float32)
    lg[0] = -np.inf
    lg[1, 4] = np.inf
    lg[2, [2, 7, 11]] = np.inf
    lg[3, :6] = np.nan
    lg[3, 6:] = np.arange(6)
    lg[4] = np.nan
    r = orc.route(lg, 4)
    assert np.all((r["ids"] >= 0) & (r["ids"] < 12))
    np.testing.assert_array_equal(r["w"][0], np.full(4, 0.25, np.float32))
    assert list(r["ids"][0]) == [0, 1, 2, 3]
    assert list(r["ids"][1][:1]) == [4] and list(r["w"][1]) == [1, 0, 0, 0]
    assert list(r["ids"][2][:3]) == [2, 7, 11]
    np.testing.assert_array_equal(r["w"][2], np.array([1 / 3, 1 / 3, 1 / 3, 0], np.float32))
    assert list(r["ids"][3]) == [11, 10, 9, 8]  # the NaN entries rank last
    np.testing.assert_array_equal(r["w"][4], np.full(4, 0.25, np.float32))
    assert np.all(np.abs(r["w"].astype(np.float64).sum(1) - 1) <= 4 * 2.0 ** -24)
