"""The rule behind the kernels' e2m1 quotient shortcut, checked on the CPU.

The quantisers take the e2m1 code of fl(v / d) from q' = fl(v * fl(1/d))
unless the bits of q' lie within 4 ulp of a significand 1, 1.25, 1.5 or 1.75
(there they divide).  The claim: outside that window q' and fl(v / d) give
the same e2m1 code.  numpy float32 arithmetic is IEEE round-to-nearest, so
this replays the rule exactly on millions of quotients, random and placed
within a few ulp of every e2m1 rounding boundary."""
import numpy as np

# e2m1 magnitude codes by round-to-nearest-even on the grid 0,.5,1,1.5,2,3,4,6
_EDGES = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)


def _code(q):
    a = np.abs(q)
    c = np.searchsorted(_EDGES, a, side="left").astype(np.int32)  # a <= edge -> lower code
    # ties at an edge go to the even code: 0.75 -> 2 (1.0), 1.75 -> 4 (2.0), 3.5 -> 6 (4.0)
    tie_up = np.isin(a, _EDGES[[1, 3, 5]])
    c = np.where(tie_up, c + 1, c)
    return np.minimum(c, 7) | (np.signbit(q).astype(np.int32) << 3)


def _check(v, d):
    v = v.astype(np.float32)
    d = d.astype(np.float32)
    exact = v / d
    r = np.float32(1) / d
    q = v * r
    bits = q.view(np.uint32)
    near = ((bits + np.uint32(4)) & np.uint32(0x1FFFFF)) <= 8
    ok = near | (_code(q) == _code(exact))
    assert ok.all(), (v[~ok][:5], d[~ok][:5])
    return near.mean()


def test_edge_table():
    q = np.array([0.25, 0.7500001, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -0.1, 0.0], np.float32)
    assert list(_code(q)) == [0, 2, 2, 2, 4, 4, 6, 6, 7, 8, 0]


def test_random_quotients():
    rng = np.random.default_rng(1)
    n = 2_000_000
    v = rng.standard_normal(n) * np.exp2(rng.integers(-20, 20, n))
    d = np.abs(rng.standard_normal(n)) * np.exp2(rng.integers(-20, 20, n)) + 1e-30
    assert _check(v, d) < 1e-3


def test_quotients_next_to_every_boundary():
    rng = np.random.default_rng(2)
    n = 400_000
    edge = rng.choice(_EDGES, n) * rng.choice([-1, 1], n)
    d = (rng.uniform(0.5, 2.0, n) * np.exp2(rng.integers(-12, 12, n))).astype(np.float32)
    # v on the float32 grid near edge * d, a few ulp either side
    v = (edge * d).astype(np.float32)
    v = v.view(np.int32) + rng.integers(-6, 7, n).astype(np.int32)
    _check(v.view(np.float32), d)
