"""Pins of the oracle's nearest-E8-point search.

E8 = D8 u (D8 + 1/2): the decoder must return a lattice point at minimum
distance.  Pinned against (1) brute-force enumeration of every candidate
within one step of coordinate-wise rounding, (2) hand-derived golden cases
including ties, (3) lattice membership, (4) the normalised second moment of
E8, G(E8) = 929/12960 (Conway & Sloane, SPLAG, Table 2.3).
"""
import itertools
import os

import numpy as np
import pytest

import oracle
import synth


def _brute_force_min(x):
    """Minimum squared distance from x to E8 over all candidates near x."""
    best = np.inf
    offs = np.array(list(itertools.product((-1, 0, 1), repeat=8)), dtype=np.float64)  # 6561 x 8
    for c in (0.0, 0.5):
        base = np.round(x - c)
        cand = base[None, :] + offs
        even = (cand.sum(axis=1) % 2) == 0
        pts = cand[even] + c
        d = ((pts - x[None, :]) ** 2).sum(axis=1)
        best = min(best, d.min())
    return best


def _check_member(a, c):
    assert int(a.sum()) % 2 == 0, "E8 points have an even integer-part sum"
    assert c in (0, 1)


@pytest.mark.parametrize("scale", [0.7, 2.0, 9.0, 300.0])
def test_matches_brute_force(scale):
    rng_x = synth.normal_f64(101 + int(scale * 10), 8 * 120) * scale
    for i in range(120):
        x = rng_x[8 * i: 8 * i + 8]
        a, c = oracle.e8_nearest(x)
        _check_member(a, c)
        q = a + 0.5 * c
        d = float(((q - x) ** 2).sum())
        assert d <= _brute_force_min(x) * (1 + 1e-12) + 1e-12


def test_adversarial_ties_brute_force():
    # half-integers and quarter points make many equal-distance candidates
    vals = synth.uniform_f64(7, 8 * 300, -3, 3)
    x_all = np.round(vals * 4) / 4
    for i in range(300):
        x = x_all[8 * i: 8 * i + 8]
        a, c = oracle.e8_nearest(x)
        _check_member(a, c)
        d = float(((a + 0.5 * c - x) ** 2).sum())
        assert abs(d - _brute_force_min(x)) <= 1e-12


def test_golden_points(golden_dir):
    rows = 0
    for line in open(os.path.join(golden_dir, "e8_points.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        xs, as_, cs = [p.strip() for p in line.split("|")]
        x = np.array([float(v) for v in xs.split()])
        want_a = np.array([int(v) for v in as_.split()])
        a, c = oracle.e8_nearest(x)
        assert c == int(cs), line
        assert (a == want_a).all(), (line, a)
        rows += 1
    assert rows >= 7


def test_second_moment_of_e8():
    """Mean squared error per dimension for uniform inputs -> G(E8) = 929/12960."""
    n = 60000
    x = synth.uniform_f64(99, 8 * n, 0.0, 64.0).reshape(n, 8)
    err = np.empty(n)
    for i in range(n):
        a, c = oracle.e8_nearest(x[i])
        err[i] = ((a + 0.5 * c - x[i]) ** 2).sum() / 8.0
    g = 929.0 / 12960.0
    se = err.std() / np.sqrt(n)
    assert abs(err.mean() - g) < 4 * se, (err.mean(), g, se)


def test_invariant_large_batch():
    x = synth.normal_f64(5, 8 * 5000).reshape(5000, 8) * 5
    for i in range(5000):
        a, c = oracle.e8_nearest(x[i])
        _check_member(a, c)
        # never farther than the covering radius of E8 (= 1)
        assert ((a + 0.5 * c - x[i]) ** 2).sum() <= 1.0 + 1e-12
