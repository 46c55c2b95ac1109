"""Pins for oracle.entmax: hand cases, brute force, limits and invariants.

None of these re-type the oracle's formula: the hand cases are derived by
hand (tests/golden), brute force enumerates every support and checks the
optimality conditions directly, and the rest are properties the definition
implies.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import entmax as em

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _ev(x):
    return float(eval(x, {"math": math}))


def test_hand_cases():
    cases = json.load(open(os.path.join(GOLD, "entmax_hand_cases.json")))["cases"]
    for c in cases:
        p, tau = em.entmax(c["s"], c["alpha"])
        np.testing.assert_allclose(p, [_ev(x) for x in c["p"]], rtol=0, atol=1e-12, err_msg=c["why"])
        assert abs(tau - _ev(c["tau"])) < 1e-12, c["why"]


def _brute_force_tau(z, alpha):
    """Enumerate supports; keep the one meeting the optimality conditions.

    For a support S the threshold solves Σ_S (z_i − τ)^β = 1 with τ ≤ min_S z
    (found by bisection on that branch, independent of the oracle's solvers).
    S is optimal iff every i ∉ S has z_i ≤ τ.
    """
    n = len(z)
    beta = 1.0 / (alpha - 1.0)
    found = []
    for r in range(1, n + 1):
        for S in itertools.combinations(range(n), r):
            zs = np.array([z[i] for i in S])
            lo_z = zs.min()
            if np.sum((zs - lo_z) ** beta) > 1.0:
                continue  # root would lie above min_S z: not a valid support
            lo, hi = lo_z - 2.0, lo_z
            while np.sum((zs - lo) ** beta) < 1.0:
                lo -= 2.0
            for _ in range(300):
                mid = 0.5 * (lo + hi)
                if np.sum((zs - mid) ** beta) >= 1.0:
                    lo = mid
                else:
                    hi = mid
            tau = 0.5 * (lo + hi)
            if all(z[i] <= tau + 1e-13 for i in range(n) if i not in S):
                found.append(tau)
    assert found
    # several supports can qualify only when some z_i equals τ; they share τ
    assert max(found) - min(found) < 1e-9
    return found[0]


@pytest.mark.parametrize("alpha", [1.5, 2.0, 1.25, 3.0])
def test_brute_force_small(alpha):
    rng = np.random.default_rng(1)
    for n in (1, 2, 3, 5, 8, 12):
        for _ in range(4 if n == 12 else 20):
            s = rng.normal(size=n) * rng.choice([0.3, 1.0, 4.0])
            z = (alpha - 1.0) * s
            tau_bf = _brute_force_tau(list(z), alpha)
            _, tau = em.entmax(s, alpha)
            assert abs(tau - tau_bf) < 1e-9, (n, alpha, s)


@pytest.mark.parametrize("alpha", [1.5, 2.0])
def test_sort_based_equals_bisection(alpha):
    rng = np.random.default_rng(2)
    for n in (1, 7, 100, 5000):
        s = rng.normal(size=n) * 3.0
        z = (alpha - 1.0) * s
        exact = em.threshold(z, alpha)
        bis = em.threshold_bisect(z, alpha)
        assert abs(exact - bis) < 1e-12


@pytest.mark.parametrize("alpha", [1.5, 2.0, 1.1, 2.5])
def test_simplex_and_exact_zeros(alpha):
    rng = np.random.default_rng(3)
    s = rng.normal(size=400) * 2.0
    p, tau = em.entmax(s, alpha)
    z = (alpha - 1.0) * s
    assert abs(p.sum() - 1.0) < 1e-12
    assert np.all(p >= 0.0)
    assert np.all((p == 0.0) == (z <= tau))
    assert (p == 0.0).any()  # exact zeros (α > 1)


@pytest.mark.parametrize("alpha", [1.5, 2.0, 1.3])
def test_shift_and_permutation(alpha):
    rng = np.random.default_rng(4)
    s = rng.normal(size=50)
    p, tau = em.entmax(s, alpha)
    p2, tau2 = em.entmax(s + 3.7, alpha)
    np.testing.assert_allclose(p2, p, atol=1e-12)
    assert abs(tau2 - (tau + (alpha - 1.0) * 3.7)) < 1e-12
    perm = rng.permutation(50)
    p3, tau3 = em.entmax(s[perm], alpha)
    np.testing.assert_allclose(p3, p[perm], atol=1e-12)
    assert abs(tau3 - tau) < 1e-12


def test_equal_scores():
    for alpha in (1.5, 2.0, 1.2, 4.0):
        for n in (1, 3, 64):
            c = 0.7
            p, tau = em.entmax(np.full(n, c), alpha)
            np.testing.assert_allclose(p, 1.0 / n, atol=1e-12)
            assert abs(tau - ((alpha - 1.0) * c - n ** (1.0 - alpha))) < 1e-12


def test_alpha_to_one_is_softmax():
    rng = np.random.default_rng(5)
    s = rng.uniform(-2.0, 2.0, size=30)
    p, _ = em.entmax(s, 1.001)
    q, _ = em.softmax(s)
    np.testing.assert_allclose(p, q, atol=1e-2)


def test_softmax_dense_and_lse():
    s = np.array([0.0, math.log(3.0)])
    p, lse = em.softmax(s)
    np.testing.assert_allclose(p, [0.25, 0.75], atol=1e-15)
    assert abs(lse - math.log(4.0)) < 1e-15
