"""α-entmax and softmax in float64 (oracle; test infrastructure only).

Definition followed. The EntmaxKV summary (gist.science, §2 "Methodology")
states that α-entmax with α > 1 gives probability vectors with exact zeros.
The formula itself is the standard one from "Sparse Sequence-to-Sequence
Models" (Peters, Niculae & Martins, 2019) and, for α = 2, "From Softmax to
Sparsemax" (Martins & Astudillo, 2016), both listed among the works EntmaxKV
builds on (mlsanity.com index page, "Builds on"):

    z_i = (α − 1)·s_i,   β = 1/(α − 1),
    p_i = [z_i − τ]_+^β,  with τ the unique number making Σ_i p_i = 1.

τ is reported on the z scale. f(τ) = Σ_i [z_i − τ]_+^β is continuous and
strictly decreasing on (−∞, max z], with f(max z − 1) ≥ 1 and f(max z) = 0,
so τ ∈ [max z − 1, max z) and is unique.
"""

from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    a = np.asarray(x, dtype=np.float64)
    if a.ndim != 1 or a.size == 0:
        raise ValueError("expected a non-empty 1-D score vector")
    return a


def threshold_bisect(z, alpha: float, iters: int = 200) -> float:
    """τ solving Σ_i [z_i − τ]_+^β = 1 by bisection on [max z − 1, max z].

    Valid for every α > 1 (z already on the (α − 1)·s scale).
    """
    if not alpha > 1.0:
        raise ValueError("α-entmax needs α > 1")
    z = _f64(z)
    beta = 1.0 / (alpha - 1.0)
    zmax = float(z.max())
    lo, hi = zmax - 1.0, zmax
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        f = float(np.sum(np.clip(z - mid, 0.0, None) ** beta))
        if f >= 1.0:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def threshold_sparsemax(z) -> float:
    """Exact τ for α = 2 (β = 1): the sparsemax closed form.

    Sort z descending as z_(1) ≥ … ≥ z_(n). With c_k = Σ_{j≤k} z_(j), the
    support size is the largest k with z_(k) > (c_k − 1)/k, and then
    τ = (c_k − 1)/k (Martins & Astudillo 2016, "From Softmax to Sparsemax").
    """
    z = np.sort(_f64(z))[::-1]
    c = np.cumsum(z)
    k = np.arange(1, z.size + 1, dtype=np.float64)
    tau_k = (c - 1.0) / k
    ok = z > tau_k
    kstar = int(np.nonzero(ok)[0].max()) + 1
    return float(tau_k[kstar - 1])


def threshold_entmax15(z) -> float:
    """Exact τ for α = 1.5 (β = 2): the sort-based algorithm of Peters et al.

    Sort z descending. For the top-k prefix let m_k be its mean and v_k its
    population variance. If the support were exactly that prefix, τ would
    solve k·τ² − 2τ·Σz + Σz² = 1 on the branch τ ≤ min of the prefix, giving
    τ_k = m_k − sqrt(1/k − v_k) (defined when 1/k ≥ v_k). The support size is
    the largest k with τ_k defined and τ_k ≤ z_(k) ("Sparse Sequence-to-
    Sequence Models", Peters, Niculae & Martins 2019, exact 1.5-entmax).
    """
    z = np.sort(_f64(z))[::-1]
    n = z.size
    k = np.arange(1, n + 1, dtype=np.float64)
    mean = np.cumsum(z) / k
    meansq = np.cumsum(z * z) / k
    var = meansq - mean * mean
    disc = 1.0 / k - var
    best = None
    for i in range(n):
        if disc[i] < 0.0:
            continue
        tau_i = mean[i] - np.sqrt(disc[i])
        if tau_i <= z[i]:
            best = tau_i
    assert best is not None  # k = 1 always qualifies: τ_1 = z_(1) − 1
    return float(best)


def threshold(z, alpha: float) -> float:
    """Exact α-entmax threshold on the z scale.

    α = 2 and α = 1.5 use their sort-based exact algorithms; every other
    α > 1 uses float64 bisection run to machine precision.
    """
    if alpha == 2.0:
        return threshold_sparsemax(z)
    if alpha == 1.5:
        return threshold_entmax15(z)
    return threshold_bisect(z, alpha)


def entmax(s, alpha: float):
    """α-entmax of raw scores s. Returns (p, τ) with τ on the z scale."""
    s = _f64(s)
    z = (alpha - 1.0) * s
    tau = threshold(z, alpha)
    beta = 1.0 / (alpha - 1.0)
    p = np.clip(z - tau, 0.0, None) ** beta
    return p, tau


def softmax(s):
    """Softmax of raw scores s. Returns (p, lse) with lse = log Σ exp(s)."""
    s = _f64(s)
    m = float(s.max())
    e = np.exp(s - m)
    tot = float(e.sum())
    return e / tot, m + float(np.log(tot))
