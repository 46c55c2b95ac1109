"""Per-page key metadata, page scores and candidate selection in float64.

Oracle; test infrastructure only. Follows "EntmaxKV: Support-Aware Decoding
for Entmax Attention", gist.science technical summary:
  §2A  the cache is split into pages; each page keeps the coordinate-wise
       minimum and maximum key (k_min, k_max) and the first and second
       moments (mean, variance) of its keys;
  §2A  the bounding box gives a deterministic upper bound on any token's
       score in the page; the moments model a page's token scores as a
       Gaussian random variable;
  §2B1 top-k selection keeps the k pages with the highest upper bounds;
  §2B2 the Gaussian-aware selector solves an approximate normalisation
       equation for τ̂ from the page statistics and keeps the pages whose
       estimated maximum score clears τ̂ lowered by a safety margin Δ.

Readings taken where the pages are silent (each is restated where used):
  * scores are s = q·k/√d, so every page quantity is in score units
    (U_p and μ_p divide by √d, σ_p² by d);
  * "variance" is the per-coordinate population variance (divide by n_p);
  * the page score model is diagonal: σ_p² = Σ_d q_d² var_{p,d} / d;
  * the normalisation equation is the expectation of the entmax normaliser
    under the page model: F(τ) = Σ_p n_p · E[(Z_p − τ)_+^β] = 1 with
    Z_p ~ N(m_p, ς_p²), m_p = (α−1)μ_p, ς_p = (α−1)σ_p;
  * a page's estimated maximum score is M̂_p = μ_p + σ_p·sqrt(2 ln n_p);
  * a page is kept when M̂_p ≥ τ̂/(α−1) − Δ, with Δ in score units; under
    grouped-query attention a KV head keeps the union over its query heads;
  * top-k ranks a KV head's pages by max over its query heads of U_p,
    ties going to the lower logical page index.
"""

from __future__ import annotations

import math

import numpy as np
from scipy.special import ndtr  # standard normal CDF Φ, a library primitive


# --------------------------------------------------------------------------
# Metadata (§2A)
# --------------------------------------------------------------------------

def page_metadata(keys, page_size: int):
    """Metadata of every page of one (sequence, KV head) from its stored keys.

    keys: [n_tokens, d] (any float dtype; converted exactly to float64).
    Returns dict with kmin, kmax, mean, var ([n_pages, d]) and n ([n_pages]),
    all from the valid tokens only (a partial last page counts only the
    tokens it holds). var is the two-pass population variance.
    """
    k = np.asarray(keys, dtype=np.float64)
    n_tok, d = k.shape
    n_pages = -(-n_tok // page_size)
    kmin = np.empty((n_pages, d))
    kmax = np.empty((n_pages, d))
    mean = np.empty((n_pages, d))
    var = np.empty((n_pages, d))
    n = np.empty(n_pages, dtype=np.int64)
    for p in range(n_pages):
        blk = k[p * page_size: min(n_tok, (p + 1) * page_size)]
        n[p] = blk.shape[0]
        kmin[p] = blk.min(axis=0)
        kmax[p] = blk.max(axis=0)
        mean[p] = blk.sum(axis=0) / n[p]
        var[p] = ((blk - mean[p]) ** 2).sum(axis=0) / n[p]
    return {"kmin": kmin, "kmax": kmax, "mean": mean, "var": var, "n": n}


def welford_append(n: int, mean, m2, x):
    """One-token update of (count, mean, sum of squared deviations).

    Welford's recurrence: n' = n + 1, δ = x − mean, mean' = mean + δ/n',
    M2' = M2 + δ·(x − mean'). Used to model appending one token to a page.
    """
    x = np.asarray(x, dtype=np.float64)
    n1 = n + 1
    delta = x - mean
    mean1 = mean + delta / n1
    return n1, mean1, m2 + delta * (x - mean1)


def chan_merge(na: int, mean_a, m2_a, nb: int, mean_b, m2_b):
    """Merge two disjoint groups' (count, mean, M2) (Chan, Golub & LeVeque).

    n = na + nb, δ = mean_b − mean_a, mean = mean_a + δ·nb/n,
    M2 = M2_a + M2_b + δ²·na·nb/n. Used to model appending a block of tokens
    to a partly filled page.
    """
    n = na + nb
    if na == 0:
        return nb, np.array(mean_b, dtype=np.float64), np.array(m2_b, dtype=np.float64)
    delta = np.asarray(mean_b, np.float64) - np.asarray(mean_a, np.float64)
    mean = mean_a + delta * (nb / n)
    m2 = m2_a + m2_b + delta * delta * (na * nb / n)
    return n, mean, m2


# --------------------------------------------------------------------------
# Page scores (§2A)
# --------------------------------------------------------------------------

def bbox_bound(q, kmin, kmax):
    """Bounding-box bound U_p = Σ_d max(q_d·kmin_{p,d}, q_d·kmax_{p,d}) / √d.

    For every token k in page p, q·k/√d ≤ U_p because each coordinate of k
    lies in [kmin_d, kmax_d] and q_d·x is maximised at an end of that range.
    q: [d]; kmin, kmax: [n_pages, d]. Returns [n_pages].
    """
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[0]
    lo = np.asarray(kmin, np.float64) * q
    hi = np.asarray(kmax, np.float64) * q
    return np.maximum(lo, hi).sum(axis=1) / math.sqrt(d)


def gauss_page_scores(q, mean, var):
    """Gaussian page-score model (μ_p, σ_p) in score units.

    A token score s = q·k/√d with k drawn from a page whose coordinates have
    the page's mean and (independent) variance has mean μ_p = q·mean_p/√d and
    variance σ_p² = Σ_d q_d²·var_{p,d} / d.
    """
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[0]
    mu = np.asarray(mean, np.float64) @ q / math.sqrt(d)
    sig2 = np.asarray(var, np.float64) @ (q * q) / d
    return mu, np.sqrt(np.maximum(sig2, 0.0))


def _phi(t):
    return np.exp(-0.5 * t * t) / math.sqrt(2.0 * math.pi)


def partial_moment(a, sig, beta: float):
    """E[(a + σ·Z)_+^β] for Z ~ N(0, 1), elementwise, β ∈ {1, 2}.

    With t = a/σ (σ > 0):
      β = 1:  a·Φ(t) + σ·φ(t)
      β = 2:  (a² + σ²)·Φ(t) + a·σ·φ(t)
    (integrate (a + σz)^β·φ(z) over z > −t). σ = 0 gives (a)_+^β.
    """
    a = np.asarray(a, dtype=np.float64)
    sig = np.asarray(sig, dtype=np.float64)
    a, sig = np.broadcast_arrays(a, sig)
    out = np.empty(a.shape)
    zero = sig <= 0.0
    if beta == 1.0:
        out[zero] = np.maximum(a[zero], 0.0)
    elif beta == 2.0:
        out[zero] = np.maximum(a[zero], 0.0) ** 2
    else:
        raise NotImplementedError("closed-form partial moments cover β ∈ {1, 2}")
    nz = ~zero
    an, sn = a[nz], sig[nz]
    t = an / sn
    Phi, ph = ndtr(t), _phi(t)
    if beta == 1.0:
        out[nz] = an * Phi + sn * ph
    else:
        out[nz] = (an * an + sn * sn) * Phi + an * sn * ph
    return out


def normaliser(tau: float, m, sig, n, beta: float) -> float:
    """F(τ) = Σ_p n_p·E[(Z_p − τ)_+^β], Z_p ~ N(m_p, ς_p²) (z scale)."""
    return float(np.sum(np.asarray(n, np.float64) *
                        partial_moment(np.asarray(m) - tau, sig, beta)))


def tauhat(m, sig, n, alpha: float, iters: int = 200) -> float:
    """τ̂ solving F(τ̂) = 1 by float64 bisection (§2B2 normalisation solve).

    m, sig: page model on the z scale ((α−1)μ_p, (α−1)σ_p); n: tokens per
    page. F is strictly decreasing. Lower bracket max_p m_p − 1: by Jensen
    E[(Z−τ)_+^β] ≥ (m−τ)_+^β, so the page with the largest m_p alone gives
    F ≥ 1 there. The upper bracket is found by doubling the step until F < 1.
    """
    beta = 1.0 / (alpha - 1.0)
    m = np.asarray(m, np.float64)
    lo = float(m.max()) - 1.0
    step = 1.0
    hi = lo + step
    while normaliser(hi, m, sig, n, beta) >= 1.0:
        lo = hi
        step *= 2.0
        hi = lo + step
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if normaliser(mid, m, sig, n, beta) >= 1.0:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def est_max(mu, sigma, n):
    """Estimated maximum score of a page: M̂_p = μ_p + σ_p·sqrt(2 ln n_p).

    The textbook leading term for the maximum of n Gaussian draws; a
    one-token page gives M̂_p = μ_p.
    """
    n = np.asarray(n, dtype=np.float64)
    return np.asarray(mu) + np.asarray(sigma) * np.sqrt(2.0 * np.log(n))


# --------------------------------------------------------------------------
# Selection (§2B)
# --------------------------------------------------------------------------

def select_topk(uhat, k: int):
    """The k pages with the largest keys, ties to the lower page index.

    uhat: [n_pages] page keys. Returns the chosen logical page indices,
    sorted ascending. k ≥ n_pages keeps every page.
    """
    uhat = np.asarray(uhat, np.float64)
    order = sorted(range(uhat.size), key=lambda p: (-uhat[p], p))
    return np.array(sorted(order[:k]), dtype=np.int64)


def select_gaussian(mhat_per_head, thr_per_head):
    """Pages whose estimated maximum clears the threshold for any head.

    mhat_per_head: [g, n_pages] M̂_p^h (score units);
    thr_per_head:  [g] τ̂_h/(α−1) − Δ. Equality selects.
    Returns ascending logical page indices (union over the g heads).
    """
    mh = np.asarray(mhat_per_head, np.float64)
    thr = np.asarray(thr_per_head, np.float64)[:, None]
    keep = np.any(mh >= thr, axis=0)
    return np.nonzero(keep)[0].astype(np.int64)
