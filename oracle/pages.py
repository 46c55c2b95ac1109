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
from scipy.special import binom, gamma, ndtr, pbdv, roots_genlaguerre  # library primitives


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


def bf16_round(x):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits and float32's exponent range. With
    x = m·2^e (frexp, 0.5 ≤ |m| < 1) the nearest value is round(m·2^8)·2^(e−8);
    both scalings are exact in float64 and ``np.round`` rounds halves to
    even. Below the smallest normal (2^-126) the spacing stays 2^-133.
    Returned as float64 (every bfloat16 value is exact there).
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    shift = np.maximum(e - 8, -133)
    return np.ldexp(np.round(np.ldexp(x, -shift)), shift)


def bf16_metadata(meta):
    """The page statistics rounded the way a cache that streams bfloat16
    copies of them stores them.

    Reading (the summary's §4 says the cost of decoding moves to page
    selection; the copies halve the bytes the Gaussian scorer streams): the
    stored mean and the sum of squared deviations m2 = n_p·var are each
    rounded to the nearest bfloat16 (ties to even) from their exact values;
    the scorer then uses var = bf16(m2)/n_p. Bounding box and counts are
    unchanged. Returns a new dict.
    """
    out = dict(meta)
    n = np.asarray(meta["n"], np.float64)[:, None]
    out["mean"] = bf16_round(meta["mean"])
    out["var"] = bf16_round(np.asarray(meta["var"], np.float64) * n) / n
    return out


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


J_LAGUERRE_TO = -2.0   # t at or below which jfun uses Gauss–Laguerre
J_SERIES_FROM = 20.0   # t at which jfun switches to the large-t series
J_LAGUERRE_NODES = 80


def jfun(t, nu: float):
    """J_ν(t) = ∫_0^∞ y^ν φ(y − t) dy = E[(t + Z)_+^ν], Z ~ N(0, 1), ν > −1.

    Three routes, each a restatement of the same integral (about 1e-15
    relative against 40-digit quadrature):
      t ≤ −2: with x = −t, φ(y + x) = φ(x)·e^{−y²/2 − xy}, and y = s/x gives
              J = φ(x)·x^{−ν−1}·∫_0^∞ s^ν e^{−s}·e^{−s²/(2x²)} ds, a smooth
              integrand under the generalized Laguerre weight, summed with
              80-node Gauss–Laguerre;
      −2 < t < 20: J = Γ(ν+1)·e^{−t²/4}·D_{−ν−1}(−t)/√(2π), the integral
              representation of the parabolic cylinder function D;
      t ≥ 20: E[(t + Z)^ν] = t^ν Σ_k C(ν, 2k)·(2k−1)!!·t^{−2k} (the binomial
              series of (1 + Z/t)^ν under the Gaussian; the part with
              t + Z < 0 is O(φ(t))), summed while its terms fall.
    """
    t = np.asarray(t, dtype=np.float64)
    out = np.empty(t.shape)
    left = t <= J_LAGUERRE_TO
    if left.any():
        x = -t[left]
        s, w = roots_genlaguerre(J_LAGUERRE_NODES, nu)
        K = np.exp(-np.outer(1.0 / (2.0 * x * x), s * s)) @ w
        out[left] = _phi(x) * x ** (-nu - 1.0) * K
    mid = (~left) & (t < J_SERIES_FROM)
    d, _ = pbdv(-nu - 1.0, -t[mid])
    out[mid] = gamma(nu + 1.0) * np.exp(-0.25 * t[mid] * t[mid]) * d / math.sqrt(2.0 * math.pi)
    th = t[t >= J_SERIES_FROM]
    if th.size:
        acc = np.ones(th.shape)
        dfact = 1.0
        for k in range(1, 30):
            dfact *= 2 * k - 1  # (2k−1)!!
            term = binom(nu, 2 * k) * dfact / th ** (2 * k)
            acc += term
            if np.all(np.abs(term) < 1e-17 * np.abs(acc)):
                break
        out[t >= J_SERIES_FROM] = th ** nu * acc
    return out


def partial_moment(a, sig, beta: float):
    """E[(a + σ·Z)_+^β] for Z ~ N(0, 1), elementwise, β > 0.

    With t = a/σ (σ > 0), integrating (a + σz)^β·φ(z) over z > −t:
      β = 1:  a·Φ(t) + σ·φ(t)
      β = 2:  (a² + σ²)·Φ(t) + a·σ·φ(t)
      other β: σ^β·J_β(t) (``jfun``), the general entmax order of the
      Gaussian selector (α = 1 + 1/β).
    σ = 0 gives (a)_+^β.
    """
    a = np.asarray(a, dtype=np.float64)
    sig = np.asarray(sig, dtype=np.float64)
    a, sig = np.broadcast_arrays(a, sig)
    out = np.empty(a.shape)
    zero = sig <= 0.0
    out[zero] = np.maximum(a[zero], 0.0) ** beta
    nz = ~zero
    an, sn = a[nz], sig[nz]
    t = an / sn
    if beta == 1.0 or beta == 2.0:
        Phi, ph = ndtr(t), _phi(t)
        if beta == 1.0:
            out[nz] = an * Phi + sn * ph
        else:
            out[nz] = (an * an + sn * sn) * Phi + an * sn * ph
    else:
        out[nz] = sn ** beta * jfun(t, beta)
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
    one-token page gives M̂_p = μ_p. n_p is the page's count of valid
    tokens (a partly filled last page uses its own count, not the page size).
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
