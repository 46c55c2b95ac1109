"""One EntmaxKV decode step for one (sequence, KV head), float64.

Oracle; test infrastructure only. Follows "EntmaxKV: Support-Aware Decoding
for Entmax Attention", gist.science technical summary:
  §2A/§2B  page scoring and candidate selection (see ``oracle.pages``);
  §2C      α-entmax over the tokens of the selected pages only; if they
           contain the full-cache support the output is exact;
  §3       δ is the full-cache probability mass of the dropped tokens and
           ‖o − õ‖ ≤ 2Bδ with B a bound on ‖v_i‖; S ⊆ I_keep gives δ = 0;
  §4       the full-cache entmax and full-cache softmax decodes are the
           baselines the method is compared against.

Plain definition of the result, for each query head h of the group and
kept token set I (all tokens of the selected pages):
  s_i = q_h·k_i/√d,  (p̃, τ) = entmax_α(s restricted to I),  o = Σ_{i∈I} p̃_i v_i.

The returned δ depends on the policy (a reading; the pages only use δ in the
analysis of §3):
  full      δ = 0 (nothing is dropped);
  topk      certified bound δ̄ = min(1, Σ_{dropped pages} n_p·[(α−1)U_p^h − τ̃]_+^β),
            valid because the kept-set threshold τ̃ ≤ the full-cache τ and
            every token of page p scores ≤ U_p^h;
  gaussian  the page model's estimate Σ_{dropped pages} n_p·E[(Z_p − τ̂)_+^β];
  softmax   δ = 0 and the "τ" slot carries log Σ_i exp(s_i).
  softmax_topk  softmax over the top-k kept set (the comparison the summary's
            §1/§4 draw against softmax attention); "τ" carries log Σ_{i∈I} exp(s_i)
            and δ is the certified bound D/(1 + D), D = Σ_{dropped pages}
            n_p·exp(U_p^h − lse_kept): with A = Σ_I e^{s} and B = Σ_{i∉I} e^{s}
            ≤ B̄ = Σ_dropped n_p e^{U_p}, δ = B/(A + B) ≤ B̄/(A + B̄) since it grows in B.
The exact δ = Σ_{i∉I} p_i^full (the full-cache weights of the same kind of
attention) is always returned as ``delta_exact``.
"""

from __future__ import annotations

import math

import numpy as np

from . import entmax as em
from . import pages as pg

POLICIES = ("full", "topk", "gaussian", "softmax", "softmax_topk")


def _beta(alpha):
    return 1.0 / (alpha - 1.0)


def attend_pages(K, V, Q, alpha: float, page_size: int, page_ids, softmax: bool = False):
    """α-entmax attention of the g query heads over the tokens of the given
    pages only (§2C), or softmax attention over them with ``softmax`` (then the
    τ slot is log Σ exp(s_i) over those tokens). Returns (out [g, d], tau [g]);
    an empty page set gives a zero output and τ = NaN."""
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    Q = np.atleast_2d(np.asarray(Q, np.float64))
    g, d = Q.shape
    n_tok = K.shape[0]
    keep = np.zeros(n_tok, dtype=bool)
    for p in np.asarray(page_ids, dtype=np.int64):
        keep[p * page_size: min(n_tok, (p + 1) * page_size)] = True
    idx = np.nonzero(keep)[0]
    out = np.zeros((g, d))
    tau = np.full(g, np.nan)
    if idx.size == 0:
        return out, tau
    s = K[idx] @ Q.T / math.sqrt(d)
    for h in range(g):
        p, tau[h] = em.softmax(s[:, h]) if softmax else em.entmax(s[:, h], alpha)
        out[h] = p @ V[idx]
    return out, tau


def decode_group(K, V, Q, alpha: float, policy: str, page_size: int,
                 budget_tokens: int = 0, margin: float = 0.0, meta=None,
                 diagnostics: bool = True):
    """Decode the g query heads that share one KV head.

    K, V: [n_tokens, d] stored keys/values (converted exactly to float64);
    Q: [g, d] stored queries. budget_tokens: top-k budget in tokens (k =
    budget // page_size pages) or, for the Gaussian policy, a cap in tokens
    (0 = no cap). margin: Δ in score units (Gaussian policy). meta: page
    metadata of K already built by ``pages.page_metadata`` (else built here).
    diagnostics=False skips the full-cache quantities (delta_exact, recall),
    which need the full-cache entmax.

    Returns a dict:
      out [g, d], tau [g], page_ids (ascending logical ids), delta [g],
      delta_kind, delta_exact [g], recall [g], capacity_flag, and the
      intermediates U [g, P], uhat [P], mu, sigma [g, P], tauhat [g],
      mhat [g, P], meta (page metadata).
    """
    if policy not in POLICIES:
        raise ValueError(policy)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    Q = np.atleast_2d(np.asarray(Q, np.float64))
    g, d = Q.shape
    n_tok = K.shape[0]
    P = page_size
    res = {"capacity_flag": False}
    if n_tok == 0:
        res.update(out=np.zeros((g, d)), tau=np.full(g, np.nan),
                   page_ids=np.zeros(0, np.int64), delta=np.zeros(g),
                   delta_kind=policy, delta_exact=np.zeros(g),
                   recall=np.ones(g))
        return res
    if meta is None:
        meta = pg.page_metadata(K, P)
    n_pages = meta["n"].size
    res["meta"] = meta

    # ---- selection -------------------------------------------------------
    if policy in ("full", "softmax"):
        sel = np.arange(n_pages, dtype=np.int64)
    elif policy in ("topk", "softmax_topk"):
        k = budget_tokens // P
        if k <= 0:
            raise ValueError("top-k needs budget_tokens >= page_size")
        U = np.stack([pg.bbox_bound(Q[h], meta["kmin"], meta["kmax"]) for h in range(g)])
        uhat = U.max(axis=0)
        sel = pg.select_topk(uhat, k)
        res["U"], res["uhat"] = U, uhat
    else:  # gaussian
        mu = np.empty((g, n_pages))
        sigma = np.empty((g, n_pages))
        for h in range(g):
            mu[h], sigma[h] = pg.gauss_page_scores(Q[h], meta["mean"], meta["var"])
        a1 = alpha - 1.0
        th = np.array([pg.tauhat(a1 * mu[h], a1 * sigma[h], meta["n"], alpha)
                       for h in range(g)])
        mhat = np.stack([pg.est_max(mu[h], sigma[h], meta["n"]) for h in range(g)])
        thr = th / a1 - margin
        sel = pg.select_gaussian(mhat, thr)
        cap = budget_tokens // P if budget_tokens > 0 else 0
        if cap > 0 and sel.size > cap:
            # Reading: on overflow keep the cap pages with the largest margin
            # max_h (M̂_p^h − threshold_h), ties to the lower page index.
            key = (mhat - thr[:, None]).max(axis=0)
            sel = pg.select_topk(np.where(np.isin(np.arange(n_pages), sel), key, -np.inf), cap)
            res["capacity_flag"] = True
        res.update(mu=mu, sigma=sigma, tauhat=th, mhat=mhat, thr=thr)

    res["page_ids"] = sel
    keep = np.zeros(n_tok, dtype=bool)
    for p in sel:
        keep[p * P: min(n_tok, (p + 1) * P)] = True
    idx = np.nonzero(keep)[0]

    # ---- attention over the kept set --------------------------------------
    scores = (K @ Q.T / math.sqrt(d)) if (diagnostics or policy == "softmax") else None
    soft = policy in ("softmax", "softmax_topk")
    out = np.zeros((g, d))
    tau = np.full(g, np.nan)
    delta = np.zeros(g)
    delta_exact = np.zeros(g)
    recall = np.ones(g)
    beta = _beta(alpha) if not soft else None
    s_kept = K[idx] @ Q.T / math.sqrt(d) if scores is None else scores[idx]
    for h in range(g):
        if policy == "softmax":
            p, lse = em.softmax(scores[:, h])
            out[h] = p @ V
            tau[h] = lse
            continue
        if diagnostics:
            p_full, tau_full = em.softmax(scores[:, h]) if soft else em.entmax(scores[:, h], alpha)
            supp = p_full > 0
            delta_exact[h] = float(p_full[~keep].sum())
            recall[h] = float((supp & keep).sum()) / float(supp.sum())
        if idx.size == 0:
            # Nothing kept: zero output, undefined threshold, all mass dropped.
            delta[h] = 1.0
            continue
        p_k, tau_k = em.softmax(s_kept[:, h]) if soft else em.entmax(s_kept[:, h], alpha)
        out[h] = p_k @ V[idx]
        tau[h] = tau_k
        dropped = np.setdiff1d(np.arange(n_pages), sel)
        if policy == "softmax_topk":
            D = float(np.sum(meta["n"][dropped] * np.exp(res["U"][h, dropped] - tau_k)))
            delta[h] = D / (1.0 + D)
        if policy == "topk":
            zb = (alpha - 1.0) * res["U"][h, dropped] - tau_k
            delta[h] = min(1.0, float(np.sum(meta["n"][dropped] * np.clip(zb, 0.0, None) ** beta)))
        elif policy == "gaussian":
            a1 = alpha - 1.0
            delta[h] = float(np.sum(meta["n"][dropped] * pg.partial_moment(
                a1 * res["mu"][h, dropped] - res["tauhat"][h],
                a1 * res["sigma"][h, dropped], beta)))
    res.update(out=out, tau=tau, delta=delta, delta_kind=policy,
               delta_exact=delta_exact, recall=recall)
    return res


def decode_sequence(K, V, Q, alpha, policy, page_size, budget_tokens=0, margin=0.0):
    """Decode every query head of one sequence.

    K, V: [Hkv, n_tokens, d]; Q: [Hq, d] with Hq = g·Hkv and query head h
    reading KV head h // g. Returns per-KV-head result dicts.
    """
    K = np.asarray(K)
    Hkv = K.shape[0]
    Q = np.asarray(Q)
    g = Q.shape[0] // Hkv
    return [decode_group(K[j], V[j], Q[j * g:(j + 1) * g], alpha, policy,
                         page_size, budget_tokens, margin) for j in range(Hkv)]
