"""Shared set-up for the GPU parity tests: build a paged cache from a seeded
synthetic workload through the library's own append, and run the oracle on
the same stored bits."""

from __future__ import annotations

import math

import numpy as np
import torch

from oracle import decode as odec
from oracle import pages as opg
from sparse_entmax_attention_gb300 import binding as B
from sparse_entmax_attention_gb300 import synth


class Built:
    """A filled cache plus the stored K/V/q it was filled from (on the GPU)."""

    def __init__(self, spec, seed=0, device="cuda", prefill_chunk=None, meta_bf16=False):
        self.spec = spec
        bt, total, need = synth.block_tables(spec, seed)
        maxp = bt.shape[1]
        self.cache = B.PagedCache(spec.num_kv_heads, spec.group, spec.head_dim, spec.page_size,
                                  spec.batch, maxp, total, spec.kv_dtype, device, meta_bf16=meta_bf16)
        self.cache.block_table.copy_(bt.to(device))
        self.q = torch.stack([synth.queries(spec, b, seed, device) for b in range(spec.batch)]).contiguous()
        self.K, self.V, self.draws = [], [], []
        for b in range(spec.batch):
            Ks, Vs, ds = [], [], []
            for j in range(spec.num_kv_heads):
                g = spec.group
                hd = synth.HeadDraws(spec, b, j, self.q[b, j * g:(j + 1) * g], seed, device)
                Ks.append(hd.k)
                Vs.append(hd.v)
                ds.append(hd)
            self.K.append(torch.stack(Ks))
            self.V.append(torch.stack(Vs))
            self.draws.append(ds)
            L = spec.context_lens[b]
            if L == 0:
                continue
            sid = torch.tensor([b], dtype=torch.int32, device=device)
            step = prefill_chunk or L
            for t0 in range(0, L, step):
                t1 = min(L, t0 + step)
                B.append(self.cache, self.K[b][:, t0:t1].unsqueeze(0).contiguous(),
                         self.V[b][:, t0:t1].unsqueeze(0).contiguous(), seq_ids=sid)
        torch.cuda.synchronize()

    def host_kv(self, b, j):
        """Stored keys/values of (sequence b, KV head j) as float64 numpy."""
        L = int(self.cache.seq_lens[b].item())
        return (self.K[b][j, :L].double().cpu().numpy(), self.V[b][j, :L].double().cpu().numpy())

    def host_meta(self, b, j, bf16=False):
        """The oracle's own float64 page metadata of the stored keys of
        (sequence b, KV head j); with ``bf16`` the mean and m2 are rounded to
        bfloat16 from their exact values (the oracle's reading of a cache that
        streams bf16 copies). Nothing here is read back from the GPU."""
        K, _ = self.host_kv(b, j)
        meta = opg.page_metadata(K, self.spec.page_size)
        return opg.bf16_metadata(meta) if bf16 else meta

    def host_q(self, b, j, q=None):
        q = self.q if q is None else q
        g = self.spec.group
        return q[b, j * g:(j + 1) * g].double().cpu().numpy()


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


# --------------------------------------------------------------------------
# bf16 statistics: the rounding-boundary band
# --------------------------------------------------------------------------

def bf16_stat_band(K, P, Q):
    """How far a page's (μ_p^h, σ_p^h) in score units can move between the
    oracle's reading (exact statistics rounded to bfloat16) and the GPU's
    copies (float32 statistics rounded to bfloat16).

    The GPU's float32 mean is within w = 2^-18·max_t |k_t,d| of the exact one
    (a float32 sum of at most 32 terms and one division, or their pairwise
    merges), and its m2 within w = 2^-17·Σ_t k_t,d². An element whose
    window [x − w, x + w] rounds to two different bfloat16 values may be
    stored as either; every other element is stored exactly as the oracle
    reads it. Returns (dmu, dsig) [g, n_pages]: bounds on |Δμ| and |Δσ|.
    """
    K = np.asarray(K, np.float64)
    Q = np.atleast_2d(np.asarray(Q, np.float64))
    n_tok, d = K.shape
    n_pages = -(-n_tok // P)
    Kp = np.zeros((n_pages * P, d))
    Kp[:n_tok] = K
    Kp = Kp.reshape(n_pages, P, d)
    meta = opg.page_metadata(K, P)
    n = meta["n"].astype(np.float64)[:, None]
    mean, m2 = meta["mean"], meta["var"] * n
    w_mean = 2.0 ** -18 * np.abs(Kp).max(axis=1)
    w_m2 = 2.0 ** -17 * (Kp * Kp).sum(axis=1)

    def spread(x, w):
        lo, hi, r = opg.bf16_round(x - w), opg.bf16_round(x + w), opg.bf16_round(x)
        return np.maximum(np.abs(hi - r), np.abs(lo - r))

    dmean, dm2 = spread(mean, w_mean), spread(m2, w_m2)
    dmu = np.abs(Q) @ dmean.T / math.sqrt(d)                 # [g, n_pages]
    dvar = (Q * Q) @ (dm2 / n).T / d
    bm = opg.bf16_metadata(meta)
    _, sig = zip(*[opg.gauss_page_scores(Q[h], bm["mean"], bm["var"]) for h in range(Q.shape[0])])
    s2 = np.stack(sig) ** 2
    dsig = np.sqrt(s2 + dvar) - np.sqrt(np.maximum(s2 - dvar, 0.0))
    return dmu, dsig


# --------------------------------------------------------------------------
# Selected-page parity record (printed at the end of the session)
# --------------------------------------------------------------------------

PARITY = {"checks": 0, "units": 0, "pages": 0, "flips": [], "min_margin": math.inf,
          "min_margin_at": None}


def record_unit(tag, n_pages, margins, eps):
    """Count one compared (sequence, KV head) unit and keep the smallest
    decision margin, relative to its ε_sel, seen so far."""
    PARITY["units"] += 1
    PARITY["pages"] += int(n_pages)
    if margins is not None and np.size(margins):
        m = float(np.min(np.abs(margins)))
        if m < PARITY["min_margin"]:
            PARITY["min_margin"] = m
            PARITY["min_margin_at"] = f"{tag} (ε_sel {eps:.2e})"


def record_flip(tag, page, margin, eps, band, why):
    PARITY["flips"].append(f"{tag}: page {page} margin {margin:+.3e} (ε_sel {eps:.2e}, "
                           f"bf16 band {band:.2e}; {why})")
