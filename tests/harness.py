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

    def host_meta(self, b, j):
        """Page metadata of (sequence b, KV head j) as the Gaussian scorer reads
        it: the oracle's float64 metadata of the stored keys, with the mean and
        variance replaced by the stored bf16 copies when the cache keeps them
        (None otherwise: the oracle then builds its own)."""
        c = self.cache
        if c.mean_bf16 is None:
            return None
        K, _ = self.host_kv(b, j)
        meta = opg.page_metadata(K, self.spec.page_size)
        phys = c.block_table[b, : len(meta["n"])].long()
        meta["mean"] = c.mean_bf16[phys, j].double().cpu().numpy()
        meta["var"] = c.m2_bf16[phys, j].double().cpu().numpy() / meta["n"][:, None]
        return meta

    def host_q(self, b, j, q=None):
        q = self.q if q is None else q
        g = self.spec.group
        return q[b, j * g:(j + 1) * g].double().cpu().numpy()


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def near_tie_topk(uhat, k, eps_rel=1e-5):
    """Pages whose key sits within eps of the k-th key (a flip there is a near tie)."""
    u = np.asarray(uhat, np.float64)
    if k >= u.size:
        return set()
    kth = np.sort(u)[::-1][k - 1]
    eps = eps_rel * max(1.0, abs(kth))
    return set(np.nonzero(np.abs(u - kth) <= eps)[0].tolist())


def near_tie_gauss(mhat, thr, eps):
    """Pages whose decision M̂ ≥ threshold is within eps for some head."""
    mh = np.asarray(mhat)
    t = np.asarray(thr)[:, None]
    return set(np.nonzero((np.abs(mh - t) <= eps).any(axis=0))[0].tolist())
