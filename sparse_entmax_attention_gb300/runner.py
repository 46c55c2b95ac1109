"""Fill a paged cache from a seeded synthetic workload through the library's
own append (the prefill), and produce the per-step decode inputs."""

from __future__ import annotations

import torch

from . import binding as B
from . import synth


class Workload:
    """A cache holding a workload's prefilled context, on one device."""

    def __init__(self, spec: synth.Spec, seed: int = 0, device="cuda", extra_steps: int = 0,
                 keep_kv: bool = False, meta_bf16: bool = False):
        self.spec, self.seed, self.device = spec, seed, torch.device(device)
        steps = max(spec.steps if spec.append_per_step else 0, extra_steps)
        if steps != (spec.steps if spec.append_per_step else 0):
            spec = synth.Spec(**{**spec.__dict__, "steps": steps, "append_per_step": True})
            self.spec = spec
        bt, total, need = synth.block_tables(spec, seed)
        self.cache = B.PagedCache(spec.num_kv_heads, spec.group, spec.head_dim, spec.page_size,
                                  spec.batch, bt.shape[1], total, spec.kv_dtype, device,
                                  meta_bf16=meta_bf16)
        self.cache.block_table.copy_(bt.to(device))
        self.q = torch.stack([synth.queries(spec, b, seed, device)
                              for b in range(spec.batch)]).contiguous()
        self.draws = []
        self.kv = [] if keep_kv else None
        for b in range(spec.batch):
            row = []
            ks, vs = [], []
            for j in range(spec.num_kv_heads):
                g = spec.group
                hd = synth.HeadDraws(spec, b, j, self.q[b, j * g:(j + 1) * g], seed, device)
                ks.append(hd.k)
                vs.append(hd.v)
                row.append(hd)
            K = torch.stack(ks).unsqueeze(0).contiguous()
            V = torch.stack(vs).unsqueeze(0).contiguous()
            for hd in row:  # the cache holds the tokens now; keep only what appends need
                hd.nk = hd.k[hd.needle_pos].float()
                hd.k = hd.k[:0]
                hd.v = hd.v[:0]
            self.draws.append(row)
            if spec.context_lens[b]:
                B.append(self.cache, K, V, seq_ids=torch.tensor([b], dtype=torch.int32, device=device))
            if keep_kv:
                self.kv.append((K[0], V[0]))
            del K, V
        torch.cuda.synchronize()

    def step_tokens(self, step: int):
        """The token appended at decode step `step` (position context + step) of
        every sequence: k, v [B, Hkv, 1, d] each."""
        spec = self.spec
        lens = [L + step for L in spec.context_lens]
        ks, vs = [], []
        for b in range(spec.batch):
            kk, vv = [], []
            for j in range(spec.num_kv_heads):
                d = self.draws[b][j]
                k, v = synth.append_token(spec, b, j, lens[b], step, d.centroids, d.out_ch,
                                          d.out_off, self.seed, self.device)
                kk.append(k)
                vv.append(v)
            ks.append(torch.stack(kk))
            vs.append(torch.stack(vv))
        return (torch.stack(ks).unsqueeze(2).contiguous(), torch.stack(vs).unsqueeze(2).contiguous())

    def step_queries(self, step: int):
        """Fresh decode queries of step `step`: [B, Hq, d]."""
        spec = self.spec
        return torch.stack([synth.step_queries(spec, b, step, [d.nk for d in self.draws[b]],
                                               self.seed, self.device)
                            for b in range(spec.batch)]).contiguous()
