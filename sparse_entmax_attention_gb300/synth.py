"""Seeded synthetic decode workloads (inputs only; none of the method's math).

Both the CUDA path and the float64 oracle are fed from here, so both see the
same stored bits. Nothing in this module scores, selects or normalises:
it only draws random numbers and plants needle keys.

Recipe (per sequence b and KV head j, each from its own seeded stream):
  * page centroids c_p ~ N(0, 0.5·I), one per logical page (including the
    pages that later appended tokens will fall into);
  * keys k_t = c_{t // P} + N(0, I); values v_t ~ N(0, I);
  * queries q ~ N(0, I), one per query head;
  * needles: ``n_needles`` distinct random positions per KV head; needle i
    belongs to query head i mod g of the group and its key is
    3·u/‖u‖·√d + N(0, 0.1·I), u that head's stored query;
  * outlier channels: ``n_outliers`` distinct channels per KV head, each
    with a constant offset ~ N(0, 4) added to every key of that head;
  * keys, values and queries are rounded once to the stored dtype.
Multi-step workloads draw one fresh query per step (optionally rotated a
fraction of the angle toward a random needle key) and, when they append,
one new token per sequence per step from the same page-centroid model.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

_MASK64 = (1 << 64) - 1


def _mix(*parts: int) -> int:
    """splitmix64 over the parts: a stable 63-bit seed for a torch.Generator."""
    x = 0x9E3779B97F4A7C15
    for p in parts:
        x = (x + (int(p) & _MASK64) + 0x9E3779B97F4A7C15) & _MASK64
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        x = z ^ (z >> 31)
    return x & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_mix(*parts))
    return g


_Q, _KV, _STEPQ, _APPEND, _TABLE, _LENS, _REPEAT = 1, 2, 3, 4, 5, 6, 7


@dataclass
class Spec:
    """Shape and recipe of one synthetic decode workload."""
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    context_lens: list
    kv_dtype: torch.dtype
    alpha: float = 1.5
    n_needles: int = 0
    n_outliers: int = 0
    steps: int = 1
    rotate: float = 0.0           # fraction of the angle toward a needle key
    append_per_step: bool = False
    shuffled_table: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.context_lens)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def _loguniform_lens(seed, n, lo, hi):
    g = _gen("cpu", seed, _LENS)
    u = torch.rand(n, generator=g, dtype=torch.float64)
    return [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]


def workload(name: str, seed: int = 0) -> Spec:
    """The named synthetic workloads (sizes in the name)."""
    bf16, f32 = torch.bfloat16, torch.float32
    if name == "single-head-d64-4k-p16-fp32":
        return Spec(name, 1, 1, 64, 16, [4096], f32, 1.5, n_needles=8,
                    extra={"topk_pages": 32})
    if name == "gqa32x8-d128-32k-p16-bf16":
        return Spec(name, 32, 8, 128, 16, [32768], bf16, 1.5, n_needles=16,
                    n_outliers=4, extra={"budget_tokens": 1024})
    if name == "gqa32x8-d128-128k-p32-bf16":
        return Spec(name, 32, 8, 128, 32, [131072], bf16, 1.5, n_needles=16,
                    n_outliers=4, steps=64, rotate=0.3,
                    extra={"alphas": [1.5, 2.0], "margins": [0.0, 0.5, 1.0]})
    if name == "gqa32x8-d128-1m-p32-bf16":
        return Spec(name, 32, 8, 128, 32, [1 << 20], bf16, 1.5, n_needles=64,
                    n_outliers=4, extra={"margin": 0.5, "budget_tokens": 2048})
    if name == "batch16-loguniform-4k-256k-p16-bf16":
        lens = _loguniform_lens(seed, 16, 4096, 262144)
        return Spec(name, 32, 8, 128, 16, lens, bf16, 1.5, n_needles=16,
                    n_outliers=4, steps=128, append_per_step=True,
                    shuffled_table=True, extra={"margin": 0.5})
    raise KeyError(name)


WORKLOAD_NAMES = (
    "single-head-d64-4k-p16-fp32",
    "gqa32x8-d128-32k-p16-bf16",
    "gqa32x8-d128-128k-p32-bf16",
    "gqa32x8-d128-1m-p32-bf16",
    "batch16-loguniform-4k-256k-p16-bf16",
)


def custom(num_q_heads, num_kv_heads, head_dim, page_size, context_lens,
           kv_dtype=torch.bfloat16, alpha=1.5, n_needles=0, n_outliers=0,
           shuffled_table=False, steps=1, append_per_step=False, name="custom") -> Spec:
    """An ad-hoc workload (small parity cases, ragged tails, edge cases)."""
    return Spec(name, num_q_heads, num_kv_heads, head_dim, page_size,
                list(context_lens), kv_dtype, alpha, n_needles=n_needles,
                n_outliers=n_outliers, shuffled_table=shuffled_table,
                steps=steps, append_per_step=append_per_step)


# --------------------------------------------------------------------------
# Draws
# --------------------------------------------------------------------------

def reserved_tokens(spec: Spec, b: int) -> int:
    """Tokens the sequence will hold after all appended steps."""
    return spec.context_lens[b] + (spec.steps if spec.append_per_step else 0)


def queries(spec: Spec, b: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Decode queries of sequence b: [Hq, d] in the stored dtype."""
    g = _gen(device, seed, _Q, b)
    q = torch.randn(spec.num_q_heads, spec.head_dim, generator=g, device=device)
    return q.to(spec.kv_dtype)


class HeadDraws:
    """Everything drawn for one (sequence, KV head); keys/values stored dtype."""

    def __init__(self, spec: Spec, b: int, j: int, q_group: torch.Tensor,
                 seed: int = 0, device="cpu"):
        d, P = spec.head_dim, spec.page_size
        L = spec.context_lens[b]
        total = reserved_tokens(spec, b)
        n_pages_total = -(-max(total, 1) // P)
        g = _gen(device, seed, _KV, b, j)
        self.centroids = torch.randn(n_pages_total, d, generator=g, device=device) * math.sqrt(0.5)
        noise = torch.randn(L, d, generator=g, device=device)
        vals = torch.randn(L, d, generator=g, device=device)
        if spec.n_outliers:
            self.out_ch = torch.randperm(d, generator=g, device=device)[: spec.n_outliers]
            self.out_off = torch.randn(spec.n_outliers, generator=g, device=device) * 2.0
        else:
            self.out_ch = torch.zeros(0, dtype=torch.long, device=device)
            self.out_off = torch.zeros(0, device=device)
        keys = noise
        keys += self.centroids[torch.arange(L, device=device) // P] if L else 0.0
        n_nd = min(spec.n_needles, L)
        if n_nd:
            pos = torch.randperm(L, generator=g, device=device)[:n_nd]
            nz = torch.randn(n_nd, d, generator=g, device=device) * math.sqrt(0.1)
            grp = q_group.float()
            owner = torch.arange(n_nd, device=device) % grp.shape[0]
            u = grp[owner]
            u = u / u.norm(dim=1, keepdim=True).clamp_min(1e-30)
            keys[pos] = 3.0 * u * math.sqrt(d) + nz
            self.needle_pos = pos
            self.needle_owner = owner
        else:
            self.needle_pos = torch.zeros(0, dtype=torch.long, device=device)
            self.needle_owner = torch.zeros(0, dtype=torch.long, device=device)
        if spec.n_outliers and L:
            keys[:, self.out_ch] += self.out_off
        self.k = keys.to(spec.kv_dtype)
        self.v = vals.to(spec.kv_dtype)
        self.spec, self.b, self.j, self.seed, self.device = spec, b, j, seed, device

    def needle_keys(self) -> torch.Tensor:
        return self.k[self.needle_pos].float()


def repeated_pages(n_pages: int, page_size: int, head_dim: int, n_distinct: int,
                   dtype=torch.bfloat16, seed: int = 0, device="cpu"):
    """Keys and values of one KV head made of ``n_distinct`` random pages
    (entries ~ N(0, I)), each logical page a copy of one of them picked at
    random: pages with equal contents give exact ties in every per-page
    bound and statistic. Returns (k, v), [n_pages·page_size, d] each."""
    g = _gen(device, seed, _REPEAT, n_pages, n_distinct)
    base_k = torch.randn(n_distinct, page_size, head_dim, generator=g, device=device)
    base_v = torch.randn(n_distinct, page_size, head_dim, generator=g, device=device)
    pick = torch.randint(0, n_distinct, (n_pages,), generator=g, device=device)
    k = base_k[pick].reshape(n_pages * page_size, head_dim)
    v = base_v[pick].reshape(n_pages * page_size, head_dim)
    return k.to(dtype), v.to(dtype)


def append_token(spec: Spec, b: int, j: int, pos: int, step: int, centroids,
                 out_ch, out_off, seed: int = 0, device="cpu"):
    """One appended (k, v) for sequence b, KV head j at position pos: [d] each."""
    g = _gen(device, seed, _APPEND, b, j, step)
    d = spec.head_dim
    k = centroids[pos // spec.page_size] + torch.randn(d, generator=g, device=device)
    v = torch.randn(d, generator=g, device=device)
    if out_ch.numel():
        k[out_ch] += out_off
    return k.to(spec.kv_dtype), v.to(spec.kv_dtype)


def step_queries(spec: Spec, b: int, step: int, needle_keys_per_kv, seed: int = 0,
                 device="cpu") -> torch.Tensor:
    """Fresh per-step queries [Hq, d] (stored dtype).

    With ``spec.rotate`` > 0 each query keeps its norm and is turned that
    fraction of the angle toward one random needle key of its KV head
    (spherical interpolation).
    """
    g = _gen(device, seed, _STEPQ, b, step)
    Hq, d, grp = spec.num_q_heads, spec.head_dim, spec.group
    q = torch.randn(Hq, d, generator=g, device=device)
    if spec.rotate > 0.0:
        for h in range(Hq):
            nk = needle_keys_per_kv[h // grp]
            if nk.shape[0] == 0:
                continue
            i = int(torch.randint(nk.shape[0], (1,), generator=g, device=device).item())
            a = q[h] / q[h].norm()
            c = nk[i] / nk[i].norm()
            cosw = float(torch.clamp(torch.dot(a, c), -1.0, 1.0))
            w = math.acos(cosw)
            if w < 1e-6:
                continue
            t = spec.rotate
            r = (math.sin((1 - t) * w) * a + math.sin(t * w) * c) / math.sin(w)
            q[h] = r * q[h].norm()
    return q.to(spec.kv_dtype)


def block_tables(spec: Spec, seed: int = 0):
    """Block table [B, max_pages] (int32, CPU), pool size and pages per seq.

    Every sequence gets ceil(reserved_tokens / P) physical pages. Without
    shuffling they are consecutive; with shuffling they are a random
    permutation of the pool.
    """
    P = spec.page_size
    need = [-(-max(reserved_tokens(spec, b), 1) // P) for b in range(spec.batch)]
    total = sum(need)
    maxp = max(need)
    if spec.shuffled_table:
        perm = torch.randperm(total, generator=_gen("cpu", seed, _TABLE))
    else:
        perm = torch.arange(total)
    bt = torch.zeros(spec.batch, maxp, dtype=torch.int32)
    off = 0
    for b in range(spec.batch):
        bt[b, : need[b]] = perm[off: off + need[b]].to(torch.int32)
        off += need[b]
    return bt, total, need
