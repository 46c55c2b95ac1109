"""One decode policy on one synthetic cache, repeated: the small cases that
kernel profiles are taken on.

    python -m sparse_entmax_attention_gb300.profile_case --policy softmax --tokens 262144

The cache has the 1M workload's shape (32 query heads over 8 KV heads,
d = 128, page 32, bf16 keys and values, bf16 metadata copies) at the given
length, filled through the library's own append. Each of --reps decodes is
preceded by a 512 MiB write, so every decode starts with cold L2, as in the
bench. Policies: gaussian, topk, softmax, softmax_topk, full, full_dense.
"""

from __future__ import annotations

import argparse

import torch

from . import binding as B
from . import runner, synth


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--policy", default="gaussian")
    ap.add_argument("--tokens", type=int, default=262144)
    ap.add_argument("--reps", type=int, default=4)
    ap.add_argument("--budget", type=int, default=2048, help="top-k budget in tokens")
    ap.add_argument("--alpha", type=float, default=1.5)
    ap.add_argument("--margin", type=float, default=0.5)
    args = ap.parse_args(argv)
    spec = synth.Spec("profile-gqa32x8-d128-p32-bf16", 32, 8, 128, 32, [args.tokens], torch.bfloat16,
                      args.alpha, n_needles=64, n_outliers=4)
    wl = runner.Workload(spec, device="cuda", meta_bf16=True)
    policy, flags = args.policy, 0
    if policy == "full_dense":
        policy, flags = "full", B.FLAG_DENSE_V
    budget = args.budget if policy in ("topk", "softmax_topk") else 0
    margin = args.margin if policy == "gaussian" else 0.0
    ws = B.alloc_workspace(wl.cache, 1, policy, budget)
    out = B.alloc_outputs(wl.cache, 1, policy, budget)
    flush = torch.empty(128 << 20, dtype=torch.int32, device="cuda")
    for _ in range(args.reps):
        flush.fill_(1)
        B.decode(wl.cache, wl.q, args.alpha, policy, budget, margin, flags, workspace=ws, outputs=out)
    torch.cuda.synchronize()
    status = wl.cache.device_status() & ~B.DEV_CAND_OVERFLOW
    print(f"{args.policy}: {args.reps} decodes of a {args.tokens}-token cache, device status {status:#x}")
    return 0 if status == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
