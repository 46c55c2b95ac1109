"""GPU: the exact dropped mass (ENTMAXKV_FLAG_EXACT_DELTA) against the oracle,
and the device status read.

δ = Σ over the tokens outside the kept pages of the full-cache α-entmax
weights (summary §3); the oracle computes it in float64 from its own full
solve. Where a near-tie flips a page, the expected δ is taken on the GPU's own
kept set. Tolerance: 2e-4 absolute, from |τ − τ_oracle| ≤ 1e-4 moving each
kept weight by at most β·p^{(β−1)/β}·1e-4.
"""

import numpy as np
import pytest
import torch

from oracle import decode as odec
from oracle import entmax as oem
from sparse_entmax_attention_gb300 import binding as B
from sparse_entmax_attention_gb300 import synth

from harness import Built

pytestmark = pytest.mark.gpu

TOL_DELTA = 2e-4


@pytest.fixture(scope="module")
def built_bf16():
    spec = synth.custom(8, 2, 128, 16, [3000, 1217], torch.bfloat16, 1.5, n_needles=6,
                        n_outliers=2, shuffled_table=True)
    return Built(spec, prefill_chunk=700)


@pytest.fixture(scope="module")
def built_f32():
    return Built(synth.workload("single-head-d64-4k-p16-fp32"))


def _exact_delta_on(K, Q, alpha, P, page_ids, soft=False):
    """Full-cache entmax (softmax with ``soft``) mass outside the given pages,
    per query head."""
    keep = np.zeros(K.shape[0], bool)
    for p in page_ids:
        keep[p * P:(p + 1) * P] = True
    s = K @ Q.T / np.sqrt(K.shape[1])
    full = (lambda x: oem.softmax(x)) if soft else (lambda x: oem.entmax(x, alpha))
    return np.array([full(s[:, h])[0][~keep].sum() for h in range(Q.shape[0])])


@pytest.mark.parametrize("policy,budget,margin,alpha", [
    ("topk", 256, 0.0, 1.5), ("topk", 512, 0.0, 2.0), ("gaussian", 0, 0.5, 1.5),
    ("gaussian", 0, 0.0, 2.0), ("gaussian", 0, 0.5, 1.25), ("softmax_topk", 256, 0.0, 1.5)])
@pytest.mark.parametrize("which", ["bf16", "f32"])
def test_exact_delta_matches_oracle(built_bf16, built_f32, which, policy, budget, margin, alpha):
    built = built_bf16 if which == "bf16" else built_f32
    spec, cache = built.spec, built.cache
    P, g = spec.page_size, spec.group
    plain = B.decode(cache, built.q, alpha, policy, budget, margin)
    o = B.decode(cache, built.q, alpha, policy, budget, margin, B.FLAG_EXACT_DELTA)
    torch.cuda.synchronize()
    assert cache.device_status() & ~B.DEV_CAND_OVERFLOW == 0, hex(cache.device_status())
    # the flag adds δ and changes nothing else (out and τ up to the order in
    # which the candidate lists were filled, which moves float sums by ulps)
    torch.testing.assert_close(o.out, plain.out, rtol=1e-6, atol=1e-7)
    torch.testing.assert_close(o.tau, plain.tau, rtol=1e-6, atol=1e-6, equal_nan=True)
    assert torch.equal(plain.n_sel, o.n_sel) and torch.equal(plain.page_ids, o.page_ids)
    assert B.delta_kind(policy, B.FLAG_EXACT_DELTA) == B.DELTA_EXACT
    delta, n_sel, pids = o.delta.cpu().numpy(), o.n_sel.cpu().numpy(), o.page_ids.cpu().numpy()
    for b in range(spec.batch):
        for j in range(spec.num_kv_heads):
            K, V = built.host_kv(b, j)
            Q = built.host_q(b, j)
            got = pids[b, j, : n_sel[b, j]]
            r = odec.decode_group(K, V, Q, alpha, policy, P, budget, margin)
            if list(got) == list(r["page_ids"]):
                want = r["delta_exact"]
            else:
                want = _exact_delta_on(K, Q, alpha, P, got, soft=policy == "softmax_topk")
            np.testing.assert_allclose(delta[b, j * g:(j + 1) * g], want, atol=TOL_DELTA, rtol=0)


def test_exact_delta_workspace_and_kinds(built_f32):
    c = built_f32.cache
    for pol in ("topk", "gaussian", "softmax_topk"):
        assert B.workspace_bytes(c, 1, pol, 256, B.FLAG_EXACT_DELTA) > B.workspace_bytes(c, 1, pol, 256)
    for pol in ("full", "softmax"):
        assert B.workspace_bytes(c, 1, pol, 0, B.FLAG_EXACT_DELTA) == B.workspace_bytes(c, 1, pol, 0)
    # a workspace sized without the flag is refused when the flag is set
    ws = B.alloc_workspace(c, 1, "topk", 256)
    with pytest.raises(B.EntmaxKVError):
        B.decode(c, built_f32.q, 1.5, "topk", 256, 0.0, B.FLAG_EXACT_DELTA, workspace=ws)


def test_read_status_reports_and_clears():
    spec = synth.custom(4, 1, 128, 16, [320], torch.bfloat16, 1.5, n_needles=2)
    built = Built(spec)
    c = built.cache
    assert c.read_status() == 0
    good = c.block_table.clone()
    c.block_table[0, 3] = c.cfg.num_phys_pages  # outside the pool
    B.decode(c, built.q, 1.5, "full")
    assert c.read_status(clear=True) & B.DEV_BAD_PAGE_TABLE
    assert c.read_status() == 0
    c.block_table.copy_(good)
