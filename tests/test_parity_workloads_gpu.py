"""GPU parity on the named synthetic workloads at their full sizes.

The 32k-token GQA workload is checked on every KV head; the 128k, 1M and
batched workloads on sampled (sequence, KV head) units, which the oracle
computes one by one, in the same launch configuration the benchmark times.
"""

import numpy as np
import pytest
import torch

from sparse_entmax_attention_gb300 import binding as B
from sparse_entmax_attention_gb300 import synth

from harness import Built
from test_parity_gpu import check_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gqa32k():
    return Built(synth.workload("gqa32x8-d128-32k-p16-bf16"))


@pytest.mark.parametrize("policy,budget,margin", [
    ("topk", 1024, 0.0), ("full", 0, 0.0), ("softmax", 0, 0.0), ("gaussian", 0, 0.5),
    ("softmax_topk", 1024, 0.0)])
def test_gqa32k_all_heads(gqa32k, policy, budget, margin):
    check_decode(gqa32k, policy, 1.5, budget, margin)


@pytest.mark.parametrize("alpha", [1.25, 3.0])
def test_gqa32k_gaussian_general_alpha(gqa32k, alpha):
    check_decode(gqa32k, "gaussian", alpha, 0, 0.5)


@pytest.fixture(scope="module")
def gqa128k():
    return Built(synth.workload("gqa32x8-d128-128k-p32-bf16"))


@pytest.mark.parametrize("alpha", [1.5, 2.0])
@pytest.mark.parametrize("margin", [0.0, 0.5, 1.0])
def test_gqa128k_rotated_steps(gqa128k, alpha, margin):
    spec = gqa128k.spec
    nk = [d.needle_keys() for d in gqa128k.draws[0]]
    for step in (1, 2):
        q = synth.step_queries(spec, 0, step, nk, device="cuda").unsqueeze(0).contiguous()
        o, _ = check_decode(gqa128k, "gaussian", alpha, 0, margin, q=q, units=[(0, 0), (0, 5)])
        n_sel = int(o.n_sel.float().mean().round())
        check_decode(gqa128k, "topk", alpha, max(1, n_sel) * spec.page_size, 0.0, q=q,
                     units=[(0, 0), (0, 5)], check_intermediates=False)


@pytest.fixture(scope="module")
def gqa1m():
    # the benchmark's cache: fp32 statistics plus the bf16 copies the
    # Gaussian scorer streams, with room in the table for one appended token
    # (the last test of this module appends it)
    spec = synth.workload("gqa32x8-d128-1m-p32-bf16")
    spec = synth.Spec(**{**spec.__dict__, "steps": 1, "append_per_step": True})
    return Built(spec, meta_bf16=True)


@pytest.mark.parametrize("policy,budget,margin", [
    ("gaussian", 0, 0.5), ("topk", 2048, 0.0), ("full", 0, 0.0), ("softmax", 0, 0.0),
    ("softmax_topk", 2048, 0.0)])
def test_gqa1m_sampled_heads(gqa1m, policy, budget, margin):
    """The 1M-token cache in the launch configuration the benchmark times; the
    Gaussian selector here streams the bf16 copies (tensor-core scorer)."""
    check_decode(gqa1m, policy, 1.5, budget, margin, units=[(0, 0), (0, 3), (0, 7)])


def test_gqa1m_gaussian_fp32_metadata(gqa1m):
    """The same Gaussian decode from the fp32 statistics (the scorer for caches
    without bf16 copies)."""
    check_decode(gqa1m, "gaussian", 1.5, 0, 0.5, units=[(0, 0), (0, 7)],
                 cache=gqa1m.cache.fp32_metadata())


def test_batched_shuffled_with_appends():
    spec = synth.workload("batch16-loguniform-4k-256k-p16-bf16")
    built = Built(spec)
    c = built.cache
    units = [(0, 0), (7, 3), (15, 6)]
    for step in range(3):
        ks, vs = [], []
        for b in range(spec.batch):
            kk, vv = [], []
            pos = int(c.seq_lens[b].item())
            for j in range(spec.num_kv_heads):
                d = built.draws[b][j]
                k, v = synth.append_token(spec, b, j, pos, step, d.centroids, d.out_ch,
                                          d.out_off, device="cuda")
                kk.append(k)
                vv.append(v)
            ks.append(torch.stack(kk))
            vs.append(torch.stack(vv))
        K = torch.stack(ks).unsqueeze(2).contiguous()  # [B, Hkv, 1, d]
        V = torch.stack(vs).unsqueeze(2).contiguous()
        B.append(c, K, V)
        for b in range(spec.batch):
            built.K[b] = torch.cat([built.K[b], K[b]], dim=1)
            built.V[b] = torch.cat([built.V[b], V[b]], dim=1)
        q = torch.stack([synth.step_queries(spec, b, step, None, device="cuda")
                         for b in range(spec.batch)]).contiguous()
        check_decode(built, "gaussian", 1.5, 0, 0.5, q=q, units=units)


def test_gqa1m_bulk_prefill_metadata(gqa1m):
    """The 1M-token prefill is one bulk append that writes the tokens and
    builds every page's metadata in the same kernel. On sampled pages of two
    KV heads (plus the last page) the stored tokens equal the input, the
    bounding box equals the oracle's exactly, the mean and variance match
    the oracle's float64 statistics of the same keys, and the bf16 copies are
    the rounded fp32 statistics."""
    from oracle import pages as opg
    spec, c = gqa1m.spec, gqa1m.cache
    P = spec.page_size
    rng = np.random.default_rng(7)
    bt = c.block_table[0].cpu().numpy()
    for j in (0, 7):
        L = int(c.seq_lens[0].item())
        n_pages = -(-L // P)
        pages = np.unique(np.concatenate([rng.choice(n_pages, 64, replace=False), [n_pages - 1]]))
        K = gqa1m.K[0][j, :L]
        for p in pages:
            rows = K[p * P:min(L, (p + 1) * P)].double().cpu().numpy()
            meta = opg.page_metadata(rows, P)
            ph = int(bt[p])
            assert np.array_equal(c.k_pool[ph, j, :rows.shape[0]].double().cpu().numpy(), rows)
            assert np.array_equal(c.kmin[ph, j].double().cpu().numpy(), meta["kmin"][0])
            assert np.array_equal(c.kmax[ph, j].double().cpu().numpy(), meta["kmax"][0])
            np.testing.assert_allclose(c.mean[ph, j].double().cpu().numpy(), meta["mean"][0], atol=2e-6, rtol=1e-5)
            np.testing.assert_allclose(c.m2[ph, j].double().cpu().numpy() / rows.shape[0], meta["var"][0],
                                       atol=1e-5, rtol=1e-4)
            assert torch.equal(c.mean_bf16[ph, j], c.mean[ph, j].to(torch.bfloat16))
            assert torch.equal(c.m2_bf16[ph, j], c.m2[ph, j].to(torch.bfloat16))


def test_gqa1m_one_token_past_eight_tauhat_blocks(gqa1m):
    """One appended token takes the 1M row to 32769 pages, as in the
    benchmark's timed steps. That is one page past the 8 × 4096 that the τ̂
    cluster holds in registers, so 7 of its 8 blocks carry pages past their
    registers. The Gaussian decode (tensor-core scorer, τ̂, passes A and B)
    and top-k against the oracle after the append. Runs last in the module:
    it grows the shared cache."""
    spec, c = gqa1m.spec, gqa1m.cache
    b = 0
    pos = int(c.seq_lens[b].item())
    kk, vv = [], []
    for j in range(spec.num_kv_heads):
        d = gqa1m.draws[b][j]
        k, v = synth.append_token(spec, b, j, pos, 0, d.centroids, d.out_ch, d.out_off, device="cuda")
        kk.append(k)
        vv.append(v)
    K = torch.stack(kk).unsqueeze(0).unsqueeze(2).contiguous()  # [1, Hkv, 1, d]
    V = torch.stack(vv).unsqueeze(0).unsqueeze(2).contiguous()
    B.append(c, K, V)
    gqa1m.K[b] = torch.cat([gqa1m.K[b], K[0]], dim=1)
    gqa1m.V[b] = torch.cat([gqa1m.V[b], V[0]], dim=1)
    L = int(c.seq_lens[b].item())
    assert L == (1 << 20) + 1 and -(-L // spec.page_size) == 8 * 4096 + 1
    check_decode(gqa1m, "gaussian", 1.5, 0, 0.5, units=[(0, 0), (0, 7)])
    check_decode(gqa1m, "topk", 1.5, 2048, 0.0, units=[(0, 0), (0, 7)])
