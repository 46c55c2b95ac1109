"""The seeded input generator: shapes, determinism, planted structure."""

import math

import torch

from sparse_entmax_attention_gb300 import synth


def test_named_workloads_shapes():
    for name in synth.WORKLOAD_NAMES:
        spec = synth.workload(name)
        assert spec.num_q_heads % spec.num_kv_heads == 0
        bt, total, need = synth.block_tables(spec)
        assert bt.shape == (spec.batch, max(need))
        used = torch.cat([bt[b, : need[b]] for b in range(spec.batch)])
        assert used.numel() == total and torch.unique(used).numel() == total
    lens = synth.workload("batch16-loguniform-4k-256k-p16-bf16").context_lens
    assert len(lens) == 16 and all(4096 <= L <= 262144 for L in lens)


def test_shuffled_table_is_a_permutation():
    spec = synth.workload("batch16-loguniform-4k-256k-p16-bf16")
    bt, total, need = synth.block_tables(spec)
    ids = torch.cat([bt[b, : need[b]] for b in range(spec.batch)])
    assert torch.equal(torch.sort(ids).values, torch.arange(total, dtype=torch.int32))
    assert not torch.equal(ids, torch.arange(total, dtype=torch.int32))


def test_head_draws_deterministic_and_needles():
    spec = synth.custom(4, 1, 64, 16, [1000], torch.bfloat16, n_needles=8, n_outliers=2)
    q = synth.queries(spec, 0)
    a = synth.HeadDraws(spec, 0, 0, q)
    b = synth.HeadDraws(spec, 0, 0, q)
    assert torch.equal(a.k, b.k) and torch.equal(a.v, b.v)
    assert a.k.dtype == torch.bfloat16 and a.k.shape == (1000, 64)
    # needles align with their owner's query: score ≈ 3·‖q‖ (plus the outlier shift)
    kf = a.k.float()
    qf = q.float()
    for p, h in zip(a.needle_pos.tolist(), a.needle_owner.tolist()):
        s = float(kf[p] @ qf[h]) / math.sqrt(64)
        others = kf @ qf[h] / math.sqrt(64)
        assert s > float(torch.quantile(others, 0.99))


def test_step_queries_keep_norm_and_turn_toward_needles():
    spec = synth.custom(2, 1, 32, 16, [256], torch.float32, n_needles=4)
    spec.rotate = 0.3
    q0 = synth.queries(spec, 0)
    hd = synth.HeadDraws(spec, 0, 0, q0)
    q1 = synth.step_queries(spec, 0, 1, [hd.needle_keys()])
    g = synth._gen("cpu", 0, synth._STEPQ, 0, 1)
    raw = torch.randn(2, 32, generator=g)
    torch.testing.assert_close(q1.norm(dim=1), raw.norm(dim=1), rtol=1e-5, atol=1e-5)
