"""The captured serving step (`binding.DecodeStep`: append + decode replayed
from a CUDA graph over fixed buffers) against the same step made of one API
call per operation, on twin caches filled from the same seed."""

import pytest
import torch

from sparse_entmax_attention_gb300 import binding as B
from sparse_entmax_attention_gb300 import runner, synth

pytestmark = pytest.mark.gpu


def _close_per_head(got, want, tol=1e-5):
    g, w = got.double().cpu(), want.double().cpu()
    err = (g - w).norm(dim=-1) / w.norm(dim=-1).clamp_min(1e-30)
    assert float(err.max()) <= tol, float(err.max())


@pytest.mark.parametrize("policy,budget,margin", [("gaussian", 0, 0.5), ("topk", 256, 0.0)])
def test_captured_step_matches_eager_calls(policy, budget, margin):
    spec = synth.custom(8, 2, 128, 32, [3000, 1217], torch.bfloat16, 1.5, n_needles=3, steps=4,
                        append_per_step=True, shuffled_table=True)
    a = runner.Workload(spec, device="cuda", meta_bf16=True)
    b = runner.Workload(spec, device="cuda", meta_bf16=True)
    step = B.DecodeStep(b.cache, spec.batch, 1.5, policy, budget, margin)
    ws = B.alloc_workspace(a.cache, spec.batch, policy, budget)
    o = B.alloc_outputs(a.cache, spec.batch, policy, budget)
    for i in range(3):
        k, v = a.step_tokens(i)
        q = a.step_queries(i)
        B.append(a.cache, k, v)
        ea = B.decode(a.cache, q, 1.5, policy, budget, margin, workspace=ws, outputs=o)
        eb = step.run(k, v, q)
        torch.cuda.synchronize()
        assert torch.equal(a.cache.seq_lens, b.cache.seq_lens)
        assert torch.equal(ea.n_sel, eb.n_sel)
        for s in range(spec.batch):
            for j in range(spec.num_kv_heads):
                n = int(ea.n_sel[s, j])
                assert torch.equal(ea.page_ids[s, j, :n], eb.page_ids[s, j, :n])
        # the output is summed with float atomics in the order blocks finish:
        # each head's output vector agrees in relative L2 (single entries
        # near zero can differ by a few ulps of the larger terms)
        _close_per_head(eb.out, ea.out)
        torch.testing.assert_close(eb.tau, ea.tau, rtol=1e-5, atol=1e-6)
    assert a.cache.device_status() & ~B.DEV_CAND_OVERFLOW == 0
    assert b.cache.device_status() & ~B.DEV_CAND_OVERFLOW == 0


def test_captured_step_with_host_io_matches_eager_calls():
    """run_host: host tensors in, one H2D and one D2H inside the step's graph."""
    spec = synth.custom(8, 2, 128, 32, [3000, 1217], torch.bfloat16, 1.5, n_needles=3, steps=4,
                        append_per_step=True)
    a = runner.Workload(spec, device="cuda", meta_bf16=True)
    b = runner.Workload(spec, device="cuda", meta_bf16=True)
    step = B.DecodeStep(b.cache, spec.batch, 1.5, "gaussian", 0, 0.5)
    ws = B.alloc_workspace(a.cache, spec.batch, "gaussian")
    o = B.alloc_outputs(a.cache, spec.batch, "gaussian")
    for i in range(3):
        k, v = a.step_tokens(i)
        q = a.step_queries(i)
        B.append(a.cache, k, v)
        ea = B.decode(a.cache, q, 1.5, "gaussian", 0, 0.5, workspace=ws, outputs=o)
        out, tau, delta, n_sel = step.run_host(k.cpu(), v.cpu(), q.cpu())
        torch.cuda.synchronize()
        assert torch.equal(a.cache.seq_lens, b.cache.seq_lens)
        assert torch.equal(n_sel, ea.n_sel.cpu())
        _close_per_head(out, ea.out.cpu())
        torch.testing.assert_close(tau, ea.tau.cpu(), rtol=1e-5, atol=1e-6)
        torch.testing.assert_close(delta, ea.delta.cpu(), rtol=1e-5, atol=1e-6)
    assert b.cache.device_status() & ~B.DEV_CAND_OVERFLOW == 0
