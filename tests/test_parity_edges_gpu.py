"""GPU edge cases: empty and one-token sequences, k ≥ pages, a bad block-table
entry, the Gaussian cap, decoding a subset of sequences, token-by-token
appends."""

import math

import numpy as np
import pytest
import torch

from oracle import decode as odec
from oracle import pages as opg
from sparse_entmax_attention_gb300 import binding as B
from sparse_entmax_attention_gb300 import synth

from harness import Built, rel_l2
from test_parity_gpu import check_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ragged():
    spec = synth.custom(4, 1, 128, 16, [0, 1, 17, 333], torch.bfloat16, 1.5, n_needles=2,
                        shuffled_table=True)
    return Built(spec)


@pytest.mark.parametrize("policy,budget", [("full", 0), ("softmax", 0), ("topk", 64),
                                           ("topk", 100000), ("gaussian", 0),
                                           ("softmax_topk", 64)])
def test_empty_and_tiny_sequences(ragged, policy, budget):
    o, _ = check_decode(ragged, policy, 1.5, budget, 0.5, units=[(1, 0), (2, 0), (3, 0)])
    # the empty sequence: zero output, NaN τ, nothing selected, no dropped mass
    assert torch.all(o.out[0] == 0)
    assert torch.all(torch.isnan(o.tau[0]))
    assert int(o.n_sel[0, 0]) == 0
    assert torch.all(o.delta[0] == 0)


def test_bad_block_table_entry_is_flagged_not_fatal():
    spec = synth.custom(4, 1, 128, 16, [320], torch.bfloat16, 1.5, n_needles=2)
    built = Built(spec)
    c = built.cache
    good = c.block_table.clone()
    c.block_table[0, 5] = -7
    c.status.zero_()
    B.decode(c, built.q, 1.5, "full")
    B.decode(c, built.q, 1.5, "topk", 64)
    B.decode(c, built.q, 1.5, "gaussian", 0, 0.5)
    B.decode(c, built.q, 1.5, "softmax")
    torch.cuda.synchronize()
    assert c.device_status() & B.DEV_BAD_PAGE_TABLE
    c.block_table.copy_(good)
    c.status.zero_()
    check_decode(built, "full", 1.5)


def test_bad_seq_id_is_flagged():
    spec = synth.custom(4, 1, 128, 16, [64], torch.bfloat16, 1.5)
    built = Built(spec)
    c = built.cache
    c.status.zero_()
    sid = torch.tensor([3], dtype=torch.int32, device="cuda")
    B.decode(c, built.q, 1.5, "full", seq_ids=sid)
    torch.cuda.synchronize()
    assert c.device_status() & B.DEV_BAD_SEQ_ID


def test_gaussian_cap_overflow_keeps_largest_margins():
    spec = synth.custom(8, 2, 128, 16, [2000], torch.bfloat16, 1.5, n_needles=4, n_outliers=2)
    built = Built(spec)
    c = built.cache
    cap_tokens = 5 * 16
    c.status.zero_()
    o = B.decode(c, built.q, 1.5, "gaussian", cap_tokens, 1.0)
    torch.cuda.synchronize()
    assert c.device_status() & B.DEV_CAPACITY
    for j in range(2):
        K, V = built.host_kv(0, j)
        r = odec.decode_group(K, V, built.host_q(0, j), 1.5, "gaussian", 16, cap_tokens, 1.0)
        assert r["capacity_flag"]
        ids = o.page_ids[0, j, : int(o.n_sel[0, j])].cpu().tolist()
        assert ids == list(r["page_ids"])
        out, tau = odec.attend_pages(K, V, built.host_q(0, j), 1.5, 16, ids)
        for h in range(4):
            assert rel_l2(o.out[0, 4 * j + h].cpu().numpy(), out[h]) <= 2e-3


def test_decode_subset_by_seq_ids():
    spec = synth.custom(8, 2, 128, 32, [900, 2100, 40], torch.bfloat16, 1.5, n_needles=3,
                        shuffled_table=True)
    built = Built(spec)
    allq = built.q
    full = B.decode(built.cache, allq, 1.5, "topk", 256)
    sid = torch.tensor([2, 1], dtype=torch.int32, device="cuda")
    sub = B.decode(built.cache, allq[[2, 1]].contiguous(), 1.5, "topk", 256, seq_ids=sid)
    torch.cuda.synchronize()
    # the page ids are exact; the output is summed with float atomics whose
    # order varies from run to run, so its last bits may differ
    torch.testing.assert_close(sub.page_ids, full.page_ids[[2, 1]], rtol=0, atol=0)
    torch.testing.assert_close(sub.n_sel, full.n_sel[[2, 1]], rtol=0, atol=0)
    torch.testing.assert_close(sub.out, full.out[[2, 1]], rtol=1e-6, atol=1e-7)
    torch.testing.assert_close(sub.tau, full.tau[[2, 1]], rtol=1e-6, atol=1e-7)


def test_token_by_token_append_matches_bulk():
    spec = synth.custom(4, 2, 64, 16, [100], torch.bfloat16, 1.5, n_needles=2)
    bulk = Built(spec)
    step = Built.__new__(Built)
    step.spec = spec
    bt, total, need = synth.block_tables(spec)
    step.cache = B.PagedCache(2, 2, 64, 16, 1, bt.shape[1], total, torch.bfloat16, "cuda")
    step.cache.block_table.copy_(bt.cuda())
    step.q, step.K, step.V = bulk.q, bulk.K, bulk.V
    for t in range(100):  # single tokens, then chunks that straddle pages
        if t < 40:
            B.append(step.cache, bulk.K[0][:, t:t + 1].unsqueeze(0).contiguous(),
                     bulk.V[0][:, t:t + 1].unsqueeze(0).contiguous())
    for t0, t1 in ((40, 45), (45, 77), (77, 100)):
        B.append(step.cache, bulk.K[0][:, t0:t1].unsqueeze(0).contiguous(),
                 bulk.V[0][:, t0:t1].unsqueeze(0).contiguous())
    torch.cuda.synchronize()
    assert int(step.cache.seq_lens[0]) == 100
    a, b = step.cache, bulk.cache
    n_pages = 7
    assert torch.equal(a.k_pool[:n_pages], b.k_pool[:n_pages])
    assert torch.equal(a.kmin[:n_pages], b.kmin[:n_pages]) and torch.equal(a.kmax[:n_pages], b.kmax[:n_pages])
    torch.testing.assert_close(a.mean[:n_pages], b.mean[:n_pages], rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(a.m2[:n_pages], b.m2[:n_pages], rtol=1e-4, atol=1e-5)
    check_decode(step, "gaussian", 1.5, 0, 0.5)


@pytest.mark.parametrize("meta_bf16", [True, False])
def test_scorer_wait_timeout_is_flagged_and_the_context_stays_usable(meta_bf16):
    """The device-side timeout path, made to run without a fault: with
    ENTMAXKV_FLAG_EXPIRE_WAITS the Gaussian scorer's waits for its staged
    copies give up at once. The decode must raise ENTMAXKV_DEV_TIMEOUT on the
    status word, let the copies it issued land, and complete with every page
    unscored (zero output, nothing selected, NaN τ); the next ordinary decode
    on the same context must match the oracle again."""
    spec = synth.custom(8, 2, 128, 32, [5000, 3000], torch.bfloat16, 1.5, n_needles=4,
                        n_outliers=2)
    built = Built(spec, meta_bf16=meta_bf16)
    c = built.cache
    assert c.read_status(clear=True) == 0
    o = B.decode(c, built.q, 1.5, "gaussian", 0, 0.5, B.FLAG_EXPIRE_WAITS)
    st = c.read_status(clear=True)
    assert st & B.DEV_TIMEOUT, hex(st)
    assert st & ~(B.DEV_TIMEOUT | B.DEV_CAND_OVERFLOW) == 0, hex(st)
    assert torch.all(o.out == 0)
    assert torch.all(o.n_sel == 0)
    assert torch.all(torch.isnan(o.tau))
    check_decode(built, "gaussian", 1.5, 0, 0.5)
    assert c.read_status() == 0


@pytest.mark.parametrize("n_pages,n_distinct,max_pages,k_top", [
    (300, 3, None, 0), (5000, 4, None, 0), (2000, 1, None, 0), (700, 3, 70000, 0), (5000, 12, None, 30)])
def test_topk_exact_ties_go_to_the_lower_page(n_pages, n_distinct, max_pages, k_top):
    """Pages with equal contents have equal bounds, so the top-k boundary can
    cut through a class of exact ties; the kept pages of that class must be
    its lowest page indices, bit for bit (summary §2B.1, ties to the lower
    index). 300 pages fall in 5 blocks of the cluster select and 5000 in all
    8, so the tie offset crosses blocks; 2000 copies of one page make every
    key equal (no radix digit at all); a table of 70000 pages per sequence
    takes the one-block select. k_top > 0 keeps that many pages of the
    largest class: k is then below the count of scoring blocks, so the
    cluster select's candidate path (keys at or above the k-th largest
    block maximum) decides, with every candidate tied."""
    P, d, g = 16, 128, 4
    spec = synth.custom(g, 1, d, P, [n_pages * P], torch.bfloat16, 1.5, shuffled_table=True)
    bt, total, _ = synth.block_tables(spec)
    maxp = max_pages or bt.shape[1]
    cache = B.PagedCache(1, g, d, P, 1, maxp, total, torch.bfloat16, "cuda")
    cache.block_table[:, : bt.shape[1]].copy_(bt.cuda())
    k, v = synth.repeated_pages(n_pages, P, d, n_distinct)
    B.append(cache, k[None, None].cuda().contiguous(), v[None, None].cuda().contiguous())
    q = synth.queries(spec, 0).cuda()[None].contiguous()
    K, V, Q = k.double().numpy(), v.double().numpy(), q[0].double().cpu().numpy()
    meta = opg.page_metadata(K, P)
    uhat = np.stack([opg.bbox_bound(Q[h], meta["kmin"], meta["kmax"]) for h in range(g)]).max(axis=0)
    classes = np.unique(uhat)[::-1]
    if k_top:
        kp = k_top
        assert (uhat == classes[0]).sum() > kp
    elif classes.size == 1:
        kp = n_pages // 3
    else:  # through the middle of the second-largest class
        kp = int((uhat > classes[1]).sum() + (uhat == classes[1]).sum() // 2)
    assert 0 < kp < n_pages
    o = B.decode(cache, q, 1.5, "topk", kp * P)
    torch.cuda.synchronize()
    # (equal pages give equal page maxima, which can fill the exact-τ
    # candidate lists and send the solve down its full-scan path)
    assert cache.device_status() & ~B.DEV_CAND_OVERFLOW == 0, hex(cache.device_status())
    r = odec.decode_group(K, V, Q, 1.5, "topk", P, kp * P)
    ids = o.page_ids[0, 0, : int(o.n_sel[0, 0])].cpu().tolist()
    assert ids == list(r["page_ids"]) == list(opg.select_topk(uhat, kp))
    for h in range(g):
        assert rel_l2(o.out[0, h].cpu().numpy(), r["out"][h]) <= 2e-3
        assert abs(float(o.tau[0, h]) - r["tau"][h]) <= 1e-4


def test_pass_a_share_longer_than_its_page_list():
    """256 (sequence, KV head) units of 3100 pages each, top-k keeping all but
    one page: a multi-sequence launch gives each unit 3 blocks on a 152-SM
    GPU, so a block's share (1033 pages) runs past its 1024-entry page list
    and continues in the global selection list. Ids, output and τ against the
    oracle on sampled units."""
    P, n_pages = 16, 3100
    spec = synth.custom(32, 32, 64, P, [n_pages * P] * 8, torch.bfloat16, 1.5, n_needles=2)
    built = Built(spec)
    budget = (n_pages - 1) * P
    check_decode(built, "topk", 1.5, budget, 0.0, units=[(0, 0), (3, 17), (7, 31)])
    check_decode(built, "gaussian", 1.5, 0, 2.0, units=[(5, 9)])
