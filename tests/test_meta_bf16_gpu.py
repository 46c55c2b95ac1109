"""GPU: caches that keep bf16 copies of the page mean and m2 for the Gaussian
scorer.

The copies themselves must equal the round-to-nearest-even bf16 of the fp32
value append keeps (which the fp32 metadata tests pin to the float64 page
statistics), including pages filled token by token. Decode parity is checked
against the oracle's own reading of such a cache: its exact float64 mean and
m2 rounded to bfloat16 (no value is read back from the GPU). Where the GPU's
float32 statistic and the exact one round to different bfloat16 neighbours
the pages can differ inside a small band; check_decode accepts and records
those as rounding-boundary near ties and fails on any other difference.
"""

import pytest
import torch

from sparse_entmax_attention_gb300 import binding as B
from sparse_entmax_attention_gb300 import synth

from harness import Built
from test_parity_gpu import check_decode

pytestmark = pytest.mark.gpu


def _copies_match(cache):
    assert torch.equal(cache.mean_bf16, cache.mean.to(torch.bfloat16))
    assert torch.equal(cache.m2_bf16, cache.m2.to(torch.bfloat16))


@pytest.fixture(scope="module")
def built_meta16():
    spec = synth.custom(8, 2, 128, 16, [3000, 1217], torch.bfloat16, 1.5, n_needles=6,
                        n_outliers=2, shuffled_table=True)
    return Built(spec, prefill_chunk=700, meta_bf16=True)


def test_copies_are_the_rounded_fp32_metadata(built_meta16):
    _copies_match(built_meta16.cache)


@pytest.mark.parametrize("alpha,margin", [(1.5, 0.5), (2.0, 0.0), (1.5, 1.0), (1.25, 0.5), (3.0, 0.0)])
def test_gaussian_decode_on_bf16_metadata(built_meta16, alpha, margin):
    check_decode(built_meta16, "gaussian", alpha, 0, margin)


# The tensor-core scorers' two operand layouts (Gaussian statistics and the
# top-k bounding box): groups of up to 4 query heads put the metadata in the
# tile's rows and the queries in its columns, larger groups the other way
# round. Shapes: d = 64 and 128, a padded head (group 3), and KV-head counts
# that leave warps of a block idle (3 and 9 of a block's 8).
@pytest.mark.parametrize("hq,hkv,d,p", [(24, 3, 64, 32), (6, 2, 64, 16), (10, 2, 128, 32), (9, 9, 128, 16)])
def test_gaussian_scorer_group_shapes(hq, hkv, d, p):
    spec = synth.custom(hq, hkv, d, p, [1900, 333], torch.bfloat16, 1.5, n_needles=3, n_outliers=1,
                        shuffled_table=True)
    built = Built(spec, meta_bf16=True)
    _copies_match(built.cache)
    for alpha, margin in ((1.5, 0.5), (2.0, 0.0)):
        check_decode(built, "gaussian", alpha, 0, margin)
    check_decode(built, "topk", 1.5, 256, 0.0)


def test_bf16_metadata_appended_token_by_token():
    spec = synth.custom(2, 2, 64, 16, [77], torch.float32, 1.5, n_needles=2)
    built = Built(spec, prefill_chunk=1, meta_bf16=True)
    _copies_match(built.cache)
    check_decode(built, "gaussian", 1.5, 0, 0.5)


def test_other_policies_ignore_the_copies(built_meta16):
    for policy, budget in (("topk", 256), ("full", 0)):
        check_decode(built_meta16, policy, 1.5, budget, 0.0)


def test_copies_must_come_in_pairs():
    spec = synth.custom(2, 1, 64, 16, [40], torch.bfloat16, 1.5, n_needles=1)
    built = Built(spec, meta_bf16=True)
    c = built.cache
    view = B.CacheView(*[getattr(c.view, f) for f, _ in B.CacheView._fields_])
    view.m2_bf16 = None
    ws = B.alloc_workspace(c, 1, "gaussian")
    o = B.alloc_outputs(c, 1, "gaussian")
    import ctypes
    rc = B.lib().entmaxkv_decode(ctypes.byref(c.cfg), ctypes.byref(view), ctypes.c_void_p(built.q.data_ptr()),
                                 None, 1, 1.5, B.POLICY_GAUSSIAN, 0, 0.5, 0, ctypes.c_void_p(ws.data_ptr()),
                                 ws.numel(), ctypes.c_void_p(o.out.data_ptr()), None, 0, None, None, None,
                                 None)
    assert rc == 1
