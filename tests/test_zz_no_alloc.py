"""The allocation-free softmax decode entry point.

Some embedders cannot call cudaMalloc at decode time (code running inside an
allocator's own callbacks, graph-building code that must not allocate, or a
runtime that owns all device memory), so the library offers one decode whose
scratch is a fixed array compiled into it. This checks, through the C ABI,
that two calls in a row match the ordinary softmax decode and the float64
oracle's full-cache softmax. Kept in its own
file, named so that pytest collects it last.
"""

import ctypes

import pytest
import torch

from oracle import decode as odec
from sparse_entmax_attention_gb300 import binding as B
from sparse_entmax_attention_gb300 import synth

from harness import Built, rel_l2

pytestmark = pytest.mark.gpu


def _noalloc(built, q, out, lse):
    L = B.lib()
    c = built.cache
    return L.entmaxkv_decode_softmax_noalloc(
        ctypes.byref(c.cfg), ctypes.byref(c.view), ctypes.c_void_p(q.data_ptr()), None,
        q.shape[0], ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_softmax_matches_decode_twice():
    spec = synth.custom(8, 2, 128, 16, [3000, 700], torch.bfloat16, 1.5, n_needles=4,
                        n_outliers=2, shuffled_table=True)
    built = Built(spec)
    q = built.q
    ref = B.decode(built.cache, q, 1.5, "softmax")
    assert B.lib().entmaxkv_noalloc_scratch_bytes() == 8 << 20
    for _ in range(2):
        out = torch.full_like(ref.out, float("nan"))
        lse = torch.full_like(ref.tau, float("nan"))
        assert _noalloc(built, q, out, lse) == 0
        torch.cuda.synchronize()
        assert built.cache.device_status() == 0
        for b in range(q.shape[0]):
            for h in range(spec.num_q_heads):
                assert rel_l2(out[b, h].cpu().numpy(), ref.out[b, h].cpu().numpy()) <= 2e-3
        torch.testing.assert_close(lse, ref.tau, rtol=0, atol=1e-4)
    # and against the float64 oracle's full-cache softmax on the stored bits
    g = spec.group
    for b in range(q.shape[0]):
        for j in range(spec.num_kv_heads):
            K, V = built.host_kv(b, j)
            r = odec.decode_group(K, V, built.host_q(b, j), 1.5, "softmax", spec.page_size, diagnostics=False)
            for h in range(g):
                assert rel_l2(out[b, j * g + h].cpu().numpy(), r["out"][h]) <= 2e-3, (b, j, h)
                assert abs(float(lse[b, j * g + h]) - r["tau"][h]) <= 1e-4, (b, j, h)


def test_noalloc_rejects_oversized_shape():
    # A cache geometry whose softmax scratch exceeds the fixed array is refused
    # before anything is queued (no device memory is touched: dummy pointers).
    cfg = B.Config(8, 4, 128, 16, 4096, 65536, 1, B.BF16)
    need = B.lib().entmaxkv_workspace_bytes(ctypes.byref(cfg), 4096, B.POLICY_SOFTMAX, 0)
    assert need > B.lib().entmaxkv_noalloc_scratch_bytes()
    view = B.CacheView(*([16] * 8), None)
    rc = B.lib().entmaxkv_decode_softmax_noalloc(ctypes.byref(cfg), ctypes.byref(view),
                                                 ctypes.c_void_p(16), None, 4096,
                                                 ctypes.c_void_p(16), None, None)
    assert rc == 3  # ENTMAXKV_ERR_WORKSPACE_TOO_SMALL
