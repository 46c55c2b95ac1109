"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects bad arguments on the host before any CUDA call
(all pointers below are dummies that are never dereferenced)."""

import ctypes
import os
import re

import numpy as np
import pytest

from sparse_entmax_attention_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "entmaxkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(entmaxkv_\w+)\s*\(", src))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from sparse_entmax_attention_gb300 import build
        build.build_library()
    return B.lib()


def test_exports_every_declared_function(lib):
    declared = _header_functions()
    assert declared == set(B.EXPORTS), declared ^ set(B.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.entmaxkv_version() == 4
    for code in range(5):
        assert lib.entmaxkv_status_string(code)
    assert lib.entmaxkv_status_string(99) == b"unknown status"


def _cfg(**kw):
    base = dict(num_kv_heads=8, group=4, head_dim=128, page_size=32, max_seqs=1,
                max_pages_per_seq=32768, num_phys_pages=32768, kv_dtype=B.BF16)
    base.update(kw)
    return B.Config(*[base[f] for f, _ in B.Config._fields_])


def _view():
    return B.CacheView(*([256] * 8), None)


def _decode(lib, cfg, **kw):
    a = dict(q=256, seq_ids=None, n=1, alpha=1.5, policy=B.POLICY_GAUSSIAN, budget=0, margin=0.5,
             flags=0, ws=256, ws_bytes=1 << 40, out=256, ids=None, stride=0, nsel=None, tau=None,
             delta=None)
    a.update(kw)
    return lib.entmaxkv_decode(ctypes.byref(cfg), ctypes.byref(_view()), ctypes.c_void_p(a["q"]),
                               a["seq_ids"], a["n"], a["alpha"], a["policy"], a["budget"],
                               a["margin"], a["flags"], ctypes.c_void_p(a["ws"]), a["ws_bytes"],
                               ctypes.c_void_p(a["out"]) if a["out"] else None, a["ids"], a["stride"],
                               a["nsel"], a["tau"], a["delta"], None)


def test_workspace_sizing(lib):
    cfg = _cfg()
    sizes = {p: lib.entmaxkv_workspace_bytes(ctypes.byref(cfg), 1, p, 2048) for p in range(5)}
    assert all(v > 0 for v in sizes.values())
    assert sizes[B.POLICY_TOPK] < sizes[B.POLICY_FULL]
    assert lib.entmaxkv_workspace_bytes(ctypes.byref(cfg), 1, B.POLICY_TOPK, 16) == 0  # < 1 page
    assert lib.entmaxkv_workspace_bytes(ctypes.byref(cfg), 1, 7, 0) == 0               # no policy
    assert lib.entmaxkv_workspace_bytes(ctypes.byref(cfg), 0, 0, 0) == 0               # no sequences
    v = B.WorkspaceView()
    assert lib.entmaxkv_workspace_layout(ctypes.byref(cfg), 1, B.POLICY_GAUSSIAN, 0, ctypes.byref(v)) == 0
    assert v.gauss_ms % 256 == 0 and v.tauhat % 256 == 0 and v.bbox_u == 2 ** 64 - 1
    assert v.total == lib.entmaxkv_workspace_bytes(ctypes.byref(cfg), 1, B.POLICY_GAUSSIAN, 0)
    assert v.z_scores % 256 == 0 and v.z_scores < v.total
    assert lib.entmaxkv_workspace_layout(ctypes.byref(cfg), 1, B.POLICY_SOFTMAX, 0, ctypes.byref(v)) == 0
    assert v.z_scores == 2 ** 64 - 1 and v.page_zmax == 2 ** 64 - 1


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 96, 2), ("page_size", 8, 2), ("group", 9, 2), ("kv_dtype", 5, 1),
    ("num_kv_heads", 0, 1), ("max_pages_per_seq", 0, 1)])
def test_bad_config_is_rejected(lib, field, value, code):
    assert _decode(lib, _cfg(**{field: value})) == code


def test_bad_decode_arguments_are_rejected(lib):
    cfg = _cfg()
    assert _decode(lib, cfg, alpha=1.0, policy=B.POLICY_FULL) == 1          # α ≤ 1
    assert _decode(lib, cfg, alpha=float("nan"), policy=B.POLICY_FULL) == 1
    # Gaussian at an order whose moment fits fail their check (β = 20): refused
    # on the host before anything is queued
    assert _decode(lib, cfg, alpha=1.05) == 2
    assert _decode(lib, cfg, policy=B.POLICY_TOPK, budget=8) == 1           # budget below one page
    assert _decode(lib, cfg, margin=float("inf")) == 1
    assert _decode(lib, cfg, out=0) == 1                                    # out is required
    assert _decode(lib, cfg, ws=256 + 8) == 3                               # misaligned workspace
    assert _decode(lib, cfg, ws_bytes=1024) == 3                            # too small
    ids = ctypes.c_void_p(256)
    assert _decode(lib, cfg, policy=B.POLICY_TOPK, budget=2048, ids=ids, stride=10) == 1
    assert _decode(lib, cfg, n=0) == 0                                      # nothing to do
    assert _decode(lib, cfg, n=-1) == 1


def test_bad_append_arguments_are_rejected(lib):
    cfg = _cfg()
    view = _view()
    f = lib.entmaxkv_append
    p = ctypes.c_void_p(256)
    assert f(ctypes.byref(cfg), ctypes.byref(view), p, p, None, 1, 0, None) == 0   # no tokens
    assert f(ctypes.byref(cfg), ctypes.byref(view), None, p, None, 1, 4, None) == 1
    assert f(ctypes.byref(cfg), ctypes.byref(view), p, p, None, -1, 4, None) == 1
    assert f(ctypes.byref(cfg), ctypes.byref(view), p, p, None, 1, 32768 * 32 + 1, None) == 1
    bad = B.CacheView(0, *([256] * 7), None)
    assert f(ctypes.byref(cfg), ctypes.byref(bad), p, p, None, 1, 4, None) == 1


def test_misaligned_cache_arrays_are_rejected(lib):
    cfg = _cfg()
    for i in range(6):  # k_pool, v_pool, kmin, kmax, mean, m2
        ptrs = [256] * 8
        ptrs[i] = 256 + 8
        view = B.CacheView(*ptrs, None)
        rc = lib.entmaxkv_decode(ctypes.byref(cfg), ctypes.byref(view), ctypes.c_void_p(256), None, 1,
                                 1.5, B.POLICY_GAUSSIAN, 0, 0.5, 0, ctypes.c_void_p(256), 1 << 40,
                                 ctypes.c_void_p(256), None, 0, None, None, None, None)
        assert rc == 1, i


def test_exact_delta_sizing_and_delta_kinds(lib):
    cfg = _cfg()
    f = lib.entmaxkv_workspace_bytes_flags
    for pol, budget in ((B.POLICY_TOPK, 2048), (B.POLICY_GAUSSIAN, 0)):
        plain = lib.entmaxkv_workspace_bytes(ctypes.byref(cfg), 1, pol, budget)
        assert f(ctypes.byref(cfg), 1, pol, budget, 0) == plain
        assert f(ctypes.byref(cfg), 1, pol, budget, B.FLAG_EXACT_DELTA) >= plain + \
            lib.entmaxkv_workspace_bytes(ctypes.byref(cfg), 1, B.POLICY_FULL, 0)
    for pol in (B.POLICY_FULL, B.POLICY_SOFTMAX):
        assert f(ctypes.byref(cfg), 1, pol, 0, B.FLAG_EXACT_DELTA) == \
            lib.entmaxkv_workspace_bytes(ctypes.byref(cfg), 1, pol, 0)
    k = lib.entmaxkv_delta_kind
    assert (k(B.POLICY_FULL, 0), k(B.POLICY_SOFTMAX, B.FLAG_EXACT_DELTA)) == (B.DELTA_ZERO, B.DELTA_ZERO)
    assert (k(B.POLICY_TOPK, 0), k(B.POLICY_GAUSSIAN, 0)) == (B.DELTA_CERTIFIED, B.DELTA_MODEL)
    assert k(B.POLICY_TOPK, B.FLAG_EXACT_DELTA) == B.DELTA_EXACT == k(B.POLICY_GAUSSIAN, B.FLAG_EXACT_DELTA)
    assert k(B.POLICY_SOFTMAX_TOPK, 0) == B.DELTA_CERTIFIED
    assert k(B.POLICY_SOFTMAX_TOPK, B.FLAG_EXACT_DELTA) == B.DELTA_EXACT
    assert k(9, 0) == -1


def test_read_status_needs_a_status_word(lib):
    view = B.CacheView(*([256] * 8), None)  # no status word
    out = ctypes.c_uint32(7)
    assert lib.entmaxkv_read_status(ctypes.byref(view), ctypes.byref(out), 0, None) == 1
    assert lib.entmaxkv_read_status(None, ctypes.byref(out), 0, None) == 1


def test_bf16_metadata_copies_come_in_pairs(lib):
    cfg = _cfg()
    view = B.CacheView(*([256] * 8), None, 256, None)  # mean copy without its m2 copy
    rc = lib.entmaxkv_decode(ctypes.byref(cfg), ctypes.byref(view), ctypes.c_void_p(256), None, 1,
                             1.5, B.POLICY_GAUSSIAN, 0, 0.5, 0, ctypes.c_void_p(256), 1 << 40,
                             ctypes.c_void_p(256), None, 0, None, None, None, None)
    assert rc == 1
    view = B.CacheView(*([256] * 8), None, 264, 256)  # misaligned copy
    rc = lib.entmaxkv_decode(ctypes.byref(cfg), ctypes.byref(view), ctypes.c_void_p(256), None, 1,
                             1.5, B.POLICY_GAUSSIAN, 0, 0.5, 0, ctypes.c_void_p(256), 1 << 40,
                             ctypes.c_void_p(256), None, 0, None, None, None, None)
    assert rc == 1


def test_gaussian_alpha_support_query(lib):
    assert B.gaussian_alpha_supported(1.5) and B.gaussian_alpha_supported(2.0)
    assert B.gaussian_alpha_supported(1.25) and B.gaussian_alpha_supported(3.0)
    assert not B.gaussian_alpha_supported(1.05)   # β = 20: the fits fail their check
    assert not B.gaussian_alpha_supported(1.0) and not B.gaussian_alpha_supported(float("nan"))


@pytest.mark.parametrize("alpha", [1.15, 1.25, 1.75, 3.0, 5.0])
def test_moment_fits_match_the_oracle(lib, alpha):
    """The host-built fits of J_ν(t) = E[(t + Z)_+^ν] (ν = β, β − 1, β − 2),
    evaluated in the kernels' float arithmetic, against the oracle's float64
    J on both sides of t = 0 and past the series switch at t = 16. The value
    is 2^E·M with a float exponent E of size up to about 100 (−t²/(2 ln 2) in
    the left tail, ν·log2 t far right), whose rounding alone is about
    |E|·2^-24 relative in 2^E; hence 1e-5. Where J is below 1e-30 (far left
    tail) only the absolute size is checked."""
    from oracle import pages as opg
    beta = 1.0 / (alpha - 1.0)
    t = np.concatenate([np.linspace(-12.0, 0.0, 97), np.linspace(0.05, 16.0, 160), np.linspace(16.5, 60.0, 30)])
    for order in range(3 if beta > 1.0 else 2):
        got = B.moment_fit_eval(alpha, order, t).astype(np.float64)
        ref = opg.jfun(t.astype(np.float32).astype(np.float64), beta - order)
        big = ref > 1e-30
        rel = np.abs(got[big] - ref[big]) / ref[big]
        assert rel.max() < 1e-5, (alpha, order, float(rel.max()), float(t[big][rel.argmax()]))
        assert np.all(np.abs(got[~big]) < 1e-29)
    with pytest.raises(B.EntmaxKVError):
        B.moment_fit_eval(1.5, 0, t)   # closed forms: no fits
    with pytest.raises(B.EntmaxKVError):
        B.moment_fit_eval(alpha, 3, t)


def test_moment_fit_cache_beyond_its_slots(lib):
    """More orders than the fit cache holds: each still builds (or comes from
    the cache) and evaluates the same as on its first use."""
    alphas = [1.2, 1.3, 1.35, 1.4, 1.45, 1.6, 1.7, 1.8, 2.5]  # nine orders, eight slots
    t = (ctypes.c_float * 3)(-1.0, 0.5, 3.0)
    first = {}
    for a in alphas + alphas[:2]:
        assert lib.entmaxkv_gaussian_alpha_supported(ctypes.c_float(a)) == 1
        out = (ctypes.c_float * 3)()
        assert lib.entmaxkv_moment_fit_eval(ctypes.c_float(a), 0, t, 3, out) == 0
        first.setdefault(a, list(out))
        assert list(out) == first[a]
