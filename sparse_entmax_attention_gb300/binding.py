"""Python binding of libentmaxkv (ctypes). Argument marshalling only.

Every step of the decode runs in the library's CUDA kernels; this module
allocates caller-owned buffers with torch, passes their device pointers and
the current CUDA stream, and turns non-zero return codes into exceptions.
There is no fallback: if the library is missing or fails to load, calls
raise.
"""

from __future__ import annotations

import copy
import ctypes
import os
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libentmaxkv.so")

F32, BF16 = 0, 1
POLICY_FULL, POLICY_TOPK, POLICY_GAUSSIAN, POLICY_SOFTMAX, POLICY_SOFTMAX_TOPK = 0, 1, 2, 3, 4
POLICIES = {"full": POLICY_FULL, "topk": POLICY_TOPK, "gaussian": POLICY_GAUSSIAN,
            "softmax": POLICY_SOFTMAX, "softmax_topk": POLICY_SOFTMAX_TOPK}
FLAG_DENSE_V, FLAG_EXACT_DELTA, FLAG_EXPIRE_WAITS = 0x1, 0x2, 0x100
DELTA_ZERO, DELTA_CERTIFIED, DELTA_MODEL, DELTA_EXACT = 0, 1, 2, 3
DEV_BAD_PAGE_TABLE, DEV_CAPACITY, DEV_TAUHAT_NOCONV = 0x1, 0x2, 0x4
DEV_CAND_OVERFLOW, DEV_TAU_NOCONV, DEV_BAD_SEQ_ID, DEV_TIMEOUT = 0x8, 0x10, 0x20, 0x40

# Symbols the header declares (kept in step with include/entmaxkv.h by a test).
EXPORTS = ("entmaxkv_version", "entmaxkv_status_string", "entmaxkv_append",
           "entmaxkv_workspace_bytes", "entmaxkv_decode", "entmaxkv_decode_profiled",
           "entmaxkv_workspace_layout", "entmaxkv_noalloc_scratch_bytes",
           "entmaxkv_decode_softmax_noalloc", "entmaxkv_workspace_bytes_flags",
           "entmaxkv_delta_kind", "entmaxkv_read_status", "entmaxkv_gaussian_alpha_supported",
           "entmaxkv_moment_fit_eval")
STAGE_EVENTS = 6
STAGES = ("clear", "score", "select", "pass_a", "pass_b")


class Config(ctypes.Structure):
    _fields_ = [("num_kv_heads", ctypes.c_int32), ("group", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_seqs", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
                ("num_phys_pages", ctypes.c_int32), ("kv_dtype", ctypes.c_int32)]


class CacheView(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("kmin", ctypes.c_void_p), ("kmax", ctypes.c_void_p),
                ("mean", ctypes.c_void_p), ("m2", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("status", ctypes.c_void_p), ("mean_bf16", ctypes.c_void_p),
                ("m2_bf16", ctypes.c_void_p)]


class WorkspaceView(ctypes.Structure):
    _fields_ = [("bbox_u", ctypes.c_size_t), ("bbox_uhat", ctypes.c_size_t),
                ("gauss_ms", ctypes.c_size_t), ("tauhat", ctypes.c_size_t),
                ("sel_bitmap", ctypes.c_size_t), ("tauhat_iters", ctypes.c_size_t),
                ("page_zmax", ctypes.c_size_t),
                ("cap_pages", ctypes.c_int32), ("splits", ctypes.c_int32),
                ("total", ctypes.c_size_t), ("z_scores", ctypes.c_size_t)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libentmaxkv.so (build it with ``python -m sparse_entmax_attention_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libentmaxkv.so not built ({LIB_PATH}); run "
                          "`python -m sparse_entmax_attention_gb300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, u32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t
    L.entmaxkv_version.restype = i32
    L.entmaxkv_status_string.restype = ctypes.c_char_p
    L.entmaxkv_status_string.argtypes = [i32]
    L.entmaxkv_append.restype = i32
    L.entmaxkv_append.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(CacheView), vp, vp, vp, i32, i32, vp]
    L.entmaxkv_workspace_bytes.restype = sz
    L.entmaxkv_workspace_bytes.argtypes = [ctypes.POINTER(Config), i32, i32, i32]
    L.entmaxkv_workspace_bytes_flags.restype = sz
    L.entmaxkv_workspace_bytes_flags.argtypes = [ctypes.POINTER(Config), i32, i32, i32, ctypes.c_uint32]
    L.entmaxkv_delta_kind.restype = i32
    L.entmaxkv_delta_kind.argtypes = [i32, ctypes.c_uint32]
    L.entmaxkv_read_status.restype = i32
    L.entmaxkv_read_status.argtypes = [ctypes.POINTER(CacheView), ctypes.POINTER(ctypes.c_uint32), i32, vp]
    L.entmaxkv_gaussian_alpha_supported.restype = i32
    L.entmaxkv_gaussian_alpha_supported.argtypes = [ctypes.c_float]
    L.entmaxkv_moment_fit_eval.restype = i32
    L.entmaxkv_moment_fit_eval.argtypes = [ctypes.c_float, i32, vp, i32, vp]
    L.entmaxkv_decode.restype = i32
    L.entmaxkv_decode.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(CacheView), vp, vp, i32,
                                  f32, i32, i32, f32, u32, vp, sz, vp, vp, i32, vp, vp, vp, vp]
    L.entmaxkv_decode_profiled.restype = i32
    L.entmaxkv_decode_profiled.argtypes = L.entmaxkv_decode.argtypes + [ctypes.POINTER(ctypes.c_void_p)]
    L.entmaxkv_noalloc_scratch_bytes.restype = sz
    L.entmaxkv_noalloc_scratch_bytes.argtypes = []
    L.entmaxkv_decode_softmax_noalloc.restype = i32
    L.entmaxkv_decode_softmax_noalloc.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(CacheView),
                                                  vp, vp, i32, vp, vp, vp]
    L.entmaxkv_workspace_layout.restype = i32
    L.entmaxkv_workspace_layout.argtypes = [ctypes.POINTER(Config), i32, i32, i32,
                                            ctypes.POINTER(WorkspaceView)]
    _lib = L
    return L


class EntmaxKVError(RuntimeError):
    pass


def _check(code: int):
    if code != 0:
        raise EntmaxKVError(f"entmaxkv: {lib().entmaxkv_status_string(code).decode()} (code {code})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


_DT = {torch.float32: F32, torch.bfloat16: BF16}


class PagedCache:
    """Caller-owned paged KV cache plus per-page key metadata (torch memory).

    meta_bf16: also keep bf16 copies of the page means and m2, which the
    Gaussian scorer then streams instead of the fp32 arrays.
    """

    def __init__(self, num_kv_heads, group, head_dim, page_size, max_seqs, max_pages_per_seq,
                 num_phys_pages, kv_dtype=torch.bfloat16, device="cuda", meta_bf16=False):
        self.cfg = Config(num_kv_heads, group, head_dim, page_size, max_seqs,
                          max_pages_per_seq, num_phys_pages, _DT[kv_dtype])
        self.dtype, self.device = kv_dtype, torch.device(device)
        Hkv, d, P = num_kv_heads, head_dim, page_size
        self.k_pool = torch.zeros(num_phys_pages, Hkv, P, d, dtype=kv_dtype, device=device)
        self.v_pool = torch.zeros_like(self.k_pool)
        self.kmin = torch.zeros(num_phys_pages, Hkv, d, dtype=kv_dtype, device=device)
        self.kmax = torch.zeros_like(self.kmin)
        self.mean = torch.zeros(num_phys_pages, Hkv, d, dtype=torch.float32, device=device)
        self.m2 = torch.zeros_like(self.mean)
        self.block_table = torch.zeros(max_seqs, max_pages_per_seq, dtype=torch.int32, device=device)
        self.seq_lens = torch.zeros(max_seqs, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.mean_bf16 = self.m2_bf16 = None
        if meta_bf16:
            self.mean_bf16 = torch.zeros(num_phys_pages, Hkv, d, dtype=torch.bfloat16, device=device)
            self.m2_bf16 = torch.zeros_like(self.mean_bf16)
        self.view = CacheView(self.k_pool.data_ptr(), self.v_pool.data_ptr(), self.kmin.data_ptr(),
                              self.kmax.data_ptr(), self.mean.data_ptr(), self.m2.data_ptr(),
                              self.block_table.data_ptr(), self.seq_lens.data_ptr(),
                              self.status.data_ptr(),
                              self.mean_bf16.data_ptr() if meta_bf16 else None,
                              self.m2_bf16.data_ptr() if meta_bf16 else None)

    def fp32_metadata(self) -> "PagedCache":
        """The same cache seen without its bf16 metadata copies (the Gaussian
        scorer then streams the fp32 mean and m2); tensors are shared."""
        other = copy.copy(self)
        other.view = CacheView(*[getattr(self.view, f) for f, _ in CacheView._fields_])
        other.view.mean_bf16 = None
        other.view.m2_bf16 = None
        other.mean_bf16 = None  # (this view streams none; self keeps the tensors alive)
        other.m2_bf16 = None
        return other

    @property
    def num_q_heads(self):
        return self.cfg.num_kv_heads * self.cfg.group

    def device_status(self) -> int:
        return int(self.status.item()) & 0xffffffff

    def read_status(self, clear=False, stream=None) -> int:
        """entmaxkv_read_status: the ENTMAXKV_DEV_* bits after the stream's work."""
        out = ctypes.c_uint32(0)
        _check(lib().entmaxkv_read_status(ctypes.byref(self.view), ctypes.byref(out), int(bool(clear)),
                                          _stream(stream)))
        return int(out.value)


def append(cache: PagedCache, k, v, seq_ids=None, stream=None):
    """entmaxkv_append: k, v [n_seqs, Hkv, n_tokens, d] in the cache dtype."""
    assert k.is_contiguous() and v.is_contiguous() and k.dtype == cache.dtype
    n_seqs, _, n_tok, _ = k.shape
    _check(lib().entmaxkv_append(ctypes.byref(cache.cfg), ctypes.byref(cache.view), _ptr(k),
                                 _ptr(v), _ptr(seq_ids), n_seqs, n_tok, _stream(stream)))


def workspace_bytes(cache: PagedCache, n_seqs, policy, budget_tokens=0, flags=0) -> int:
    return int(lib().entmaxkv_workspace_bytes_flags(ctypes.byref(cache.cfg), n_seqs,
                                                    POLICIES.get(policy, policy), budget_tokens,
                                                    int(flags)))


def delta_kind(policy, flags=0) -> int:
    return int(lib().entmaxkv_delta_kind(POLICIES.get(policy, policy), int(flags)))


def workspace_layout(cache: PagedCache, n_seqs, policy, budget_tokens=0) -> WorkspaceView:
    v = WorkspaceView()
    _check(lib().entmaxkv_workspace_layout(ctypes.byref(cache.cfg), n_seqs,
                                           POLICIES.get(policy, policy), budget_tokens,
                                           ctypes.byref(v)))
    return v


def alloc_workspace(cache: PagedCache, n_seqs, policy, budget_tokens=0, flags=0):
    n = workspace_bytes(cache, n_seqs, policy, budget_tokens, flags)
    if n == 0:
        raise EntmaxKVError("invalid decode arguments for workspace sizing")
    return torch.empty(n, dtype=torch.uint8, device=cache.device)  # caching allocator: 256-B aligned


@dataclass
class DecodeOutputs:
    out: torch.Tensor
    page_ids: torch.Tensor
    n_sel: torch.Tensor
    tau: torch.Tensor
    delta: torch.Tensor


def page_capacity(cache: PagedCache, policy, budget_tokens) -> int:
    p = POLICIES.get(policy, policy)
    maxp, P = cache.cfg.max_pages_per_seq, cache.cfg.page_size
    if p in (POLICY_TOPK, POLICY_SOFTMAX_TOPK):
        return min(budget_tokens // P, maxp)
    if p == POLICY_GAUSSIAN and budget_tokens > 0:
        return min(budget_tokens // P, maxp)
    return maxp


def alloc_outputs(cache: PagedCache, n_seqs, policy, budget_tokens=0) -> DecodeOutputs:
    dev, Hq, Hkv = cache.device, cache.num_q_heads, cache.cfg.num_kv_heads
    cap = page_capacity(cache, policy, budget_tokens)
    return DecodeOutputs(
        out=torch.empty(n_seqs, Hq, cache.cfg.head_dim, dtype=torch.float32, device=dev),
        page_ids=torch.full((n_seqs, Hkv, cap), -1, dtype=torch.int32, device=dev),
        n_sel=torch.empty(n_seqs, Hkv, dtype=torch.int32, device=dev),
        tau=torch.empty(n_seqs, Hq, dtype=torch.float32, device=dev),
        delta=torch.empty(n_seqs, Hq, dtype=torch.float32, device=dev))


def decode(cache: PagedCache, q, alpha=1.5, policy="gaussian", budget_tokens=0, margin=0.0,
           flags=0, seq_ids=None, workspace=None, outputs: DecodeOutputs | None = None,
           stream=None, events=None) -> DecodeOutputs:
    """entmaxkv_decode: q [n_seqs, Hq, d] in the cache dtype.

    With ``events`` (STAGE_EVENTS torch.cuda.Event objects) this calls
    entmaxkv_decode_profiled, which records them between the stages.
    """
    assert q.is_contiguous() and q.dtype == cache.dtype
    n_seqs = q.shape[0]
    pol = POLICIES.get(policy, policy)
    if workspace is None:
        workspace = alloc_workspace(cache, n_seqs, pol, budget_tokens, flags)
    if outputs is None:
        outputs = alloc_outputs(cache, n_seqs, pol, budget_tokens)
    o = outputs
    args = [ctypes.byref(cache.cfg), ctypes.byref(cache.view), _ptr(q), _ptr(seq_ids), n_seqs,
            float(alpha), pol, int(budget_tokens), float(margin), int(flags), _ptr(workspace),
            workspace.numel(), _ptr(o.out), _ptr(o.page_ids), o.page_ids.shape[-1], _ptr(o.n_sel),
            _ptr(o.tau), _ptr(o.delta), _stream(stream)]
    if events is None:
        _check(lib().entmaxkv_decode(*args))
    else:
        assert len(events) == STAGE_EVENTS
        arr = (ctypes.c_void_p * STAGE_EVENTS)(*[ctypes.c_void_p(e.cuda_event) for e in events])
        _check(lib().entmaxkv_decode_profiled(*args, arr))
    return o


class DecodeStep:
    """One serving step, append one token per sequence and decode, captured
    once as CUDA graphs of the library's launches over fixed buffers.

    `run(k, v, q)` takes device tensors: it copies them into the step's
    buffers and replays the launches. `run_host(k, v, q)` takes host tensors:
    they are copied into one pinned staging buffer, and a second graph moves
    them to the device in one copy, runs the launches and returns out, τ, δ
    and n_sel to pinned host memory in one copy; it returns those host views
    once the step is done. Capturing launches nothing: the cache changes only
    on replay. Arguments as for `append` and `decode`; k and v are
    [n_seqs, Hkv, 1, d], q is [n_seqs, Hq, d]."""

    def __init__(self, cache: PagedCache, n_seqs, alpha=1.5, policy="gaussian", budget_tokens=0,
                 margin=0.0, flags=0, seq_ids=None):
        dev, d = cache.device, cache.cfg.head_dim
        self.cache = cache
        Hkv, Hq = cache.cfg.num_kv_heads, cache.num_q_heads
        el = torch.tensor([], dtype=cache.dtype).element_size()
        shapes_in = [(n_seqs, Hkv, 1, d), (n_seqs, Hkv, 1, d), (n_seqs, Hq, d)]
        n_in = [int(torch.Size(sh).numel()) * el for sh in shapes_in]
        self.dev_in = torch.zeros(sum(n_in), dtype=torch.uint8, device=dev)
        self.host_in = torch.zeros(sum(n_in), dtype=torch.uint8).pin_memory()

        def views(buf):
            out, off = [], 0
            for sh, n in zip(shapes_in, n_in):
                out.append(buf[off:off + n].view(cache.dtype).view(sh))
                off += n
            return out

        self.k, self.v, self.q = views(self.dev_in)
        self._hk, self._hv, self._hq = views(self.host_in)
        # outputs: out, τ, δ, n_sel packed in one buffer (one copy back); page ids apart
        cap = page_capacity(cache, policy, budget_tokens)
        shapes_out = [((n_seqs, Hq, d), torch.float32), ((n_seqs, Hq), torch.float32),
                      ((n_seqs, Hq), torch.float32), ((n_seqs, Hkv), torch.int32)]
        n_out = [int(torch.Size(sh).numel()) * 4 for sh, _ in shapes_out]
        self.dev_out = torch.zeros(sum(n_out), dtype=torch.uint8, device=dev)
        self.host_out = torch.zeros(sum(n_out), dtype=torch.uint8).pin_memory()

        def out_views(buf):
            res, off = [], 0
            for (sh, dt), n in zip(shapes_out, n_out):
                res.append(buf[off:off + n].view(dt).view(sh))
                off += n
            return res

        out, tau, delta, n_sel = out_views(self.dev_out)
        self.outputs = DecodeOutputs(out=out, tau=tau, delta=delta, n_sel=n_sel,
                                     page_ids=torch.full((n_seqs, Hkv, cap), -1, dtype=torch.int32, device=dev))
        self.host_outputs = out_views(self.host_out)
        self.workspace = alloc_workspace(cache, n_seqs, policy, budget_tokens, flags)
        args = (alpha, policy, budget_tokens, margin, flags)

        def launches():
            append(cache, self.k, self.v, seq_ids=seq_ids)
            decode(cache, self.q, *args, seq_ids=seq_ids, workspace=self.workspace, outputs=self.outputs)

        # one decode outside the captures: first-launch set-up (shared-memory
        # attributes, moment fits) happens here, and no token is appended
        decode(cache, self.q, *args, seq_ids=seq_ids, workspace=self.workspace, outputs=self.outputs)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            launches()
        self.graph_io = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph_io):
            self.dev_in.copy_(self.host_in, non_blocking=True)
            launches()
            self.host_out.copy_(self.dev_out, non_blocking=True)

    def run(self, k, v, q) -> DecodeOutputs:
        """Device tensors in; the outputs stay on the device."""
        self.k.copy_(k, non_blocking=True)
        self.v.copy_(v, non_blocking=True)
        self.q.copy_(q, non_blocking=True)
        self.graph.replay()
        return self.outputs

    def run_host(self, k, v, q, wait=True):
        """Host tensors in; returns (out, τ, δ, n_sel) as pinned host tensors.
        With wait=True the call returns once the step has finished; with
        wait=False the caller synchronises the current stream before reading
        them (and before the next call reuses the staging buffer)."""
        self._hk.copy_(k)
        self._hv.copy_(v)
        self._hq.copy_(q)
        self.graph_io.replay()
        if wait:
            torch.cuda.current_stream(self.cache.device).synchronize()
        return self.host_outputs


def stage_events():
    """STAGE_EVENTS timing events with their CUDA handles already created."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(STAGE_EVENTS)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    return evs


def gaussian_alpha_supported(alpha: float) -> bool:
    """entmaxkv_gaussian_alpha_supported (host only)."""
    return bool(lib().entmaxkv_gaussian_alpha_supported(float(alpha)))


def moment_fit_eval(alpha: float, order: int, t):
    """entmaxkv_moment_fit_eval: the fitted J_ν(t), ν = β − order, on the host
    in the kernels' float arithmetic. t: 1-d float32 array-like."""
    import numpy as np
    ta = np.ascontiguousarray(np.asarray(t, dtype=np.float32))
    out = np.empty_like(ta)
    _check(lib().entmaxkv_moment_fit_eval(float(alpha), int(order), ta.ctypes.data_as(ctypes.c_void_p),
                                          int(ta.size), out.ctypes.data_as(ctypes.c_void_p)))
    return out
