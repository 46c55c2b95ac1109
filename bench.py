#!/usr/bin/env python
"""EntmaxKV decode-step benchmark on one GB300 (or N independent replicas).

One step = append one new token to every sequence (page write + metadata
update) and decode it with the Gaussian-aware selector (Δ = 0.5): page
scoring, τ̂ solve and selection, sparse α-entmax over the kept pages. The
workload is the 1M-token GQA cache (32 query / 8 KV heads, d = 128, page 32,
bf16 K/V; seeded synthetic data). Besides the headline step the run times the
top-k policy (2048 tokens), the full-cache entmax decode and the full-cache
softmax decode on the same cache, the dominant kernel on its own stream, an
end-to-end step from pinned host buffers, and the float64 oracle on a bounded
sample of host cores.

Prints one JSON line (rank 0). `--impl reference` times the oracle instead.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "μs/decode step and KV GB/s at 1M ctx; fraction of 8 TB/s HBM roofline"
WORKLOAD = "gqa32x8-d128-1m-p32-bf16"
ALPHA, MARGIN, TOPK_BUDGET = 1.5, 0.5, 2048
NOMINAL_HBM_GBS = 8000.0
L2_FLUSH_BYTES = 512 << 20   # > 129 MB L2: read between timed steps
# DRAM bytes (read + write) of one launch of the dominant kernel on this
# workload: an ncu capture of the same kernel on a 512k-token cache of the
# same shape (67,208,704 B read, 497,152 B written; reads 1.001 x that
# launch's metadata bytes) scaled by the page count to 1M; reset to None
# whenever that kernel changes.
NCU_TRAFFIC_PER_LAUNCH = 2 * (67208704 + 497152)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="headline step only")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the timed rows of the other synthetic workloads")
    ap.add_argument("--policies", default="gaussian,gaussian_meta_f32,gaussian_alpha1.25,topk,softmax_topk,full_dense,full_skipv,softmax",
                    help="rows of the per-policy table")
    return ap.parse_args()


# --------------------------------------------------------------------------
# clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------
# our arm

def algorithmic_bytes(wl, policy, o, ws, view):
    """Bytes the method must move for one decode (page metadata it scans,
    K pages it gathers, V pages with some p > 0, q in, outputs out)."""
    import torch
    spec, cache = wl.spec, wl.cache
    P, d, Hkv, G = spec.page_size, spec.head_dim, spec.num_kv_heads, spec.group
    el = torch.tensor([], dtype=spec.kv_dtype).element_size()
    n_pages = sum(-(-int(L) // P) for L in cache.seq_lens.tolist())
    page_kv = P * d * el                           # one (page, KV head) slab
    io = spec.batch * spec.num_q_heads * d * (el + 4) + spec.batch * spec.num_q_heads * 8
    if policy in ("full_dense", "softmax"):
        return 2 * n_pages * Hkv * page_kv + io, {"k_pages": n_pages * Hkv, "v_pages": n_pages * Hkv}
    meta = 0
    if policy in ("gaussian", "gaussian_alpha1.25"):  # mean + m2: the bf16 copies when the cache keeps them
        meta = n_pages * Hkv * d * (2 if cache.mean_bf16 is not None else 4) * 2
    elif policy == "gaussian_meta_f32":
        meta = n_pages * Hkv * d * 4 * 2
    elif policy in ("topk", "softmax_topk"):
        meta = n_pages * Hkv * d * el * 2          # kmin + kmax
    n_sel = o.n_sel.cpu()
    k_pages = int(n_sel.sum())
    if policy == "softmax_topk":                   # softmax reads V of every kept page
        return meta + 2 * k_pages * page_kv + io, {"k_pages": k_pages, "v_pages": k_pages,
                                                   "meta_bytes": meta}
    # V pages actually read: some head's page max z above its τ
    cap = view.cap_pages
    pm = ws[view.page_zmax: view.page_zmax + spec.batch * Hkv * cap * G * 4].view(torch.float32)
    pm = pm.view(spec.batch, Hkv, cap, G).cpu()
    tau = o.tau.view(spec.batch, Hkv, G).cpu()
    v_pages = 0
    for b in range(spec.batch):
        for j in range(Hkv):
            n = int(n_sel[b, j])
            if policy == "full_skipv":
                n = -(-int(cache.seq_lens[b]) // P)
            v_pages += int((pm[b, j, :n] > tau[b, j][None, :]).any(dim=1).sum())
    return meta + (k_pages + v_pages) * page_kv + io, {"k_pages": k_pages, "v_pages": v_pages,
                                                       "meta_bytes": meta}


def run_ours(args, rank, world):
    import torch
    from sparse_entmax_attention_gb300 import binding as B
    from sparse_entmax_attention_gb300 import replicas, runner, synth

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    K, W = args.steps, args.warmup
    spec = synth.workload(WORKLOAD)
    n_append = 4 * (K + W) + 8  # the timed steps, then the eager and the captured e2e steps
    wl = runner.Workload(spec, seed=0, device=dev, extra_steps=n_append, meta_bf16=True)
    cache = wl.cache
    peaks, peak_kind = measured_peaks()
    # inputs of every step, resident in HBM before timing
    toks = [wl.step_tokens(i) for i in range(n_append)]
    # every step decodes with the workload's query (the one its needles were
    # planted for); one new token per step
    qs = [wl.q for i in range(K + W)]
    kbuf, vbuf = toks[0][0].clone(), toks[0][1].clone()
    qbuf = qs[0].clone()
    flush_buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    flush_out = torch.empty((), dtype=torch.int64, device=dev)

    class _Flush:
        # Reading 512 MiB evicts everything the previous step left in the
        # 129 MB L2 without leaving dirty lines behind to be written back.
        @staticmethod
        def zero_():
            torch.sum(flush_buf, dim=0, dtype=torch.int64, out=flush_out)

    flush = _Flush()
    n_app = [0]

    def set_step(i):
        kbuf.copy_(toks[n_app[0]][0])
        vbuf.copy_(toks[n_app[0]][1])
        qbuf.copy_(qs[i % len(qs)])

    ws_g = B.alloc_workspace(cache, spec.batch, "gaussian", 0)
    out_g = B.alloc_outputs(cache, spec.batch, "gaussian", 0)

    def step():
        B.append(cache, kbuf, vbuf)
        B.decode(cache, qbuf, ALPHA, "gaussian", 0, MARGIN, workspace=ws_g, outputs=out_g)

    # eager warm-up (also loads every kernel), then capture one step as a graph
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        set_step(0)
        step()
        n_app[0] += 1
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    def timed(fn, n, tag_steps):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            tag_steps(i)
            flush.zero_()
            starts[i].record()
            fn()
            ends[i].record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) * 1e3 for a, b in zip(starts, ends)]  # μs

    def adv(i):
        set_step(i)
        n_app[0] += 1

    # graph capture appended nothing (capture does not execute); the counter
    # tracks the appends the replays perform.
    timed(graph.replay, W, adv)
    torch.cuda.synchronize()
    replicas.barrier()
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    clk.start()
    t0 = time.perf_counter()
    step_us = timed(graph.replay, K, lambda i: adv(W + i))
    replicas.barrier()
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    clocks = clk.stop()
    mean_us = replicas.max_over_ranks(statistics.mean(step_us), device=dev)
    assert cache.device_status() & ~B.DEV_CAND_OVERFLOW == 0, hex(cache.device_status())

    view_g = B.workspace_layout(cache, spec.batch, "gaussian", 0)
    bytes_g, counts_g = algorithmic_bytes(wl, "gaussian", out_g, ws_g, view_g)
    append_bytes = spec.batch * spec.num_kv_heads * spec.head_dim * (2 * 2 + 2 * 2 + 2 * 4 * 2)
    step_bytes = bytes_g + append_bytes
    res = {
        "metric": METRIC,
        "value": round(mean_us, 2),
        "unit": "us/step",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(mean_us / 1e3, 5),
        "steps_per_s_all_ranks": round(world * 1e6 / mean_us, 1),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded generator: page centroids + noise, needles, outlier channels)",
        "config": {"workload": WORKLOAD, "batch": 1, "context": spec.context_lens[0],
                   "q_heads": spec.num_q_heads, "kv_heads": spec.num_kv_heads,
                   "head_dim": spec.head_dim, "page_size": spec.page_size, "alpha": ALPHA,
                   "policy": "gaussian", "margin": MARGIN,
                   "metadata": "fp32 mean/m2 kept for appends; their bf16 copies streamed by the scorer",
                   "step": "append 1 token + Gaussian-selector decode (CUDA graph)",
                   "queries": "the workload's decode queries (needles planted for them)",
                   "l2": "flushed between timed steps by reading a 512 MiB buffer; per-step CUDA events",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "kv_gbs": round(step_bytes / (mean_us * 1e-6) / 1e9, 1),
        "frac_8tbs": round(step_bytes / (mean_us * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 4),
        "frac_measured_hbm": round(step_bytes / (mean_us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
        "bytes_per_step": step_bytes,
        "selected": counts_g,
        "wall_s_timed_loop": round(wall, 4),
        "gpu_launches": 5 * K,  # per step: append, scoring, τ̂ + bits, pass A, pass B
        "clocks": clocks,
    }
    if rank != 0:
        return None
    if not args.no_extras:
        res["policies"] = policy_table(wl, B, flush, qbuf, timed, K, peaks, args.policies.split(","))
        res["dropped_mass_exact"] = dropped_mass(wl, B, qbuf)
        res["roofline"] = roofline(wl, B, flush, qbuf, K, peaks, peak_kind)
        res["prefill"] = prefill(wl, B, K, W, peaks)
        if not args.no_e2e:
            res["e2e"] = e2e(wl, B, toks, qs, n_app, K, W)
    del ws_g, out_g, graph
    if not args.no_workloads:
        res["workloads"] = workload_rows(B, flush, min(K, 20), peaks, dev)
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, qbuf)
    return res


def policy_table(wl, B, flush, qbuf, timed, K, peaks, names):
    import torch
    cache, spec = wl.cache, wl.spec
    rows = {}
    # (name, policy, budget, flags, α); α = 1.25 runs the selector on the
    # fitted partial moments of order β = 4
    cases = [("gaussian", "gaussian", 0, 0, ALPHA), ("gaussian_meta_f32", "gaussian", 0, 0, ALPHA),
             ("gaussian_alpha1.25", "gaussian", 0, 0, 1.25),
             ("topk", "topk", TOPK_BUDGET, 0, ALPHA),
             ("softmax_topk", "softmax_topk", TOPK_BUDGET, 0, ALPHA),
             ("full_dense", "full", 0, B.FLAG_DENSE_V, ALPHA), ("full_skipv", "full", 0, 0, ALPHA),
             ("softmax", "softmax", 0, 0, ALPHA)]
    for name, pol, budget, flags, alpha in cases:
        if name not in names:
            continue
        c = cache.fp32_metadata() if name == "gaussian_meta_f32" else cache
        ws = B.alloc_workspace(c, spec.batch, pol, budget)
        o = B.alloc_outputs(c, spec.batch, pol, budget)
        fn = lambda: B.decode(c, qbuf, alpha, pol, budget, MARGIN, flags, workspace=ws, outputs=o)
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        us = timed(g.replay, K, lambda i: None)
        mean = statistics.mean(us)
        view = B.workspace_layout(cache, spec.batch, pol, budget)
        nbytes, counts = algorithmic_bytes(wl, name, o, ws, view)
        evs = B.stage_events()
        flush.zero_()
        B.decode(c, qbuf, alpha, pol, budget, MARGIN, flags, workspace=ws, outputs=o, events=evs)
        torch.cuda.synchronize()
        stage = {n: round(evs[k].elapsed_time(evs[k + 1]) * 1e3, 1) for k, n in enumerate(B.STAGES)}
        rows[name] = {"us": round(mean, 2), "bytes": nbytes, "stage_us_once": stage,
                      "gbs": round(nbytes / (mean * 1e-6) / 1e9, 1),
                      "frac_8tbs": round(nbytes / (mean * 1e-6) / 1e9 / NOMINAL_HBM_GBS, 4),
                      **counts}
        del ws
    for name in ("gaussian_meta_f32", "topk", "softmax_topk", "full_dense", "full_skipv", "softmax"):
        if name in rows and "gaussian" in rows:
            rows[name]["gaussian_speedup"] = round(rows[name]["us"] / rows["gaussian"]["us"], 2)
    return rows


def dropped_mass(wl, B, qbuf):
    """Exact dropped mass δ per query head (untimed, ENTMAXKV_FLAG_EXACT_DELTA)
    of entmax top-k, softmax top-k at the same budget, and the Gaussian
    selector: how much of the full-cache attention each kept set loses."""
    import torch
    cache, spec = wl.cache, wl.spec
    res = {"budget_tokens": TOPK_BUDGET}
    kinds = {B.DELTA_CERTIFIED: "certified bound", B.DELTA_MODEL: "model estimate", B.DELTA_EXACT: "exact"}
    for name, pol, budget in (("entmax_topk", "topk", TOPK_BUDGET),
                              ("softmax_topk", "softmax_topk", TOPK_BUDGET), ("gaussian", "gaussian", 0)):
        o = B.decode(cache, qbuf, ALPHA, pol, budget, MARGIN, B.FLAG_EXACT_DELTA)
        torch.cuda.synchronize()
        dl = o.delta.float().cpu()
        # the δ a decode returns without the flag, beside the exact one
        r = B.decode(cache, qbuf, ALPHA, pol, budget, MARGIN)
        torch.cuda.synchronize()
        dr = r.delta.float().cpu()
        res[name] = {"mean": round(float(dl.mean()), 5), "max": round(float(dl.max()), 5),
                     "reported_kind": kinds.get(B.delta_kind(pol), "?"),
                     "reported_mean": round(float(dr.mean()), 5), "reported_max": round(float(dr.max()), 5),
                     "pages_per_kv_head": round(float(o.n_sel.float().mean()), 1)}
    return res


def prefill(wl, B, K, W, peaks):
    """Bulk prefill of the whole context of sequence 0 into a second cache of
    the same shape (same block table, bf16 metadata copies on): one
    entmaxkv_append that writes every token and builds every page's bounding
    box, mean, m2 and their bf16 copies in the same kernel. Inputs are
    device-resident synthetic keys and values (4.3 GB at 1M tokens, far above
    L2); before each timed append the length is reset to 0, so every page is
    new and its metadata is built from scratch."""
    import torch
    spec, dev = wl.spec, wl.cache.device
    L, P, Hkv, d = spec.context_lens[0], spec.page_size, spec.num_kv_heads, spec.head_dim
    c = B.PagedCache(Hkv, spec.group, d, P, 1, wl.cache.block_table.shape[1], wl.cache.cfg.num_phys_pages,
                     spec.kv_dtype, dev, meta_bf16=True)
    c.block_table[0].copy_(wl.cache.block_table[0])
    g = torch.Generator(device=dev)
    g.manual_seed(12345)
    k = torch.randn(1, Hkv, L, d, generator=g, device=dev, dtype=spec.kv_dtype)
    v = torch.randn(1, Hkv, L, d, generator=g, device=dev, dtype=spec.kv_dtype)
    us = []
    for i in range(W + K):
        c.seq_lens.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        B.append(c, k, v)
        b.record()
        torch.cuda.synchronize()
        if i >= W:
            us.append(a.elapsed_time(b) * 1e3)
    assert c.device_status() == 0, hex(c.device_status())
    n_pages = -(-L // P)
    esz = torch.tensor([], dtype=spec.kv_dtype).element_size()
    # read k, v; write them into the pool; per (page, KV head): kmin, kmax in the
    # KV dtype, mean and m2 in fp32, their bf16 copies
    nbytes = 4 * Hkv * L * d * esz + Hkv * n_pages * d * (2 * esz + 2 * 4 + 2 * 2)
    mean = statistics.mean(us)
    gbs = nbytes / (mean * 1e-6) / 1e9
    del c, k, v
    return {"us": round(mean, 1), "tokens": L, "tokens_per_s": round(L / (mean * 1e-6), 1),
            "bytes": nbytes, "gbs": round(gbs, 1), "frac_measured_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "steps": K, "what": "one bulk entmaxkv_append of the whole context (tokens + page metadata)"}


def roofline(wl, B, flush, qbuf, K, peaks, peak_kind):
    """Dominant kernel = Gaussian page scoring (streams mean + m2 of every
    page): its per-launch time from CUDA events recorded around it on the
    stream it runs on (the library's stage-timed decode)."""
    import torch
    cache, spec = wl.cache, wl.spec
    ws = B.alloc_workspace(cache, spec.batch, "gaussian", 0)
    o = B.alloc_outputs(cache, spec.batch, "gaussian", 0)
    view = B.workspace_layout(cache, spec.batch, "gaussian", 0)
    evs = B.stage_events()
    per = {n: [] for n in B.STAGES}
    for i in range(K + 1):
        flush.zero_()
        B.decode(cache, qbuf, ALPHA, "gaussian", 0, MARGIN, workspace=ws, outputs=o, events=evs)
        torch.cuda.synchronize()
        if i == 0:
            continue
        for k, n in enumerate(B.STAGES):
            per[n].append(evs[k].elapsed_time(evs[k + 1]) * 1e3)
    stages = {n: round(statistics.mean(v), 2) for n, v in per.items()}
    n_pages = -(-int(cache.seq_lens[0]) // spec.page_size)
    el = 2 if cache.mean_bf16 is not None else 4             # the metadata the scorer streams
    alg = n_pages * spec.num_kv_heads * spec.head_dim * el * 2  # mean + m2 bytes per launch
    t = stages["score"] * 1e-6
    ach = alg / t / 1e9
    it = ws[view.tauhat_iters: view.tauhat_iters + spec.batch * spec.num_q_heads * 4].view(torch.int32)
    kname = ("gauss_mma_kernel (Gaussian page scoring on the tensor cores, bf16 metadata)"
             if el == 2 else "gauss_kernel (Gaussian page scoring, fp32 metadata)")
    return {"kernel": kname, "bound": "hbm",
            "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / peaks["hbm_gbs"], 4), "peak_kind": peak_kind + " (copy, burst)",
            "traffic": NCU_TRAFFIC_PER_LAUNCH, "algorithmic_bytes": alg,
            "stage_us": stages, "tauhat_iters_mean": round(float(it.float().mean()), 2)}


def e2e(wl, B, toks, qs, n_app, K, W):
    """Same step through the public API from host buffers: H2D of the new
    token and the queries, append + decode, D2H of out/τ/δ/n_sel. The value
    is the library's captured serving step (`B.DecodeStep.run_host`: the
    inputs staged in pinned memory, one H2D copy, the launches and one D2H
    copy replayed from a CUDA graph, and the wait for the results); `eager`
    is the same step by one API call per operation, with one copy per
    tensor."""
    import torch
    cache, spec = wl.cache, wl.spec
    hk = [toks[n_app[0] + i][0].cpu().pin_memory() for i in range(2 * (K + W))]
    hv = [toks[n_app[0] + i][1].cpu().pin_memory() for i in range(2 * (K + W))]
    hq = [qs[i % len(qs)].cpu().pin_memory() for i in range(2 * (K + W))]
    dk, dv, dq = hk[0].cuda(), hv[0].cuda(), hq[0].cuda()
    ws = B.alloc_workspace(cache, spec.batch, "gaussian", 0)
    o = B.alloc_outputs(cache, spec.batch, "gaussian", 0)
    ho = [torch.empty_like(t, device="cpu").pin_memory() for t in (o.out, o.tau, o.delta, o.n_sel)]

    def eager(i):
        dk.copy_(hk[i], non_blocking=True)
        dv.copy_(hv[i], non_blocking=True)
        dq.copy_(hq[i], non_blocking=True)
        B.append(cache, dk, dv)
        B.decode(cache, dq, ALPHA, "gaussian", 0, MARGIN, workspace=ws, outputs=o)
        for h, d in zip(ho, (o.out, o.tau, o.delta, o.n_sel)):
            h.copy_(d, non_blocking=True)

    step = B.DecodeStep(cache, spec.batch, ALPHA, "gaussian", 0, MARGIN)

    def captured(i):  # the step's own copies: separate H2D / D2H around the graphed launches
        step.run(hk[i], hv[i], hq[i])
        for h, d in zip(ho, (step.outputs.out, step.outputs.tau, step.outputs.delta, step.outputs.n_sel)):
            h.copy_(d, non_blocking=True)

    def captured_io(i):  # staged inputs, one H2D, the launches and one D2H in one graph
        step.run_host(hk[i], hv[i], hq[i], wait=False)

    def timed(fn, i0):
        us = []
        for i in range(K + W):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn(i0 + i)
            b.record()
            b.synchronize()
            if i >= W:
                us.append(a.elapsed_time(b) * 1e3)
        return statistics.mean(us)

    v_eager = timed(eager, 0)
    v_graph = timed(captured, K + W)
    v_io = timed(captured_io, K + W)
    h2d = sum(t.numel() * t.element_size() for t in (hk[0], hv[0], hq[0]))
    d2h = sum(t.numel() * t.element_size() for t in ho)
    best = min(v_graph, v_io)
    return {"value": round(best, 2), "unit": "us/step",
            "path": "DecodeStep.run_host" if v_io <= v_graph else "DecodeStep.run + copies",
            "graph_dev": round(v_graph, 2),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "eager": round(v_eager, 2), "graph_io": round(v_io, 2),
            "how": "per-step CUDA events around H2D + append + decode + D2H, the GPU's own clock; "
                   "graph_dev: DecodeStep.run (an H2D per tensor, the graphed launches, a D2H per "
                   "tensor), graph_io: DecodeStep.run_host (staged inputs, one H2D, the launches and "
                   "one D2H in one graph), value: the faster of the two, eager: one API call and one "
                   "copy per tensor"}


# --------------------------------------------------------------------------
# the other synthetic workloads: timed rows and quality reports

def graph_of(fn):
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def time_replays(g, n, flush, before=None):
    """µs of n replays of graph g, each after `before(i)` (untimed input
    copies) and a 512 MiB L2-flushing read; CUDA events on the current stream."""
    import torch
    us = []
    for i in range(n):
        if before is not None:
            before(i)
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        us.append(a.elapsed_time(b) * 1e3)
    return us


class FullRef:
    """The full-cache α-entmax decode of the same queries (the library's own
    policy-full path): output, τ and every token's z, for the quality report."""

    def __init__(self, B, cache, q, alpha):
        import torch
        S = q.shape[0]
        self.ws = B.alloc_workspace(cache, S, "full")
        self.o = B.decode(cache, q, alpha, "full", workspace=self.ws)
        view = B.workspace_layout(cache, S, "full")
        cfg = cache.cfg
        shape = (S, cfg.num_kv_heads, view.cap_pages, cfg.page_size, cfg.group)
        n = 4 * math.prod(shape)
        torch.cuda.synchronize()
        self.z = self.ws[view.z_scores: view.z_scores + n].view(torch.float32).view(*shape)


def quality(B, cache, q, alpha, policy, budget, margin, o, ref):
    """δ (exact dropped mass, the library's EXACT_DELTA decode), support recall
    (the full-cache support's tokens inside the kept pages) and the relative
    L2 error of the output against the full-cache output, per query head;
    returned as means and extremes."""
    import torch
    S, Hq = q.shape[0], cache.num_q_heads
    Hkv, G = cache.cfg.num_kv_heads, cache.cfg.group
    ex = B.decode(cache, q, alpha, policy, budget, margin, B.FLAG_EXACT_DELTA)
    torch.cuda.synchronize()
    maxp = ref.z.shape[2]
    kept = torch.zeros(S, Hkv, maxp, dtype=torch.bool, device=q.device)
    n_sel = o.n_sel.long()
    for b in range(S):
        for j in range(Hkv):
            ids = o.page_ids[b, j, : int(n_sel[b, j])].long()
            kept[b, j, ids] = True
    tau_full = ref.o.tau.view(S, Hkv, 1, 1, G)
    supp = ref.z > tau_full                                    # [S, Hkv, maxp, P, G]
    n_supp = supp.sum(dim=(2, 3)).double()                      # [S, Hkv, G]
    n_hit = (supp & kept[:, :, :, None, None]).sum(dim=(2, 3)).double()
    recall = (n_hit / n_supp.clamp_min(1)).view(S, Hq)
    err = ((o.out - ref.o.out).norm(dim=-1) / ref.o.out.norm(dim=-1).clamp_min(1e-30)).view(S, Hq)
    d = ex.delta.float()
    return {"delta_exact_mean": round(float(d.mean()), 5), "delta_exact_max": round(float(d.max()), 5),
            "recall_mean": round(float(recall.mean()), 5), "recall_min": round(float(recall.min()), 5),
            "rel_err_mean": round(float(err.mean()), 6), "rel_err_max": round(float(err.max()), 6),
            "pages_per_kv_head": round(float(o.n_sel.float().mean()), 1)}


def timed_row(B, wl, q, alpha, policy, budget, margin, flags, flush, n, peaks, ref=None):
    """One policy on one workload: µs per decode (graph replay, L2 flushed),
    algorithmic bytes and GB/s, and the quality report against `ref`."""
    import torch
    cache, spec = wl.cache, wl.spec
    S = q.shape[0]
    ws = B.alloc_workspace(cache, S, policy, budget)
    o = B.alloc_outputs(cache, S, policy, budget)
    g = graph_of(lambda: B.decode(cache, q, alpha, policy, budget, margin, flags, workspace=ws, outputs=o))
    us = statistics.mean(time_replays(g, n, flush))
    view = B.workspace_layout(cache, S, policy, budget)
    name = "full_dense" if (policy == "full" and flags & B.FLAG_DENSE_V) else \
        ("full_skipv" if policy == "full" else policy)
    nbytes, counts = algorithmic_bytes(wl, name, o, ws, view)
    gbs = nbytes / (us * 1e-6) / 1e9
    row = {"us": round(us, 2), "bytes": nbytes, "gbs": round(gbs, 1),
           "frac_8tbs": round(gbs / NOMINAL_HBM_GBS, 4), "frac_measured_hbm": round(gbs / peaks["hbm_gbs"], 4),
           **counts}
    if ref is not None and policy not in ("full", "softmax"):
        row.update(quality(B, cache, q, alpha, policy, budget, margin, o, ref))
    del g
    return row


def workload_rows(B, flush, n, peaks, dev):
    """The four other synthetic workloads, each timed per decode step (CUDA
    graph replays, L2 flushed before each) with δ, support recall and
    relative output error of every selective policy against the full-cache
    α-entmax decode of the same query."""
    import torch
    from sparse_entmax_attention_gb300 import runner, synth
    rows = {}
    # 4k tokens, one head, d = 64, fp32: full vs top-k 32 pages (launch-bound sizes)
    spec = synth.workload("single-head-d64-4k-p16-fp32")
    wl = runner.Workload(spec, device=dev)
    ref = FullRef(B, wl.cache, wl.q, 1.5)
    rows[spec.name] = {
        "full_dense": timed_row(B, wl, wl.q, 1.5, "full", 0, 0.0, B.FLAG_DENSE_V, flush, n, peaks),
        "topk_512": timed_row(B, wl, wl.q, 1.5, "topk", 512, 0.0, 0, flush, n, peaks, ref),
        "note": "8 MB of K/V: launch-bound, the roofline fraction is not meaningful"}
    del wl, ref
    # 32k tokens, GQA 32/8, bf16: top-k 1024 tokens vs full
    spec = synth.workload("gqa32x8-d128-32k-p16-bf16")
    wl = runner.Workload(spec, device=dev)
    ref = FullRef(B, wl.cache, wl.q, 1.5)
    rows[spec.name] = {
        "full_dense": timed_row(B, wl, wl.q, 1.5, "full", 0, 0.0, B.FLAG_DENSE_V, flush, n, peaks),
        "softmax": timed_row(B, wl, wl.q, 1.5, "softmax", 0, 0.0, 0, flush, n, peaks),
        "topk_1024": timed_row(B, wl, wl.q, 1.5, "topk", 1024, 0.0, 0, flush, n, peaks, ref),
        "softmax_topk_1024": timed_row(B, wl, wl.q, 1.5, "softmax_topk", 1024, 0.0, 0, flush, n, peaks)}
    del wl, ref
    rows["gqa32x8-d128-128k-p32-bf16"] = rotated_steps(B, flush, peaks, dev)
    rows["batch16-loguniform-4k-256k-p16-bf16"] = batched_serving(B, flush, peaks, dev)
    torch.cuda.empty_cache()
    return rows


def rotated_steps(B, flush, peaks, dev):
    """128k tokens, page 32: 64 decode steps, each with fresh queries rotated
    30% toward a needle key. Gaussian selector at α ∈ {1.5, 2}, Δ ∈ {0, 0.5, 1},
    against top-k with its k matched to the Gaussian n_sel of the same step
    (mean over KV heads). µs per step from one graph replay per step."""
    import torch
    from sparse_entmax_attention_gb300 import runner, synth
    spec = synth.workload("gqa32x8-d128-128k-p32-bf16")
    wl = runner.Workload(spec, device=dev, meta_bf16=True)
    cache, P = wl.cache, spec.page_size
    qs = [wl.step_queries(i) for i in range(spec.steps)]
    qbuf = qs[0].clone()
    out = {"steps": spec.steps}
    for alpha in spec.extra["alphas"]:
        refs = []
        for i in range(spec.steps):
            qbuf.copy_(qs[i])
            r = FullRef(B, cache, qbuf, alpha)
            refs.append((r.o, r.z.clone()))  # per step: full output, τ and z
            del r
        for margin in spec.extra["margins"]:
            ws = B.alloc_workspace(cache, 1, "gaussian")
            o = B.alloc_outputs(cache, 1, "gaussian")
            g = graph_of(lambda: B.decode(cache, qbuf, alpha, "gaussian", 0, margin, workspace=ws, outputs=o))
            us_g, us_t, qual_g, qual_t, ksel, bytes_g = [], [], [], [], [], []
            graphs_t = {}
            for i in range(spec.steps):
                us_g += time_replays(g, 1, flush, lambda _i: qbuf.copy_(qs[i]))
                view = B.workspace_layout(cache, 1, "gaussian")
                bytes_g.append(algorithmic_bytes(wl, "gaussian", o, ws, view)[0])
                ref = _Ref(*refs[i])
                qual_g.append(quality(B, cache, qbuf, alpha, "gaussian", 0, margin, o, ref))
                k = max(1, int(round(float(o.n_sel.float().mean()))))
                ksel.append(k)
                if k not in graphs_t:
                    wt = B.alloc_workspace(cache, 1, "topk", k * P)
                    ot = B.alloc_outputs(cache, 1, "topk", k * P)
                    gt = graph_of(lambda: B.decode(cache, qbuf, alpha, "topk", k * P, 0.0, workspace=wt,
                                                   outputs=ot))
                    graphs_t[k] = (gt, wt, ot)
                gt, wt, ot = graphs_t[k]
                us_t += time_replays(gt, 1, flush)
                qual_t.append(quality(B, cache, qbuf, alpha, "topk", k * P, 0.0, ot, ref))
            mg, mt = statistics.mean(us_g), statistics.mean(us_t)
            gbs = statistics.mean(bytes_g) / (mg * 1e-6) / 1e9
            out[f"alpha{alpha}_margin{margin}"] = {
                "gaussian": {"us": round(mg, 2), "gbs": round(gbs, 1),
                             "frac_8tbs": round(gbs / NOMINAL_HBM_GBS, 4), **_mean_quality(qual_g)},
                "topk_matched": {"us": round(mt, 2), "pages_per_kv_head": round(statistics.mean(ksel), 1),
                                 **{k: v for k, v in _mean_quality(qual_t).items() if k != "pages_per_kv_head"}}}
            del g, graphs_t
    del wl
    return out


class _Ref:
    def __init__(self, o, z):
        self.o, self.z = o, z


def _mean_quality(rows):
    keys = rows[0].keys()
    agg = {}
    for k in keys:
        vals = [r[k] for r in rows]
        agg[k] = round(max(vals) if k.endswith("_max") else min(vals) if k.endswith("_min")
                       else statistics.mean(vals), 6)
    return agg


def batched_serving(B, flush, peaks, dev):
    """16 sequences (lengths log-uniform in [4096, 262144], shuffled block
    table, page 16): 128 steps, each appending one token to every sequence
    (page metadata updated in place) and decoding all 16 with the Gaussian
    selector (Δ = 0.5). µs per step from one graph replay per step; quality
    on every 32nd step."""
    import torch
    from sparse_entmax_attention_gb300 import runner, synth
    spec = synth.workload("batch16-loguniform-4k-256k-p16-bf16")
    wl = runner.Workload(spec, device=dev, meta_bf16=True)
    cache = wl.cache
    toks = [wl.step_tokens(i) for i in range(spec.steps)]
    qs = [wl.step_queries(i) for i in range(spec.steps)]
    kb, vb, qb = toks[0][0].clone(), toks[0][1].clone(), qs[0].clone()
    ws = B.alloc_workspace(cache, spec.batch, "gaussian")
    o = B.alloc_outputs(cache, spec.batch, "gaussian")

    def step():
        B.append(cache, kb, vb)
        B.decode(cache, qb, 1.5, "gaussian", 0, 0.5, workspace=ws, outputs=o)

    # kernels loaded by an eager decode (no state change), then the step is
    # captured without executing it: the first replay is step 0
    B.decode(cache, qb, 1.5, "gaussian", 0, 0.5, workspace=ws, outputs=o)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    torch.cuda.synchronize()

    def before(i):
        kb.copy_(toks[i][0])
        vb.copy_(toks[i][1])
        qb.copy_(qs[i])

    us, qual, nbytes = [], [], []
    view = B.workspace_layout(cache, spec.batch, "gaussian")
    for i in range(spec.steps):
        us += time_replays(g, 1, flush, lambda _i: before(i))
        nbytes.append(algorithmic_bytes(wl, "gaussian", o, ws, view)[0])
        if i % 32 == 31:
            ref = FullRef(B, cache, qb, 1.5)
            qual.append(quality(B, cache, qb, 1.5, "gaussian", 0, 0.5, o, ref))
            del ref
    assert cache.device_status() & ~B.DEV_CAND_OVERFLOW == 0, hex(cache.device_status())
    append_bytes = spec.batch * spec.num_kv_heads * spec.head_dim * (2 * 2 + 2 * 2 + 2 * 4 * 2)
    m = statistics.mean(us)
    gbs = (statistics.mean(nbytes) + append_bytes) / (m * 1e-6) / 1e9
    del g, wl
    return {"steps": spec.steps, "us_per_step": round(m, 2), "us_first": round(us[0], 2),
            "us_last": round(us[-1], 2), "tokens_per_s": round(spec.batch / (m * 1e-6), 1),
            "gbs": round(gbs, 1), "frac_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
            "frac_measured_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "context_tokens": sum(spec.context_lens), "quality_every_32_steps": _mean_quality(qual),
            "step": "append 1 token to each of 16 sequences + Gaussian decode of all 16 (CUDA graph)"}


# --------------------------------------------------------------------------
# oracle (CPU) legs

def host_sample(wl, qdev, kvh=0):
    """Stored K/V of one KV head (all pages, via the block table) and its g
    queries, as float64 host arrays."""
    import torch
    cache, spec = wl.cache, wl.spec
    L = int(cache.seq_lens[0])
    n_pages = -(-L // spec.page_size)
    phys = cache.block_table[0, :n_pages].long()
    K = cache.k_pool[phys, kvh].reshape(-1, spec.head_dim)[:L].double().cpu().numpy()
    V = cache.v_pool[phys, kvh].reshape(-1, spec.head_dim)[:L].double().cpu().numpy()
    g = spec.group
    Q = qdev[0, kvh * g:(kvh + 1) * g].double().cpu().numpy()
    return K, V, Q


def oracle_decode_step(heads, P):
    """One whole Gaussian decode step by the oracle: every KV head with its
    query heads; (K, V, Q, page metadata) per KV head."""
    from oracle import decode as odec
    for K, V, Q, meta in heads:
        odec.decode_group(K, V, Q, ALPHA, "gaussian", P, 0, MARGIN, meta=meta, diagnostics=False)


def oracle_heads_from_cache(wl, qdev):
    """The stored K/V bits of every KV head of the cache (as float32, exact for
    bf16) with the oracle's reading of the page statistics the GPU path
    streams (exact statistics rounded to bf16: the cache keeps bf16 copies)."""
    from oracle import pages as opg
    spec = wl.spec
    heads = []
    for kvh in range(spec.num_kv_heads):
        K, V, Q = host_sample(wl, qdev, kvh)
        K, V = K.astype("float32"), V.astype("float32")
        meta = opg.page_metadata(K, spec.page_size)
        heads.append((K, V, Q, opg.bf16_metadata(meta) if wl.cache.mean_bf16 is not None else meta))
    return heads


def cpu_baseline(wl, qdev, min_s=10.0, max_reps=3):
    """Whole Gaussian decode steps (every KV head and its query heads) by the
    oracle on the cache's stored bits, repeated until at least `min_s` seconds
    of oracle time."""
    spec = wl.spec
    heads = oracle_heads_from_cache(wl, qdev)   # the cache keeps the metadata: not per step
    per_step, total, reps = [], 0.0, 0
    while reps < max_reps and (reps == 0 or total < min_s):
        t0 = time.perf_counter()
        oracle_decode_step(heads, spec.page_size)
        dt = time.perf_counter() - t0
        per_step.append(dt)
        total += dt
        reps += 1
    us = statistics.mean(per_step) * 1e6
    return {"value": round(us, 1), "unit": "us/step", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{reps} x one whole Gaussian decode step at 1M tokens ({spec.num_kv_heads} KV "
                      f"heads x {spec.group} query heads) on the cache's stored bits, float64 numpy, "
                      f"{total:.1f} s of oracle time; page metadata prebuilt (the cache keeps it); "
                      f"BLAS default threads"}


def reference_inputs(K, W):
    """The bench's 1M-token workload with the same spec the GPU arm uses (its
    appended steps change how much each generator draws), drawn by the same
    seeded generator on the GPU when one is present (torch's Philox: the GPU
    arm's exact bits) and copied to the host; per KV head (K, V, Q, metadata)."""
    import torch
    from oracle import pages as opg
    from sparse_entmax_attention_gb300 import synth
    spec = synth.workload(WORKLOAD)
    n_append = 4 * (K + W) + 8  # the timed steps, then the eager and the captured e2e steps
    spec = synth.Spec(**{**spec.__dict__, "steps": n_append, "append_per_step": True})
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    q = synth.queries(spec, 0, 0, dev)
    g = spec.group
    heads = []
    for j in range(spec.num_kv_heads):
        hd = synth.HeadDraws(spec, 0, j, q[j * g:(j + 1) * g], 0, dev)
        Kh = hd.k.float().cpu().numpy()
        Vh = hd.v.float().cpu().numpy()
        Q = q[j * g:(j + 1) * g].double().cpu().numpy()
        del hd
        heads.append((Kh, Vh, Q, opg.bf16_metadata(opg.page_metadata(Kh, spec.page_size))))
    return spec, heads, dev


def one_thread_step_s(K, W):
    """One whole oracle step with BLAS and OpenMP held to one thread (a child
    process, since thread pools are fixed when numpy loads)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import bench, time; spec, heads, _ = bench.reference_inputs(%d, %d); t = time.perf_counter(); "
            "bench.oracle_decode_step(heads, spec.page_size); print(time.perf_counter() - t)" % (K, W))
    try:
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=900)
        return float(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError):
        return None


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is one whole float64
    Gaussian decode step of the 1M workload (all 8 KV heads and their query
    heads) on the GPU arm's stored bits, timed on the host cores."""
    if rank != 0:
        return None
    spec, heads, dev = reference_inputs(args.steps, args.warmup)
    for _ in range(args.warmup):
        oracle_decode_step(heads, spec.page_size)
    t0 = time.perf_counter()
    us = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle_decode_step(heads, spec.page_size)
        us.append((time.perf_counter() - t) * 1e6)
    wall = time.perf_counter() - t0
    v = statistics.mean(us)
    del heads
    one = one_thread_step_s(args.steps, args.warmup)
    return {"impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "us/step",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(v / 1e3, 3), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64",
            "data": f"synthetic: the GPU arm's seeded generator, drawn on {dev} and copied to the host",
            "config": {"workload": WORKLOAD, "policy": "gaussian", "margin": MARGIN, "alpha": ALPHA},
            "cpu_baseline": {"value": round(v, 1), "unit": "us/step", "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"{args.steps} whole decode steps ({spec.num_kv_heads} KV heads x "
                                       f"{spec.group} query heads, 1M tokens each), BLAS default threads",
                             "one_thread_us_per_step": None if one is None else round(one * 1e6, 1)},
            "e2e": {"value": round(v, 1), "unit": "us/step", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s_timed_loop": round(wall, 3)}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        res = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            torch.distributed.init_process_group("nccl")
        res = run_ours(args, rank, world)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if res is not None and rank == 0:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
