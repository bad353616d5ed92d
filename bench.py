#!/usr/bin/env python
"""Benchmark of one step of the path on the 4M-token workload (default).

A step is one pass of the whole hot path over one chunk with every input
resident in HBM: page representatives of all pages -> Top-K selection ->
sparse attention forward -> sparse attention backward with in-place paged
dK/dV.  The metric is the method's: sparse-attention fwd+bwd TFLOP/s, counting
14 * D * Hq flops per unmasked (query, key) pair, with tokens/s per chunk and
the fraction of the bf16 tensor peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...    # the CPU float64 oracle, bounded sample

For N > 1 (torchrun), every rank runs an independent replica on its own GPU
(the path has no exchange step); value = all ranks' work / the slowest rank.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from paged_sparse_attention_oomb_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "sparse attn fwd+bwd TFLOP/s and tokens/s per chunk at 256K–4M ctx; % of bf16 peak"
DEFAULT_WORKLOAD = "qwen7b_ctx4m_k128"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def pairs_per_head(wl, rows=None):
    """Unmasked (query, key) pairs of one query head for the chunk (or its
    first `rows` rows): every selected key, plus the causal own keys."""
    c = wl.chunk_len if rows is None else rows
    return wl.n_sel * wl.page_size * c + c * (c + 1) // 2


def attn_flops(wl, rows=None):
    return 14.0 * wl.head_dim * wl.num_q_heads * pairs_per_head(wl, rows)


def max_over_ranks(x, world, device="cpu"):
    """The slowest rank's value (replicas: the job ends when the last one does)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_value(flops_per_replica, ms_slowest, world):
    """Whole-job throughput in TFLOP/s: every replica's work over the slowest time."""
    return world * flops_per_replica / ms_slowest / 1e9


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
REASON_COLS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        cmd = ["nvidia-smi", "-i", str(self.gpu),
               "--query-gpu=clocks.sm,clocks.max.sm,power.draw,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
               "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(REASON_COLS, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
CHUNK_PASS_WORKLOAD = "qwen7b_dense_ctx32k"


def chunk_pass_flops(wl):
    """14 * D * Hq * unmasked pairs, summed over the chunks of a whole pass:
    chunk c attends min(top_k, c * C / P) past pages plus its causal own keys."""
    c, p = wl.chunk_len, wl.page_size
    pairs = sum(min(wl.top_k, ci * c // p) * p * c + c * (c + 1) // 2
                for ci in range(wl.context // c))
    return 14.0 * wl.head_dim * wl.num_q_heads * pairs


def measure_offload(wl, x, kv, reps, dev, n_chunks=4, passes=5):
    """The last ``n_chunks`` chunks of the workload as a chunk-recurrent pass
    (forward in order, backward in reverse), with the pools resident in HBM and
    with the K, V, dK, dV pools in pinned host memory behind a device page cache
    (oomb_offload_*), the next chunk's tiles brought in on a second stream while
    the current chunk computes.  Offloaded passes start from an empty cache
    ("cold": the host gradients hold earlier sums, so gradient tiles are copied
    in) or, in addition, from zeroed host gradients declared with zero_grads()
    ("zero_grads": a new pass of training, gradient tiles zero-filled in the
    cache).  Then the same two with the host K/V pools stored as E4M3 codes (an
    fp8 KV cache, expanded to bf16 as tiles are fetched).  Every pass is timed
    alone with CUDA events after an untimed preparation (emptying the cache,
    zeroing the host gradients), the variants interleaved pass by pass with the
    resident pass; each figure is the median over ``passes`` rounds after one
    warm-up round, and each overhead is against the resident median of the same
    rounds."""
    import statistics
    from paged_sparse_attention_oomb_gb300 import oomb
    c, p, hkv = wl.chunk_len, wl.page_size, wl.num_kv_heads
    start = wl.context - n_chunks * c
    g = torch.Generator(device=dev)
    g.manual_seed(2)
    shape = (n_chunks * c, wl.num_q_heads, wl.head_dim)
    q = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
    do = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
    t_host0 = time.time()
    host = oomb.PagedKV(torch.empty(x.k_pool.shape, dtype=x.k_pool.dtype, pin_memory=True),
                        torch.empty(x.k_pool.shape, dtype=x.k_pool.dtype, pin_memory=True),
                        x.page_table.cpu(),
                        torch.empty(x.k_pool.shape, dtype=x.k_pool.dtype, pin_memory=True),
                        torch.empty(x.k_pool.shape, dtype=x.k_pool.dtype, pin_memory=True))
    host.k.copy_(x.k_pool)
    host.v.copy_(x.v_pool)
    host.dk.zero_()
    host.dv.zero_()
    setup_s = time.time() - t_host0
    slots = 2 * (wl.top_k * hkv + c // p) + 64

    def resident():
        oomb.chunk_recurrent_pass(q, do, kv, c, wl.top_k, start=start, reps=reps)

    def offloaded(cache, zero):
        def prep():
            if zero:
                host.dk.zero_()
                host.dv.zero_()
                cache.zero_grads()
            cache.flush(drop=True)
        return prep, lambda: oomb.chunk_recurrent_pass_offloaded(q, do, cache, c, wl.top_k,
                                                                 start=start, reps=reps)

    def rounds(variants):
        """variants: name -> (cache or None, prep or None, run); medians in ms
        and per-pass move counters over the timed rounds."""
        times = {k: [] for k in variants}
        moved = {k: {} for k in variants}
        for i in range(passes + 1):
            for name, (cache, prep, run) in variants.items():
                if prep is not None:
                    prep()
                torch.cuda.synchronize()
                s0 = cache.stats() if cache is not None else None
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                run()
                e1.record()
                torch.cuda.synchronize()
                if i == 0:
                    continue                     # warm-up round
                times[name].append(e0.elapsed_time(e1))
                if cache is not None:
                    s1 = cache.stats()
                    for key in ("bytes_in", "bytes_out", "tiles_zero_filled"):
                        moved[name][key] = moved[name].get(key, 0) + (s1[key] - s0[key]) / passes
        return ({k: statistics.median(v) for k, v in times.items()},
                {k: [round(t, 3) for t in v] for k, v in times.items()}, moved)

    def entry(name, med, all_ms, moved, res_key):
        m = moved[name]
        return {"ms_per_pass_offloaded": med[name], "overhead": med[name] / med[res_key] - 1.0,
                "ms_per_pass_resident": med[res_key], "passes_ms": all_ms[name],
                "bytes_in_per_pass": m["bytes_in"], "bytes_out_per_pass": m["bytes_out"],
                "tiles_zero_filled_per_pass": m["tiles_zero_filled"]}

    cache = oomb.OffloadCache(host, slots, dev)
    med, all_ms, moved = rounds({"resident": (None, None, resident),
                                 "cold": (cache,) + offloaded(cache, False),
                                 "zero_grads": (cache,) + offloaded(cache, True)})
    res = {"workload": f"{wl.name}, last {n_chunks} chunks", "chunks": n_chunks,
           "cache_slots": cache.cache_slots,
           "cache_bytes": 4 * cache.ck.numel() * cache.ck.element_size(),
           "host_pool_bytes": 4 * host.k.numel() * host.k.element_size(),
           "host_setup_s": setup_s, "timing": f"median of {passes} interleaved passes",
           "resident_passes_ms": all_ms["resident"]}
    res.update(entry("cold", med, all_ms, moved, "resident"))
    res["what"] = ("fwd in order + bwd in reverse, cold cache per pass; next chunk's tiles "
                   "fetched on a second stream")
    res["zero_grads"] = entry("zero_grads", med, all_ms, moved, "resident")
    res["zero_grads"]["what"] = ("each pass starts a new pass: host dK/dV zeroed (untimed) and "
                                 "declared with zero_grads(); gradient tiles still zero on the "
                                 "host are zero-filled in the cache")
    cache.close()
    # fp8 KV: E4M3 host K/V pools (half the bytes over the link), same gradients
    del host.k, host.v                  # the bf16 host K/V pools are not needed any more
    t_host0 = time.time()
    k8 = torch.empty(x.k_pool.shape, dtype=torch.float8_e4m3fn, pin_memory=True)
    v8 = torch.empty(x.v_pool.shape, dtype=torch.float8_e4m3fn, pin_memory=True)
    for dst, src in ((k8, x.k_pool), (v8, x.v_pool)):
        for b0 in range(0, src.shape[0], 4096):
            dst[b0:b0 + 4096].copy_(src[b0:b0 + 4096].to(torch.float8_e4m3fn))
    setup8 = time.time() - t_host0
    cache8 = oomb.OffloadCache(oomb.PagedKV(k8, v8, x.page_table.cpu(), host.dk, host.dv),
                               slots, dev)
    med, all_ms, moved = rounds({"resident": (None, None, resident),
                                 "cold": (cache8,) + offloaded(cache8, False),
                                 "zero_grads": (cache8,) + offloaded(cache8, True)})
    res["fp8_kv"] = entry("cold", med, all_ms, moved, "resident")
    res["fp8_kv"].update({"host_pool_bytes": 2 * k8.numel() + 4 * k8.numel(),
                          "host_setup_s": setup8,
                          "what": "host K/V as E4M3 codes expanded to bf16 on fetch; overhead "
                                  "against the resident bf16 pass of the same rounds"})
    res["fp8_kv"]["new_pass"] = entry("zero_grads", med, all_ms, moved, "resident")
    cache8.close()
    return res


def measure_chunk_pass(dev, peak_t, passes=3):
    """The chunk-recurrent pass over the whole 32K-token sequence (8 chunks of
    4096, every past page selected): forward over the chunks in order, with the
    representatives of each chunk's pages computed after its forward, then the
    backward in reverse order accumulating dK/dV in place -- one call of
    ``oomb.chunk_recurrent_pass``, timed with CUDA events."""
    from paged_sparse_attention_oomb_gb300 import oomb
    wl = WORKLOADS[CHUNK_PASS_WORKLOAD]
    x = make_inputs(wl, seed=0, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    shape = (wl.context, wl.num_q_heads, wl.head_dim)
    q_full = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
    do_full = torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
    kv = oomb.PagedKV(x.k_pool, x.v_pool, x.page_table, torch.zeros_like(x.k_pool),
                      torch.zeros_like(x.v_pool))
    oomb.chunk_recurrent_pass(q_full, do_full, kv, wl.chunk_len, wl.top_k)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(passes):
        oomb.chunk_recurrent_pass(q_full, do_full, kv, wl.chunk_len, wl.top_k)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / passes
    flops = chunk_pass_flops(wl)
    return {"workload": wl.name, "context": wl.context, "chunks": wl.context // wl.chunk_len,
            "chunk_len": wl.chunk_len, "passes": passes, "ms_per_pass": ms,
            "TFLOP/s": flops / ms / 1e9, "frac_bf16": flops / ms / 1e9 / peak_t,
            "what": "reps + selection + fwd per chunk in order, bwd in reverse; dK/dV in place"}


# DRAM bytes (read + write) of one backward call -- bwd_prep_kernel +
# sparse_attn_bwd_kernel + dq_convert_kernel -- from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by workload, with the
# SHA-256 of the backward's source files at the time of the capture: when the
# sources differ the figure describes another kernel and the bench reports
# the traffic as null.
BWD_TRAFFIC = {
    "qwen7b_ctx4m_k128": {
        "bytes": 2205717504, "sha": "bae900ecdadd924e",
        "how": "ncu dram__bytes_read.sum + dram__bytes_write.sum of bwd_prep_kernel (253.5 MB), "
               "sparse_attn_bwd_kernel (1811.3 MB) and dq_convert_kernel (141.0 MB), first "
               "backward call, captured on the same backward launches over a 512K-token cache "
               "(bench.py --context 524288: same chunk, Top-K, page size and heads, so the same "
               "selected and own pages per launch)"},
}
BWD_SOURCES = ["k_attn_bwd_bf16.cu", "sm100.cuh", "tmap.h"]


def bwd_source_sha():
    import hashlib
    h = hashlib.sha256()
    for f in BWD_SOURCES:
        with open(os.path.join(ROOT, "paged_sparse_attention_oomb_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


class PathStep:
    """Buffers and workspaces of one step of the path on one workload: page
    representatives of all pages -> Top-K selection -> forward -> backward
    (dK/dV in place), the four C ABI calls, on the current stream."""
    NAMES = ["page_reps", "select_topk", "attn_fwd", "attn_bwd"]
    LAUNCHES = 1 + 1 + 1 + 3          # kernels per step: reps; selection; fwd; prep/bwd/convert

    def __init__(self, wl, dev):
        from paged_sparse_attention_oomb_gb300 import oomb
        self.oomb, self.wl = oomb, wl
        self.x = x = make_inputs(wl, seed=0, device=dev)
        self.kv = kv = oomb.PagedKV(x.k_pool, x.v_pool, x.page_table, torch.zeros_like(x.k_pool),
                                    torch.zeros_like(x.v_pool))
        hkv, d, c, hq = wl.num_kv_heads, wl.head_dim, wl.chunk_len, wl.num_q_heads
        self.reps = torch.empty((wl.num_pages, hkv, d), dtype=torch.float32, device=dev)
        self.sel = torch.empty((hkv, max(wl.n_sel, 1)), dtype=torch.int32, device=dev)
        self.o = torch.empty_like(x.q)
        self.o_lo = oomb.o_residual_like(self.o)
        self.lse = torch.empty((hq, c), dtype=torch.float32, device=dev)
        self.dq = torch.empty_like(x.q)
        self.ws = [oomb.workspace(oomb.OOMB_OP_PAGE_REPS, kv),
                   oomb.workspace(oomb.OOMB_OP_SELECT_TOPK, kv, hq, c, wl.top_k),
                   oomb.workspace(oomb.OOMB_OP_ATTN_FWD, kv, hq, c),
                   oomb.workspace(oomb.OOMB_OP_ATTN_BWD, kv, hq, c)]
        self.stream = torch.cuda.current_stream()

    def __call__(self, ev=None):
        oomb, wl, kv, st = self.oomb, self.wl, self.kv, self.stream
        q, dout = self.x.q, self.x.do
        ws_r, ws_s, ws_f, ws_b = self.ws
        if ev is not None:
            ev[0].record(st)
        oomb.oomb_page_reps(kv, 0, wl.num_pages, self.reps, ws_r, st)
        if ev is not None:
            ev[1].record(st)
        oomb.oomb_select_topk(q, wl.start, self.reps, kv, wl.top_k, self.sel, ws_s, stream=st)
        if ev is not None:
            ev[2].record(st)
        oomb.oomb_sparse_attn_fwd(q, kv, self.sel, wl.n_sel, wl.start, self.o, self.lse, ws_f,
                                  stream=st, o_lo=self.o_lo)
        if ev is not None:
            ev[3].record(st)
        oomb.oomb_sparse_attn_bwd(q, self.o, dout, self.lse, kv, self.sel, wl.n_sel, wl.start,
                                  self.dq, ws_b, stream=st, o_lo=self.o_lo)
        if ev is not None:
            ev[4].record(st)

    def check_status(self):
        for w in self.ws:
            code, where, blk = self.oomb.oomb_device_status(w)
            if code != 0:
                raise RuntimeError(f"device status {self.oomb.oomb_status_string(code)} "
                                   f"at {where}/{blk}")

    def time(self, steps):
        """Per-call CUDA events over `steps` steps on the launching stream;
        returns (total ms, {call: [ms per step]})."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(self.stream)
        for i in range(steps):
            self(evs[i])
        t1.record(self.stream)
        torch.cuda.synchronize()
        per = {n: [evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(steps)]
               for k, n in enumerate(self.NAMES)}
        return t0.elapsed_time(t1), per


def kernel_figures(wl, per, pk, peak_key):
    """Per-call rooflines: bytes (HBM-bound calls) or flops (attention) per call
    over the mean CUDA-event time, against the measured peaks."""
    hkv, d, c, hq = wl.num_kv_heads, wl.head_dim, wl.chunk_len, wl.num_q_heads
    pairs_total = pairs_per_head(wl) * hq
    bytes_reps = wl.num_pages * hkv * wl.page_size * d * 2 + wl.num_pages * hkv * d * 4
    bytes_sel = c * hq * d * 2 + wl.num_candidates * hkv * d * 4 + hkv * wl.n_sel * 4
    work = {"page_reps": ("GB/s", bytes_reps / 1e6, pk["hbm_gbs"], "frac_hbm"),
            "select_topk": ("GB/s", bytes_sel / 1e6, pk["hbm_gbs"], "frac_hbm"),
            "attn_fwd": ("TFLOP/s", 4.0 * d * pairs_total / 1e9, pk[peak_key], "frac_bf16"),
            "attn_bwd": ("TFLOP/s", 10.0 * d * pairs_total / 1e9, pk[peak_key], "frac_bf16")}
    out = {}
    for n, v in per.items():
        ms = statistics.mean(v)
        unit, amount, peak, fkey = work[n]
        out[n] = {"ms": ms, unit: amount / ms, fkey: amount / ms / peak,
                  "ms_median": statistics.median(v), "ms_min": min(v)}
    return out


def replica_timing(run, world, sync, barrier):
    """The timed region of one replica: barrier and device sync on both sides
    of ``run()`` (which returns its own elapsed ms), then the slowest rank's
    time (replicas: the job ends when the last one does)."""
    if world > 1:
        barrier()
    sync()
    ms = run()
    sync()
    if world > 1:
        barrier()
    return ms, max_over_ranks(ms, world)


def measure_configs(names, dev, steps, warmup, pk, peak_key):
    """The other workloads of the evaluation ladder, one after another: a few
    warm-up steps, then `steps` timed steps each (per-call CUDA events)."""
    out = {}
    for name in names:
        wl = WORKLOADS[name]
        step = PathStep(wl, dev)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        step.check_status()
        total, per = step.time(steps)
        step.check_status()
        ms = total / steps
        fwd_bwd_ms = statistics.mean(per["attn_fwd"]) + statistics.mean(per["attn_bwd"])
        flops = attn_flops(wl)
        out[name] = {"context": wl.context, "page_size": wl.page_size, "chunk_len": wl.chunk_len,
                     "top_k": wl.top_k, "steps": steps, "ms_per_step": ms,
                     "TFLOP/s": flops / ms / 1e9, "frac_of_bf16_peak": flops / ms / 1e9 / pk[peak_key],
                     "fwd_bwd_ms": fwd_bwd_ms, "fwd_bwd_TFLOP/s": flops / fwd_bwd_ms / 1e9,
                     "fwd_bwd_frac": flops / fwd_bwd_ms / 1e9 / pk[peak_key],
                     "tokens_per_s_per_chunk": wl.chunk_len / (ms / 1e3),
                     "kernels": kernel_figures(wl, per, pk, peak_key)}
        del step
        torch.cuda.empty_cache()
    return out


OTHER_CONFIGS = ["qwen7b_ctx256k_k64", "qwen7b_ctx1m_k128", "qwen7b_dense_ctx32k"]


def workload_of(args):
    """The named workload, or with ``--context`` the same chunk, heads, page
    size and Top-K over a shorter cache: the attention kernels then do the same
    work per launch (the same number of selected and own pages) on a pool that
    fits a profiler's capture."""
    wl = WORKLOADS[args.workload]
    ctx = args.context
    if not ctx or ctx == wl.context:
        return wl
    if ctx % wl.page_size or (ctx - wl.chunk_len) // wl.page_size < min(wl.top_k, 1 << 20):
        raise SystemExit(f"--context {ctx}: needs whole pages of {wl.page_size} and at least "
                         f"top_k={wl.top_k} candidate pages before the last chunk")
    return wl.with_(name=f"{wl.name}@ctx{ctx}", context=ctx)


def run_ours(args, rank, world, dev):
    from paged_sparse_attention_oomb_gb300 import oomb

    wl = workload_of(args)
    torch.cuda.set_device(dev)
    step = PathStep(wl, dev)
    x, kv, stream = step.x, step.kv, step.stream
    hkv, d, c, hq = wl.num_kv_heads, wl.head_dim, wl.chunk_len, wl.num_q_heads
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    step.check_status()

    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    phys = vis.split(",")[dev.index] if vis and vis.split(",")[0].isdigit() else dev.index
    box = {}

    def run():
        box["total"], box["per"] = step.time(args.steps)
        return box["total"]

    with ClockSampler(phys) as clk:
        total_ms, slowest_ms = replica_timing(run, world, torch.cuda.synchronize,
                                              torch.distributed.barrier if world > 1 else None)
    per = box["per"]
    ms = slowest_ms / args.steps
    timed_s = total_ms / 1e3
    step.check_status()
    sel_gpu = step.sel[:, :wl.n_sel].cpu().numpy()

    # end to end through the public API with host buffers: per step the chunk's
    # queries and output grads come from pinned host memory and the outputs (O,
    # LSE, dQ) go back to pinned host memory, inside the timed region.
    # oomb.StepPipeline overlaps those copies (copy engines) with the compute of
    # the neighbouring steps, as a user streaming chunks would.
    q_h = x.q.cpu().pin_memory()
    do_h = x.do.cpu().pin_memory()
    o_h = torch.empty_like(q_h).pin_memory()
    dq_h = torch.empty_like(q_h).pin_memory()
    lse_h = torch.empty(step.lse.shape, dtype=step.lse.dtype).pin_memory()
    pipe = oomb.StepPipeline(kv, wl.start, c, hq, wl.top_k)
    for _ in range(2):
        pipe.step(q_h, do_h, o_h, lse_h, dq_h)
    pipe.finish()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipe.begin()
    for _ in range(args.steps):
        pipe.step(q_h, do_h, o_h, lse_h, dq_h)
    stream.wait_stream(pipe.d2h)
    e1.record(stream)
    torch.cuda.synchronize()
    pipe.finish()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    h2d = q_h.numel() * q_h.element_size() + do_h.numel() * do_h.element_size()
    d2h = (o_h.numel() * o_h.element_size() + dq_h.numel() * dq_h.element_size()
           + lse_h.numel() * lse_h.element_size())
    del pipe
    step.check_status()

    flops = attn_flops(wl)
    pk, pk_src = peaks()
    # the timed region lasts well under a second at the maximum clock: the
    # burst peak is the one that applies; a region of seconds would hold the
    # sustained one (the peak measured under the power cap)
    peak_key = "bf16_tflops" if timed_s < 1.0 else "bf16_tflops_sustained"

    def optional(fn):
        # the side measurements must not cost the step's line: a failure (for
        # example pinned host memory refused) is reported in place of the figures
        try:
            return fn()
        except Exception as e:  # noqa: BLE001
            torch.cuda.synchronize()
            return {"error": f"{type(e).__name__}: {e}"[:300]}

    chunk_pass = (optional(lambda: measure_chunk_pass(dev, pk[peak_key]))
                  if args.chunk_pass and wl.dtype == "bf16" else None)
    offload = (optional(lambda: measure_offload(wl, x, kv, step.reps, dev))
               if args.offload and wl.dtype == "bf16" and wl.n_sel > 0 else None)
    kern = kernel_figures(wl, per, pk, peak_key)
    for n in ("attn_fwd", "attn_bwd"):
        kern[n]["frac_bf16_sustained"] = kern[n]["TFLOP/s"] / pk["bf16_tflops_sustained"]
    achieved = kern["attn_bwd"]["TFLOP/s"]
    sha = bwd_source_sha()
    rec = BWD_TRAFFIC.get(wl.name)
    fresh = rec is not None and rec["sha"] == sha
    clocks = clk.summary()
    res = {
        "metric": METRIC,
        "value": job_value(flops, ms, world),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; clustered page keys, N(0,1) values/queries/grads)",
        "config": {"workload": wl.name, "context": wl.context, "page_size": wl.page_size,
                   "chunk_len": c, "chunk_start": wl.start, "top_k": wl.top_k,
                   "num_q_heads": hq, "num_kv_heads": hkv, "head_dim": d,
                   "page_table": "shuffled" if wl.shuffled else "identity",
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: each step streams the whole K pool"},
        "tokens_per_s_per_chunk": world * c / (ms / 1e3),
        "frac_of_bf16_peak": flops / ms / 1e9 / pk[peak_key],
        "kernels": kern,
        "chunk_pass": chunk_pass,
        "offload": offload,
        "roofline": {"kernel": "oomb_sparse_attn_bwd (delta prep + sparse_attn_bwd_kernel + dq convert)",
                     "bound": "tensor", "achieved": achieved, "peak": pk[peak_key],
                     "peak_source": f"{pk_src} {peak_key}: timed region {timed_s:.2f} s at a "
                                    f"median {clocks.get('sm_mhz')} MHz",
                     "unit": "TFLOP/s", "frac": achieved / pk[peak_key],
                     "frac_sustained": achieved / pk["bf16_tflops_sustained"],
                     "traffic": rec["bytes"] if fresh else None,
                     "traffic_source": (rec["how"] if fresh else
                                        "no capture of the current backward sources "
                                        f"(sha {sha})")},
        "e2e": {"value": world * flops / e2e_ms / 1e9, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "steps": args.steps},
        "gpu_launches": args.steps * PathStep.LAUNCHES,
        "clocks": clocks,
    }
    return res, step, sel_gpu, peak_key


def selection_vs_oracle(sel_gpu, sel_o, scores_o, gap=1e-4):
    """The GPU selection against the oracle's: per KV head, the pages only one
    side picked must pair up with oracle fp32 scores closer than ``gap``
    (near-ties, counted); anything else is a mismatch."""
    swaps, worst, mismatch = 0, 0.0, 0
    for g in range(sel_o.shape[0]):
        a = sorted(set(sel_gpu[g].tolist()) - set(sel_o[g].tolist()))
        b = sorted(set(sel_o[g].tolist()) - set(sel_gpu[g].tolist()))
        if len(a) != len(b):
            mismatch += 1
            continue
        sa = sorted(float(scores_o[g][i]) for i in a)
        sb = sorted(float(scores_o[g][i]) for i in b)
        for u, v in zip(sa, sb):
            if abs(u - v) >= gap:
                mismatch += 1
            worst = max(worst, abs(u - v))
        swaps += len(a)
    return {"heads": int(sel_o.shape[0]), "k": int(sel_o.shape[1]), "near_tie_swaps": swaps,
            "largest_swap_gap": worst, "mismatches": mismatch, "gap_exempt": gap}


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample of the same workload
# ---------------------------------------------------------------------------
def oracle_setup(wl, x=None):
    """Host copies of what the oracle needs and the oracle's own selection."""
    import oracle
    from paged_sparse_attention_oomb_gb300.workloads import to_numpy64
    if x is None:
        dev = "cuda:0" if torch.cuda.is_available() else "cpu"
        x = make_inputs(wl, seed=0, device=dev)
    pt = x.page_table.cpu().long()
    k_host = x.k_pool.cpu()
    reps = np.concatenate([oracle.page_reps(k_host[pt[b:b + 512]].float().numpy(),
                                            np.arange(min(512, wl.num_pages - b)))
                           for b in range(0, wl.num_pages, 512)])
    q = to_numpy64(x.q)
    do = to_numpy64(x.do)
    scores = oracle.page_scores(oracle.query_summary(q, wl.num_kv_heads), reps,
                                wl.num_candidates)
    sel = oracle.select_topk(scores, wl.top_k)
    own = np.arange(wl.start // wl.page_size, (wl.start + wl.chunk_len) // wl.page_size)
    need = np.unique(np.concatenate([sel.reshape(-1), own]))
    slots = pt.numpy()[need]
    kc = k_host[torch.as_tensor(slots)].float().numpy()
    vc = x.v_pool.cpu()[torch.as_tensor(slots)].float().numpy()
    ptc = np.full(wl.num_pages, -1, np.int64)
    ptc[need] = np.arange(need.size)
    return dict(q=q, do=do, sel=sel, scores=scores, kc=kc, vc=vc, ptc=ptc)


def oracle_step(wl, st, rows):
    """fwd + bwd of the oracle for the first `rows` rows of the chunk (all heads)."""
    import oracle
    q, do = st["q"][:rows], st["do"][:rows]
    o, lse = oracle.attn_fwd(q, st["kc"], st["vc"], st["ptc"], st["sel"], wl.start, wl.page_size)
    shp = (st["kc"].shape[0],) + st["kc"].shape[1:]
    oracle.attn_bwd(q, st["kc"], st["vc"], st["ptc"], st["sel"], wl.start, wl.page_size, o, lse,
                    do, dk_acc=np.zeros(shp), dv_acc=np.zeros(shp), acc_rows=st["ptc"])


def cpu_baseline(wl, st, rows, reps=1):
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(wl, st, rows)
    dt = (time.perf_counter() - t0) / reps
    return {"value": attn_flops(wl, rows) / dt / 1e12, "unit": "TFLOP/s",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"first {rows} chunk rows, all {wl.num_q_heads} heads, fwd+bwd "
                      f"(float64 NumPy); oracle's own selection made outside the timed part",
            "seconds": dt}


def run_reference(args, rank, world):
    wl = workload_of(args)
    if rank != 0:
        return None
    st = oracle_setup(wl)
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_step(wl, st, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(wl, st, rows)
    dt = (time.perf_counter() - t0) / args.steps
    val = attn_flops(wl, rows) / dt / 1e12
    cb = {"value": val, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
          "sample": f"first {rows} chunk rows, all heads, fwd+bwd per step (float64 NumPy)"}
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": {"workload": wl.name, "rows_per_step": rows},
            "cpu_baseline": cb,
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def relaunch_as_replicas(n):
    """bench.py --gpus N started without torchrun: start it again under
    torchrun with one rank (one replica) per GPU; refuse if there are fewer."""
    have = torch.cuda.device_count() if torch.cuda.is_available() else 0
    if have < n:
        sys.stderr.write(f"bench.py: --gpus {n} asks for {n} GPUs, {have} visible\n")
        sys.exit(2)
    import socket
    with socket.socket() as s_:
        s_.bind(("127.0.0.1", 0))
        port = s_.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr=127.0.0.1", f"--master-port={port}",
           os.path.abspath(__file__)] + sys.argv[1:]
    os.execv(sys.executable, cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--context", type=int, default=0,
                    help="shorter cache for the workload (same chunk, Top-K and heads): "
                         "a small case for profiler captures")
    ap.add_argument("--cpu-rows", type=int, default=512)
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-chunk-pass", dest="chunk_pass", action="store_false",
                    help="skip the whole-sequence chunk-recurrent pass measurement")
    ap.add_argument("--no-offload", dest="offload", action="store_false",
                    help="skip the host-offload measurement")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the 256K, 1M and dense 32K workloads")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world == 1 and args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        relaunch_as_replicas(args.gpus)
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
    else:
        dev = torch.device("cuda", local)
        res, step, sel_gpu, peak_key = run_ours(args, rank, world, dev)
        wl = step.wl
        st = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            st = oracle_setup(wl, step.x)          # host copies, then the device frees them
        del step
        torch.cuda.empty_cache()
        if rank == 0 and args.configs:
            pk, _ = peaks()
            res["configs"] = measure_configs([n for n in OTHER_CONFIGS if n != wl.name], dev,
                                             min(args.steps, 20), args.warmup, pk, peak_key)
        if st is not None:
            res["selection_vs_oracle"] = selection_vs_oracle(sel_gpu, st["sel"], st["scores"])
            res["cpu_baseline"] = cpu_baseline(wl, st, args.cpu_rows)
        if rank == 0:
            print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
