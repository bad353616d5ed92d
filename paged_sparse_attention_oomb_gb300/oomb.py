"""Thin Python binding of liboomb (C ABI in include/oomb.h), same call names.

Argument marshalling only: torch tensors are passed as device pointers with
their sizes; every step of the path runs in liboomb's CUDA kernels.  The
library is loaded from this package directory and an ``OombError`` is raised
if it is missing -- there is no other implementation behind these calls.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboomb.so")

OOMB_OK, OOMB_ERR_INVALID_ARG, OOMB_ERR_UNSUPPORTED = 0, 1, 2
OOMB_ERR_CUDA, OOMB_ERR_TIMEOUT, OOMB_ERR_DEVICE_BOUNDS, OOMB_ERR_NONFINITE = 3, 4, 5, 6
OOMB_BF16, OOMB_FP32, OOMB_FP8_E4M3 = 0, 1, 2
OOMB_OP_VALIDATE, OOMB_OP_PAGE_REPS, OOMB_OP_SELECT_TOPK = 0, 1, 2
OOMB_OP_ATTN_FWD, OOMB_OP_ATTN_BWD = 3, 4

EXPORTED = [
    "oomb_workspace_bytes", "oomb_validate_page_table_host", "oomb_validate_page_table",
    "oomb_page_reps", "oomb_select_topk", "oomb_select_topk_noalloc", "oomb_sparse_attn_fwd",
    "oomb_sparse_attn_fwd_own_reps", "oomb_sparse_attn_bwd",
    "oomb_offload_create", "oomb_offload_acquire", "oomb_offload_flush", "oomb_offload_writeback",
    "oomb_offload_writeback_pages",
    "oomb_offload_stats", "oomb_offload_destroy", "oomb_offload_zero_grads",
    "oomb_device_status", "oomb_set_wait_limit_ns", "oomb_debug_wait_unset_flag",
    "oomb_status_string", "oomb_last_error",
]


class OombError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{_STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


_STATUS_NAMES = {0: "OOMB_OK", 1: "OOMB_ERR_INVALID_ARG", 2: "OOMB_ERR_UNSUPPORTED",
                 3: "OOMB_ERR_CUDA", 4: "OOMB_ERR_TIMEOUT", 5: "OOMB_ERR_DEVICE_BOUNDS",
                 6: "OOMB_ERR_NONFINITE"}


class OombOffloadDesc(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dk", ctypes.c_void_p),
                ("dv", ctypes.c_void_p), ("host_page_table", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("num_host_slots", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("cache_k", ctypes.c_void_p), ("cache_v", ctypes.c_void_p),
                ("cache_dk", ctypes.c_void_p), ("cache_dv", ctypes.c_void_p),
                ("cache_slots", ctypes.c_int32), ("dev_staging", ctypes.c_void_p),
                ("dev_staging_bytes", ctypes.c_int64), ("backing_kv_dtype", ctypes.c_int32)]


class OombPagedKV(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("dk", ctypes.c_void_p),
                ("dv", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("num_pages", ctypes.c_int32), ("num_slots", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


_lib = None


def load():
    """Load liboomb.so (built in-tree by ``build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise OombError(-1, f"{LIB_PATH} is missing: run __graft_entry__.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    kvp = ctypes.POINTER(OombPagedKV)
    sig = {
        "oomb_workspace_bytes": (sz, [ctypes.c_int, kvp, i32, i32, i32]),
        "oomb_validate_page_table_host": (ctypes.c_int, [vp, i32, i32]),
        "oomb_validate_page_table": (ctypes.c_int, [kvp, vp, sz, vp]),
        "oomb_page_reps": (ctypes.c_int, [kvp, i32, i32, vp, vp, sz, vp]),
        "oomb_select_topk": (ctypes.c_int, [vp, i32, i32, i32, vp, kvp, i32, vp, vp, vp, sz, vp]),
        "oomb_select_topk_noalloc": (ctypes.c_int, [vp, i32, i32, i32, vp, kvp, i32, vp, vp, vp]),
        "oomb_sparse_attn_fwd": (ctypes.c_int, [vp, kvp, vp, i32, i32, i32, i32, ctypes.c_float,
                                                vp, vp, vp, vp, sz, vp]),
        "oomb_sparse_attn_fwd_own_reps": (ctypes.c_int, [vp, kvp, vp, i32, i32, i32, i32,
                                                         ctypes.c_float, vp, vp, vp, vp, vp, sz,
                                                         vp]),
        "oomb_sparse_attn_bwd": (ctypes.c_int, [vp, vp, vp, vp, vp, kvp, vp, i32, i32, i32, i32,
                                                ctypes.c_float, vp, vp, sz, vp]),
        "oomb_offload_create": (ctypes.c_int, [ctypes.POINTER(OombOffloadDesc),
                                                ctypes.POINTER(ctypes.c_void_p)]),
        "oomb_offload_acquire": (ctypes.c_int, [vp, vp, i32, i32, i32, i32, vp, vp]),
        "oomb_offload_flush": (ctypes.c_int, [vp, i32, vp]),
        "oomb_offload_writeback": (ctypes.c_int, [vp, i32, i32, vp]),
        "oomb_offload_writeback_pages": (ctypes.c_int, [vp, vp, i32, vp]),
        "oomb_offload_stats": (ctypes.c_int, [vp, vp]),
        "oomb_offload_zero_grads": (ctypes.c_int, [vp]),
        "oomb_offload_destroy": (None, [vp]),
        "oomb_device_status": (ctypes.c_int, [vp, vp, vp]),
        "oomb_set_wait_limit_ns": (None, [ctypes.c_uint64]),
        "oomb_debug_wait_unset_flag": (ctypes.c_int, [vp, sz, vp]),
        "oomb_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "oomb_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(code):
    if code != OOMB_OK:
        raise OombError(code, load().oomb_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)


@dataclass
class PagedKV:
    """The paged KV cache (and its paged gradient buffers) as torch tensors.

    k, v, dk, dv: ``[num_slots, Hkv, P, D]``; page_table: int32 ``[num_pages]``
    on the device (logical page -> slot).
    """
    k: torch.Tensor
    v: torch.Tensor
    page_table: torch.Tensor
    dk: Optional[torch.Tensor] = None
    dv: Optional[torch.Tensor] = None

    def struct(self) -> OombPagedKV:
        ns, hkv, p, d = self.k.shape
        dt = {torch.bfloat16: OOMB_BF16, torch.float32: OOMB_FP32}.get(self.k.dtype)
        if dt is None:
            raise OombError(OOMB_ERR_UNSUPPORTED, f"pools of {self.k.dtype}: the kernels read bf16 "
                            "or fp32 (fp8 K/V go behind an OffloadCache)")
        return OombPagedKV(self.k.data_ptr(), self.v.data_ptr(),
                           self.dk.data_ptr() if self.dk is not None else None,
                           self.dv.data_ptr() if self.dv is not None else None,
                           self.page_table.data_ptr(), self.page_table.numel(), ns, p, hkv, d, dt)


def oomb_workspace_bytes(op, kv: PagedKV, num_q_heads=0, chunk_len=0, top_k=0) -> int:
    s = kv.struct()
    return load().oomb_workspace_bytes(op, ctypes.byref(s), num_q_heads, chunk_len, top_k)


def workspace(op, kv: PagedKV, num_q_heads=0, chunk_len=0, top_k=0) -> torch.Tensor:
    """A zero-filled device workspace of the size ``op`` needs (caller-owned)."""
    n = oomb_workspace_bytes(op, kv, num_q_heads, chunk_len, top_k)
    return torch.zeros(n, dtype=torch.uint8, device=kv.k.device)


def oomb_validate_page_table_host(page_table, num_slots):
    pt = torch.as_tensor(page_table, dtype=torch.int32).contiguous().cpu()
    _check(load().oomb_validate_page_table_host(ctypes.c_void_p(pt.data_ptr()), pt.numel(),
                                                num_slots))


def oomb_validate_page_table(kv: PagedKV, ws: torch.Tensor, stream=None):
    s = kv.struct()
    _check(load().oomb_validate_page_table(ctypes.byref(s), _ptr(ws), ws.numel(), _stream(stream)))


def oomb_page_reps(kv: PagedKV, first_page, n_pages, reps: torch.Tensor, ws: torch.Tensor,
                   stream=None):
    s = kv.struct()
    _check(load().oomb_page_reps(ctypes.byref(s), first_page, n_pages, _ptr(reps), _ptr(ws),
                                 ws.numel(), _stream(stream)))


def oomb_select_topk(q, chunk_start, reps, kv: PagedKV, top_k, sel, ws, scores=None,
                     stream=None):
    s = kv.struct()
    c, hq, _ = q.shape
    _check(load().oomb_select_topk(_ptr(q), hq, c, chunk_start, _ptr(reps), ctypes.byref(s), top_k,
                                   _ptr(sel), _ptr(scores), _ptr(ws), ws.numel(),
                                   _stream(stream)))


def oomb_select_topk_noalloc(q, chunk_start, reps, kv: PagedKV, top_k, sel, scores=None,
                             stream=None):
    """oomb_select_topk without a workspace (scratch inside the library; see oomb.h)."""
    s = kv.struct()
    c, hq, _ = q.shape
    _check(load().oomb_select_topk_noalloc(_ptr(q), hq, c, chunk_start, _ptr(reps),
                                           ctypes.byref(s), top_k, _ptr(sel), _ptr(scores),
                                           _stream(stream)))


def oomb_sparse_attn_fwd(q, kv: PagedKV, sel, n_sel, chunk_start, o, lse, ws, scale=0.0,
                         stream=None, o_lo=None):
    """o_lo (bf16 pools, optional): receives the rounding residual of o, for
    the backward's Delta (see oomb.h)."""
    s = kv.struct()
    c, hq, _ = q.shape
    _check(load().oomb_sparse_attn_fwd(_ptr(q), ctypes.byref(s), _ptr(sel), n_sel, hq, c,
                                       chunk_start, float(scale), _ptr(o), _ptr(o_lo), _ptr(lse),
                                       _ptr(ws), ws.numel(), _stream(stream)))


def oomb_sparse_attn_fwd_own_reps(q, kv: PagedKV, sel, n_sel, chunk_start, o, lse, reps, ws,
                                  scale=0.0, stream=None, o_lo=None):
    """The forward plus the representatives of the chunk's own pages into ``reps``."""
    s = kv.struct()
    c, hq, _ = q.shape
    _check(load().oomb_sparse_attn_fwd_own_reps(_ptr(q), ctypes.byref(s), _ptr(sel), n_sel, hq,
                                                c, chunk_start, float(scale), _ptr(o),
                                                _ptr(o_lo), _ptr(lse), _ptr(reps), _ptr(ws),
                                                ws.numel(), _stream(stream)))


def oomb_sparse_attn_bwd(q, o, dout, lse, kv: PagedKV, sel, n_sel, chunk_start, dq, ws,
                         scale=0.0, stream=None, o_lo=None):
    """o_lo: the forward's residual of o (or None: Delta from o alone)."""
    s = kv.struct()
    c, hq, _ = q.shape
    _check(load().oomb_sparse_attn_bwd(_ptr(q), _ptr(o), _ptr(o_lo), _ptr(dout), _ptr(lse),
                                       ctypes.byref(s), _ptr(sel), n_sel, hq, c, chunk_start,
                                       float(scale), _ptr(dq), _ptr(ws), ws.numel(),
                                       _stream(stream)))


def o_residual_like(o: torch.Tensor) -> Optional[torch.Tensor]:
    """A buffer for the forward's rounding residual of ``o`` (bf16 only; None
    for fp32, whose o is not rounded)."""
    return torch.empty_like(o) if o.dtype == torch.bfloat16 else None


def oomb_device_status(ws: torch.Tensor, stream=None):
    """Read and clear the device status word; returns (code, where, block)."""
    info = (ctypes.c_int32 * 2)()
    code = load().oomb_device_status(_ptr(ws), _stream(stream), info)
    return code, info[0], info[1]


def oomb_set_wait_limit_ns(ns: int):
    load().oomb_set_wait_limit_ns(ctypes.c_uint64(int(ns)))


def oomb_debug_wait_unset_flag(ws: torch.Tensor, stream=None):
    _check(load().oomb_debug_wait_unset_flag(_ptr(ws), ws.numel(), _stream(stream)))


def oomb_status_string(code: int) -> str:
    return load().oomb_status_string(code).decode()


def oomb_last_error() -> str:
    return load().oomb_last_error().decode()


# ---------------------------------------------------------------------------
# Convenience: one full pass of the path on one chunk (allocations by torch).
# ---------------------------------------------------------------------------
def sparse_attention_step(q, dout, kv: PagedKV, chunk_start, top_k, reps=None, stream=None):
    """reps (all pages) -> Top-K selection -> forward -> backward (dK/dV in place).

    Returns dict(reps, sel, o, lse, dq).  Every call here is one of the C ABI
    entry points above; outputs and workspaces are caller (torch) allocations.
    """
    ns, hkv, p, d = kv.k.shape
    c, hq, _ = q.shape
    n_pages = kv.page_table.numel()
    dev = q.device
    ws_r = workspace(OOMB_OP_PAGE_REPS, kv)
    if reps is None:
        reps = torch.empty((n_pages, hkv, d), dtype=torch.float32, device=dev)
        oomb_page_reps(kv, 0, n_pages, reps, ws_r, stream)
    n_sel = min(top_k, chunk_start // p)
    sel = torch.empty((hkv, max(n_sel, 1)), dtype=torch.int32, device=dev)
    ws_s = workspace(OOMB_OP_SELECT_TOPK, kv, hq, c, top_k)
    oomb_select_topk(q, chunk_start, reps, kv, n_sel, sel, ws_s, stream=stream)
    o = torch.empty_like(q)
    o_lo = o_residual_like(o)
    lse = torch.empty((hq, c), dtype=torch.float32, device=dev)
    ws_f = workspace(OOMB_OP_ATTN_FWD, kv, hq, c)
    oomb_sparse_attn_fwd(q, kv, sel, n_sel, chunk_start, o, lse, ws_f, stream=stream, o_lo=o_lo)
    dq = torch.empty_like(q)
    ws_b = workspace(OOMB_OP_ATTN_BWD, kv, hq, c)
    oomb_sparse_attn_bwd(q, o, dout, lse, kv, sel, n_sel, chunk_start, dq, ws_b, stream=stream,
                         o_lo=o_lo)
    for w in (ws_r, ws_s, ws_f, ws_b):
        code, where, blk = oomb_device_status(w, stream)
        if code != OOMB_OK:
            raise OombError(code, f"device status (where {where}, block {blk})")
    return dict(reps=reps, sel=sel[:, :n_sel], o=o, lse=lse, dq=dq)


class StepPipeline:
    """Steps of the path on chunks whose inputs and outputs live in pinned host
    memory, with the copies overlapped: step i+1's Q and dO go host -> device on
    one copy stream while step i computes, and step i's O, LSE and dQ go device ->
    host on another while step i+1 computes (the copy engines, not the SMs).
    Device buffers are double-buffered.  Every step is representatives of all
    pages -> Top-K selection -> forward -> backward (dK/dV in place), the same
    four C ABI calls as sparse_attention_step; results are identical to running
    the steps one after another (dQ up to the order of its fp32 atomic sums).

    step(q_h, do_h, o_h, lse_h, dq_h) enqueues one step and returns at once; the
    host buffers must stay untouched until finish() (or two steps later).
    """

    def __init__(self, kv: PagedKV, chunk_start, chunk_len, num_q_heads, top_k, scale=0.0):
        ns, hkv, p, d = kv.k.shape
        dev = kv.k.device
        self.kv, self.chunk_start, self.top_k, self.scale = kv, chunk_start, top_k, scale
        self.n_pages = kv.page_table.numel()
        self.n_sel = min(top_k, chunk_start // p)
        shape = (chunk_len, num_q_heads, d)
        dt = kv.k.dtype
        self.q = [torch.empty(shape, dtype=dt, device=dev) for _ in range(2)]
        self.do = [torch.empty(shape, dtype=dt, device=dev) for _ in range(2)]
        self.o = [torch.empty(shape, dtype=dt, device=dev) for _ in range(2)]
        self.o_lo = [o_residual_like(o) for o in self.o]     # stays on the device
        self.dq = [torch.empty(shape, dtype=dt, device=dev) for _ in range(2)]
        self.lse = [torch.empty((num_q_heads, chunk_len), dtype=torch.float32, device=dev)
                    for _ in range(2)]
        self.reps = torch.empty((self.n_pages, hkv, d), dtype=torch.float32, device=dev)
        self.sel = torch.empty((hkv, max(self.n_sel, 1)), dtype=torch.int32, device=dev)
        self.ws_r = workspace(OOMB_OP_PAGE_REPS, kv)
        self.ws_s = workspace(OOMB_OP_SELECT_TOPK, kv, num_q_heads, chunk_len, top_k)
        self.ws_f = workspace(OOMB_OP_ATTN_FWD, kv, num_q_heads, chunk_len)
        self.ws_b = workspace(OOMB_OP_ATTN_BWD, kv, num_q_heads, chunk_len)
        self.comp = torch.cuda.current_stream(dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.comp_done = [None, None]     # compute of the step that last used buffer b
        self.out_done = [None, None]      # copy-out of the step that last used buffer b
        self.i = 0

    def step(self, q_h, do_h, o_h, lse_h, dq_h):
        b = self.i & 1
        with torch.cuda.stream(self.h2d):
            if self.comp_done[b] is not None:
                self.h2d.wait_event(self.comp_done[b])   # step i-2 has read buffer b
            self.q[b].copy_(q_h, non_blocking=True)
            self.do[b].copy_(do_h, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(self.h2d)
        self.comp.wait_event(ready)
        if self.out_done[b] is not None:
            self.comp.wait_event(self.out_done[b])       # step i-2's outputs are home
        kv, st = self.kv, self.comp
        oomb_page_reps(kv, 0, self.n_pages, self.reps, self.ws_r, st)
        oomb_select_topk(self.q[b], self.chunk_start, self.reps, kv, self.top_k, self.sel,
                         self.ws_s, stream=st)
        oomb_sparse_attn_fwd(self.q[b], kv, self.sel, self.n_sel, self.chunk_start, self.o[b],
                             self.lse[b], self.ws_f, self.scale, st, o_lo=self.o_lo[b])
        oomb_sparse_attn_bwd(self.q[b], self.o[b], self.do[b], self.lse[b], kv, self.sel,
                             self.n_sel, self.chunk_start, self.dq[b], self.ws_b, self.scale, st,
                             o_lo=self.o_lo[b])
        done = torch.cuda.Event()
        done.record(self.comp)
        self.comp_done[b] = done
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(done)
            o_h.copy_(self.o[b], non_blocking=True)
            lse_h.copy_(self.lse[b], non_blocking=True)
            dq_h.copy_(self.dq[b], non_blocking=True)
            out = torch.cuda.Event()
            out.record(self.d2h)
        self.out_done[b] = out
        self.i += 1

    def begin(self):
        """Order the next copies after everything already on the compute stream."""
        self.h2d.wait_stream(self.comp)
        self.d2h.wait_stream(self.comp)

    def finish(self):
        """Make the compute stream wait for every copy; then check the status words."""
        self.comp.wait_stream(self.d2h)
        self.comp.wait_stream(self.h2d)
        for w in (self.ws_r, self.ws_s, self.ws_f, self.ws_b):
            code, where, blk = oomb_device_status(w, self.comp)
            if code != OOMB_OK:
                raise OombError(code, f"device status (where {where}, block {blk})")


def _rows(t: Optional[torch.Tensor], r0, n):
    return None if t is None else t[r0:r0 + n]


def chunk_recurrent_pass(q_full, dout_full, kv: PagedKV, chunk_len, top_k, scale=0.0,
                         stream=None, start=0, reps=None):
    """One chunk-recurrent pass over a sequence, through the C ABI only.

    Chunk-Recurrent Training Framework item: the sequence is processed chunk by
    chunk.  Forward, chunks in order: chunk c selects its Top-K past pages from
    the representatives of the pages written so far, attends them plus its own
    pages, and the same forward call writes the representatives of its own
    pages (they become candidates for the later chunks).  Backward, chunks in
    reverse: the same selections are reused and every chunk adds its dK/dV into
    the paged gradient buffers of ``kv`` in place.  O and LSE of each chunk are
    kept for its backward (the attention itself is recomputed inside the
    backward).

    q_full, dout_full: ``[T, Hq, D]``, the tokens at positions [start, start + T)
    (start and chunk_len multiples of P, so that every chunk starts on a page;
    when T is not a multiple of chunk_len the last chunk is shorter, and when
    start + T is not a multiple of P it ends in a partial page).  reps: float
    ``[num_pages, Hkv, D]`` holding the representatives of the pages before
    ``start`` (computed here from the pool if None).  Returns
    ``(o_full, dq_full, sels)``; sels[c] is ``[Hkv, n_sel_c]``.
    """
    t, hq, d = q_full.shape
    ns, hkv, p, _ = kv.k.shape
    n_pages = kv.page_table.numel()
    if t < 1 or chunk_len < 1 or chunk_len % p or start % p or start + t > n_pages * p:
        raise OombError(OOMB_ERR_INVALID_ARG, "chunks must start on pages inside the cache")
    dev = q_full.device
    if reps is None:
        reps = torch.empty((n_pages, hkv, d), dtype=torch.float32, device=dev)
        if start:
            ws_r = workspace(OOMB_OP_PAGE_REPS, kv)
            oomb_page_reps(kv, 0, start // p, reps, ws_r, stream)
    ws_s = workspace(OOMB_OP_SELECT_TOPK, kv, hq, chunk_len, top_k)
    ws_f = workspace(OOMB_OP_ATTN_FWD, kv, hq, chunk_len)
    ws_b = workspace(OOMB_OP_ATTN_BWD, kv, hq, chunk_len)
    o_full = torch.empty_like(q_full)
    o_lo_full = o_residual_like(o_full)
    dq_full = torch.empty_like(q_full)
    lses, sels = [], []
    n_chunks = -(-t // chunk_len)                 # the last chunk may be shorter
    for c in range(n_chunks):
        r0 = c * chunk_len
        t0 = start + r0
        q = q_full[r0:r0 + chunk_len]
        n_sel = min(top_k, t0 // p)
        sel = torch.zeros((hkv, max(n_sel, 1)), dtype=torch.int32, device=dev)
        if n_sel:
            oomb_select_topk(q, t0, reps, kv, n_sel, sel, ws_s, stream=stream)
        lse = torch.empty((hq, q.shape[0]), dtype=torch.float32, device=dev)
        oomb_sparse_attn_fwd_own_reps(q, kv, sel, n_sel, t0, o_full[r0:r0 + chunk_len], lse, reps,
                                      ws_f, scale, stream, o_lo=_rows(o_lo_full, r0, chunk_len))
        lses.append(lse)
        sels.append((sel, n_sel))
    for c in reversed(range(n_chunks)):
        r0 = c * chunk_len
        sel, n_sel = sels[c]
        oomb_sparse_attn_bwd(q_full[r0:r0 + chunk_len], o_full[r0:r0 + chunk_len],
                             dout_full[r0:r0 + chunk_len], lses[c], kv, sel, n_sel, start + r0,
                             dq_full[r0:r0 + chunk_len], ws_b, scale, stream,
                             o_lo=_rows(o_lo_full, r0, chunk_len))
    for w in (ws_s, ws_f, ws_b):
        code, where, blk = oomb_device_status(w, stream)
        if code != OOMB_OK:
            raise OombError(code, f"device status (where {where}, block {blk})")
    return o_full, dq_full, [s[:, :n] for s, n in sels]


# ---------------------------------------------------------------------------
# Host-tier pools with a device page cache (oomb_offload_* in oomb.h).
# ---------------------------------------------------------------------------
class OffloadCache:
    """A device cache of ``cache_slots`` page slots in front of host pools.

    host: a PagedKV whose k, v (and dk, dv) are pinned CPU tensors
    ``[num_host_slots, Hkv, P, D]`` -- or, without staging, device tensors (a
    compact tier in HBM) -- and whose page_table is a CPU int32 tensor (logical
    page -> host slot).  k and v may be ``torch.float8_e4m3fn`` (an fp8 KV
    cache, expanded to bf16 tile by tile as it is fetched; dk/dv bf16).  The
    cache pools (and, with staging_bytes > 0, the device staging buffer the
    moves go through) are allocated here on ``device`` (torch); the library's
    handle holds only host state.
    """

    def __init__(self, host: PagedKV, cache_slots: int, device="cuda", staging_bytes=0):
        ns, hkv, p, d = host.k.shape
        self.host = host
        self.num_pages = host.page_table.numel()
        self.page_size, self.hkv, self.head_dim = p, hkv, d
        self.cache_slots = cache_slots
        fp8 = host.k.dtype == torch.float8_e4m3fn
        cdt = torch.bfloat16 if fp8 else host.k.dtype   # what the kernels compute on
        shape = (cache_slots, hkv, p, d)
        self.ck = torch.empty(shape, dtype=cdt, device=device)
        self.cv = torch.empty(shape, dtype=cdt, device=device)
        grads = host.dk is not None
        self.cdk = torch.empty(shape, dtype=cdt, device=device) if grads else None
        self.cdv = torch.empty(shape, dtype=cdt, device=device) if grads else None
        self._pt_host = host.page_table.to(torch.int32).contiguous()
        # staging_bytes > 0: moves through a device staging buffer and the copy
        # engines; 0: zero-copy copy kernel
        self.staging = (torch.empty(staging_bytes, dtype=torch.uint8, device=device)
                        if staging_bytes else None)
        dt = OOMB_BF16 if cdt == torch.bfloat16 else OOMB_FP32
        ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
        desc = OombOffloadDesc(ptr(host.k), ptr(host.v), ptr(host.dk), ptr(host.dv),
                               self._pt_host.data_ptr(), self.num_pages, ns, p, hkv, d, dt,
                               ptr(self.ck), ptr(self.cv), ptr(self.cdk), ptr(self.cdv),
                               cache_slots, ptr(self.staging), staging_bytes,
                               OOMB_FP8_E4M3 if fp8 else dt)
        h = ctypes.c_void_p()
        _check(load().oomb_offload_create(ctypes.byref(desc), ctypes.byref(h)))
        self._h = h

    def pass_state(self, dev, hq, chunk_len, top_k) -> dict:
        """The copy stream, device page tables and workspaces of
        chunk_recurrent_pass_offloaded for these shapes, made on first use and
        kept, so that a pass does not allocate them each time."""
        key = (str(dev), hq, chunk_len, top_k)
        cached = getattr(self, "_pass_states", None)
        if cached is None:
            cached = self._pass_states = {}
        if key not in cached:
            pts = [torch.full((self.num_pages,), -1, dtype=torch.int32, device=dev)
                   for _ in range(3)]
            kv0 = self.device_kv(pts[0])
            cached[key] = {
                "copy": torch.cuda.Stream(dev, priority=-1),
                "pts": pts[:2], "pt_last": pts[2],
                "ws": [workspace(OOMB_OP_PAGE_REPS, kv0),
                       workspace(OOMB_OP_SELECT_TOPK, kv0, hq, chunk_len, top_k),
                       workspace(OOMB_OP_ATTN_FWD, kv0, hq, chunk_len),
                       workspace(OOMB_OP_ATTN_BWD, kv0, hq, chunk_len)]}
        return cached[key]

    def device_kv(self, page_table_dev) -> PagedKV:
        """The cache as a PagedKV for the chunk whose acquire wrote page_table_dev."""
        return PagedKV(self.ck, self.cv, page_table_dev, self.cdk, self.cdv)

    def acquire(self, sel_host, n_sel, chunk_start, chunk_len, with_grads, page_table_dev,
                stream=None):
        """sel_host: CPU int32 ``[Hkv, n_sel]`` (or None when n_sel == 0)."""
        sp = None
        if n_sel:
            sel_host = sel_host[:, :n_sel].to(torch.int32).contiguous()
            sp = ctypes.c_void_p(sel_host.data_ptr())
        _check(load().oomb_offload_acquire(self._h, sp, n_sel, chunk_start, chunk_len,
                                           1 if with_grads else 0, _ptr(page_table_dev),
                                           _stream(stream)))

    def flush(self, drop=False, stream=None):
        _check(load().oomb_offload_flush(self._h, 1 if drop else 0, _stream(stream)))

    def writeback(self, first_page, n_pages, stream=None):
        """Write the modified gradient tiles of these pages back now."""
        _check(load().oomb_offload_writeback(self._h, first_page, n_pages, _stream(stream)))

    def writeback_pages(self, pages, stream=None):
        """Write the modified gradient tiles of these logical pages back now."""
        pages = torch.as_tensor(list(pages), dtype=torch.int32).contiguous()
        _check(load().oomb_offload_writeback_pages(self._h, ctypes.c_void_p(pages.data_ptr()),
                                                   pages.numel(), _stream(stream)))

    def zero_grads(self):
        """Declare the host dK/dV pools zeroed (a new pass): the cached gradient
        tiles are dropped, and tiles still zero on the host are brought in as
        zero fills on the device instead of copies."""
        _check(load().oomb_offload_zero_grads(self._h))

    def stats(self) -> dict:
        out = (ctypes.c_int64 * 7)()
        _check(load().oomb_offload_stats(self._h, out))
        keys = ["tiles_in", "tiles_out", "bytes_in", "bytes_out", "acquires", "slots_reused",
                "tiles_zero_filled"]
        return dict(zip(keys, list(out)))

    def close(self):
        if getattr(self, "_h", None):
            load().oomb_offload_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def chunk_recurrent_pass_offloaded(q_full, dout_full, cache: OffloadCache, chunk_len, top_k,
                                   scale=0.0, start=0, reps=None, prefetch=True):
    """chunk_recurrent_pass with the pools in host memory behind ``cache``.

    Fourth optimisation of the method (asynchronous CPU offloading): each
    chunk's tiles are brought into the device cache by oomb_offload_acquire.
    With ``prefetch``, a second stream does the moves while the compute stream
    runs the attention: in the forward, chunk c+1's acquire overlaps chunk c's
    forward (the representatives of chunk c's pages and chunk c+1's selection,
    which need chunk c's tiles and every SM, run just before chunk c's forward),
    and the last chunk's gradient tiles come in during the forward of the chunk
    before it; in the backward, chunk c-1's acquire overlaps chunk c's
    backward, and chunk c's own pages -- final once its backward is done, since
    no earlier chunk reads them -- go back to the host during the backward of
    chunk c-1; during the last backward, every page the first chunk does not
    touch goes back as well, so the final flush moves only the first chunk's
    tiles.  O, the selections and the host dK/dV are bit-identical to
    chunk_recurrent_pass on resident pools (the same kernels run on bit copies
    of the same tiles, and every modified gradient tile is written back); dQ is
    equal up to the order of its fp32 atomic sums.

    reps: float ``[num_pages, Hkv, D]`` on the device with the representatives
    of the pages before ``start`` (required when start > 0: those pages are in
    host memory).  Returns ``(o_full, dq_full, sels)`` like chunk_recurrent_pass.
    """
    t, hq, d = q_full.shape
    p, hkv, n_pages = cache.page_size, cache.hkv, cache.num_pages
    if t < 1 or chunk_len < 1 or chunk_len % p or start % p or start + t > n_pages * p:
        raise OombError(OOMB_ERR_INVALID_ARG, "chunks must start on pages inside the cache")
    if start and reps is None:
        raise OombError(OOMB_ERR_INVALID_ARG, "reps of the pages before start are required")
    dev = q_full.device
    comp = torch.cuda.current_stream(dev)
    st = cache.pass_state(dev, hq, chunk_len, top_k)
    # the moves run at high priority: their CTAs are scheduled as soon as an SM
    # frees up between attention CTAs, rather than after the whole attention grid
    copy = st["copy"] if prefetch else comp
    copy.wait_stream(comp)                        # after everything before this pass
    # device page tables: chunks c and c+1 in flight use pts[c % 2]; the last
    # chunk's backward uses pt_last (written while its forward may still run)
    pts, pt_last = st["pts"], st["pt_last"]
    if reps is None:
        reps = torch.empty((n_pages, hkv, d), dtype=torch.float32, device=dev)
    kv0 = cache.device_kv(pts[0])
    ws_r, ws_s, ws_f, ws_b = st["ws"]
    o_full = torch.empty_like(q_full)
    o_lo_full = o_residual_like(o_full)
    dq_full = torch.empty_like(q_full)
    n_chunks = -(-t // chunk_len)                 # the last chunk may be shorter
    last = n_chunks - 1
    sels, lses = [None] * n_chunks, [None] * n_chunks

    def length(c):
        return min(chunk_len, t - c * chunk_len)
    ready, done = [None] * n_chunks, [None] * n_chunks
    ready_last = [None]

    def cur():
        return torch.cuda.current_stream(dev)

    def mark():
        ev = torch.cuda.Event()
        ev.record(cur())
        return ev

    def select(c):
        # on the current stream; needs the representatives of pages < t0 / P.
        # The selection is copied to pinned host memory behind it; host_sel
        # waits for that copy alone, not for what the stream does next.
        t0 = start + c * chunk_len
        n_sel = min(top_k, t0 // p)
        sel = torch.zeros((hkv, max(n_sel, 1)), dtype=torch.int32, device=dev)
        if n_sel:
            oomb_select_topk(q_full[c * chunk_len:(c + 1) * chunk_len], t0, reps, kv0, n_sel, sel,
                             ws_s, stream=cur())
        sel_h = torch.empty(sel.shape, dtype=torch.int32, pin_memory=True)
        sel_h.copy_(sel, non_blocking=True)
        return [sel, sel_h, n_sel, mark()]

    def host_sel(c):
        sels[c][3].synchronize()

    def acquire(c, grads, pt):
        host_sel(c)
        sel_h, n_sel = sels[c][1], sels[c][2]
        cache.acquire(sel_h, n_sel, start + c * chunk_len, length(c), grads, pt, cur())

    def acquire_fwd(c):
        acquire(c, False, pts[c % 2])
        ready[c] = mark()
        if c == last:
            # the last chunk's gradient tiles: same pages, so no slot is reused
            # while the forwards before it run
            acquire(c, True, pt_last)
            ready_last[0] = mark()

    # forward, chunks in order.  Chunk c+1's selection needs the representatives
    # of chunk c's pages, which need chunk c's tiles: on the copy stream, after
    # chunk c's acquire and between the forwards of chunks c-1 and c (the
    # selection is one kernel over every SM; run beside a forward it would
    # stall it), then chunk c+1's acquire runs beside chunk c's forward.
    # Chunk 0's own pages do not depend on its selection: they come in first,
    # and chunk 1's selection (which needs their representatives) runs while
    # the host plans the rest of chunk 0's acquire.
    early = prefetch and start > 0 and n_chunks > 1
    with torch.cuda.stream(copy):
        if early:
            cache.acquire(None, 0, start, length(0), False, pts[0], cur())
        sels[0] = select(0)
        if early:
            oomb_page_reps(cache.device_kv(pts[0]), start // p, chunk_len // p, reps, ws_r, copy)
            sels[1] = select(1)
        acquire_fwd(0)
    for c in range(n_chunks):
        r0 = c * chunk_len
        if c + 1 < n_chunks and not (early and c == 0):
            with torch.cuda.stream(copy):
                if c >= 1:
                    copy.wait_event(done[c - 1])
                oomb_page_reps(cache.device_kv(pts[c % 2]), (start + r0) // p, chunk_len // p,
                               reps, ws_r, copy)
                sels[c + 1] = select(c + 1)
                comp.wait_event(mark())
        comp.wait_event(ready[c])
        sel, n_sel = sels[c][0], sels[c][2]
        lses[c] = torch.empty((hq, length(c)), dtype=torch.float32, device=dev)
        oomb_sparse_attn_fwd(q_full[r0:r0 + chunk_len], cache.device_kv(pts[c % 2]), sel, n_sel,
                             start + r0, o_full[r0:r0 + chunk_len], lses[c], ws_f, scale, comp,
                             o_lo=_rows(o_lo_full, r0, chunk_len))
        done[c] = torch.cuda.Event()
        done[c].record(comp)
        if c + 1 < n_chunks:
            with torch.cuda.stream(copy):
                host_sel(c + 1)                   # before the wait: the host waits only for it
                if c >= 1:
                    copy.wait_event(done[c - 1])  # slots of chunk c-1 may be reused now
                acquire_fwd(c + 1)
    fwd_done = done[last]

    def touched(c):                               # the pages chunk c reads and adds into
        c0 = start + c * chunk_len
        own = set(range(c0 // p, -(-(c0 + length(c)) // p)))
        n_sel = sels[c][2]
        return own | (set(sels[c][1][:, :n_sel].flatten().tolist()) if n_sel else set())
    touched_first = touched(0)
    touched_later = set().union(*(touched(c) for c in range(1, n_chunks)))
    # backward, chunks in reverse
    for c in reversed(range(n_chunks)):
        r0 = c * chunk_len
        comp.wait_event(ready_last[0] if c == last else ready[c])
        sel, n_sel = sels[c][0], sels[c][2]
        pt = pt_last if c == last else pts[c % 2]
        oomb_sparse_attn_bwd(q_full[r0:r0 + chunk_len], o_full[r0:r0 + chunk_len],
                             dout_full[r0:r0 + chunk_len], lses[c], cache.device_kv(pt),
                             sel, n_sel, start + r0, dq_full[r0:r0 + chunk_len], ws_b, scale, comp,
                             o_lo=_rows(o_lo_full, r0, chunk_len))
        done[c] = torch.cuda.Event()
        done[c].record(comp)
        with torch.cuda.stream(copy):
            if c >= 1:
                # slots (and the page table) of the chunk before in comp order may be
                # reused now: the last forward for c == last, else backward c + 1
                copy.wait_event(fwd_done if c == last else done[c + 1])
                acquire(c - 1, True, pts[(c - 1) % 2])
                ready[c - 1] = mark()
            if c == 0 and n_chunks > 1:
                # during the last backward the link is otherwise idle: every page
                # that the first chunk neither owns nor selected is final (the
                # backward of chunk 1 is done), so its tiles go back now rather than
                # in the final flush.  (Doing the same after every chunk measured
                # slower: those moves took SMs from the backwards.)
                cache.writeback_pages(sorted(touched_later - touched_first), copy)
            # chunk c's own pages are final: no earlier chunk reads them
            copy.wait_event(done[c])
            cache.writeback((start + r0) // p, -(-length(c) // p), copy)
    comp.wait_stream(copy)
    cache.flush(stream=comp)
    for w in (ws_r, ws_f, ws_b):
        code, where, blk = oomb_device_status(w, comp)
        if code != OOMB_OK:
            raise OombError(code, f"device status (where {where}, block {blk})")
    return o_full, dq_full, [s[0][:, :s[2]] for s in sels]
