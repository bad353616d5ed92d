"""C-ABI checks that need no GPU: the library loads, exports every function
declared in include/oomb.h, and rejects bad arguments on the host before any
launch (the pointers below are never dereferenced)."""
import ctypes
import os
import re

import pytest
import torch

from paged_sparse_attention_oomb_gb300 import oomb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(oomb.LIB_PATH):
        from paged_sparse_attention_oomb_gb300.build import build
        build()
    return oomb.load()


def _declared():
    with open(os.path.join(ROOT, "include", "oomb.h")) as f:
        txt = f.read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(oomb_[a-z_]+)\s*\(", txt)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(oomb.EXPORTED) == names


def test_status_strings(lib):
    assert oomb.oomb_status_string(0) == "OOMB_OK"
    assert oomb.oomb_status_string(4) == "OOMB_ERR_TIMEOUT"
    assert oomb.oomb_status_string(6) == "OOMB_ERR_NONFINITE"
    assert oomb.oomb_status_string(99) == "OOMB_ERR_UNKNOWN"


def test_validate_page_table_host(lib):
    oomb.oomb_validate_page_table_host([3, 0, 2, 1], 4)
    oomb.oomb_validate_page_table_host([5, 0], 8)
    with pytest.raises(oomb.OombError, match="outside"):
        oomb.oomb_validate_page_table_host([0, 4], 4)
    with pytest.raises(oomb.OombError, match="outside"):
        oomb.oomb_validate_page_table_host([-1, 0], 4)
    with pytest.raises(oomb.OombError, match="more than one page"):
        oomb.oomb_validate_page_table_host([1, 2, 1], 4)


FAKE = 1 << 20   # aligned, never dereferenced: every case below fails host checks first


def _kv(**kw):
    d = dict(k=FAKE, v=FAKE, dk=FAKE, dv=FAKE, page_table=FAKE, num_pages=64, num_slots=64,
             page_size=64, num_kv_heads=4, head_dim=128, dtype=oomb.OOMB_BF16)
    d.update(kw)
    return oomb.OombPagedKV(**d)


def _fwd(lib, kv, q=FAKE, n_sel=0, hq=28, clen=256, cstart=3840, ws=FAKE, ws_bytes=1 << 20,
         o_lo=0):
    return lib.oomb_sparse_attn_fwd(ctypes.c_void_p(q), ctypes.byref(kv), ctypes.c_void_p(FAKE),
                                    n_sel, hq, clen, cstart, 0.0, ctypes.c_void_p(FAKE),
                                    ctypes.c_void_p(o_lo) if o_lo else None,
                                    ctypes.c_void_p(FAKE), ctypes.c_void_p(ws), ws_bytes, None)


@pytest.mark.parametrize("kw,code,msg", [
    (dict(page_size=48), 2, "page_size"),
    (dict(head_dim=64), 2, "head_dim"),
    (dict(dtype=7), 1, "dtype"),
    (dict(dtype=oomb.OOMB_FP8_E4M3), 2, "storage format"),
    (dict(num_slots=0), 1, "num_slots"),
    (dict(num_kv_heads=0), 2, "num_kv_heads"),
    (dict(k=FAKE + 8), 1, "aligned"),
    (dict(page_table=0), 1, "page_table"),
])
def test_bad_cache_rejected(lib, kw, code, msg):
    rc = _fwd(lib, _kv(**kw))
    assert rc == code
    assert msg in oomb.oomb_last_error()


@pytest.mark.parametrize("args,msg", [
    (dict(hq=30), "multiple of Hkv"),
    (dict(clen=0), "chunk_len"),
    (dict(clen=-3), "chunk_len"),
    (dict(cstart=3968, clen=129), "runs past"),   # a partial page past the last one
    (dict(cstart=100), "chunk_start"),
    (dict(cstart=4032), "runs past"),
    (dict(n_sel=61), "n_sel"),
    (dict(n_sel=-1), "n_sel"),
    (dict(ws_bytes=16), "ws has"),
    (dict(ws=FAKE + 64), "256-byte"),
    (dict(q=FAKE + 4), "aligned"),
    (dict(o_lo=FAKE + 8), "aligned"),
])
def test_bad_call_rejected(lib, args, msg):
    rc = _fwd(lib, _kv(), **args)
    assert rc == oomb.OOMB_ERR_INVALID_ARG
    assert msg in oomb.oomb_last_error()


@pytest.mark.parametrize("reps,msg", [(0, "reps must be set"), (FAKE + 4, "16-byte")])
def test_fwd_own_reps_checks_reps(lib, reps, msg):
    kv = _kv()
    rc = lib.oomb_sparse_attn_fwd_own_reps(ctypes.c_void_p(FAKE), ctypes.byref(kv),
                                           ctypes.c_void_p(FAKE), 8, 28, 256, 3840, 0.0,
                                           ctypes.c_void_p(FAKE), None, ctypes.c_void_p(FAKE),
                                           ctypes.c_void_p(reps) if reps else None,
                                           ctypes.c_void_p(FAKE), 1 << 30, None)
    assert rc == oomb.OOMB_ERR_INVALID_ARG and msg in oomb.oomb_last_error()


def test_offload_calls_refuse_a_null_handle(lib):
    assert lib.oomb_offload_zero_grads(None) == oomb.OOMB_ERR_INVALID_ARG
    assert lib.oomb_offload_flush(None, 0, None) == oomb.OOMB_ERR_INVALID_ARG
    assert lib.oomb_offload_writeback(None, 0, 1, None) == oomb.OOMB_ERR_INVALID_ARG
    pages = (ctypes.c_int32 * 1)(0)
    assert lib.oomb_offload_writeback_pages(None, pages, 1, None) == oomb.OOMB_ERR_INVALID_ARG
    out = (ctypes.c_int64 * 7)()
    assert lib.oomb_offload_stats(None, out) == oomb.OOMB_ERR_INVALID_ARG


def test_offload_create_checks_memory_kinds(lib):
    """The host pools must be pinned host memory and the cache pools device
    memory; a plain host buffer is refused before anything is allocated."""
    buf = (ctypes.c_uint8 * (1 << 16))()
    pt = (ctypes.c_int32 * 4)(0, 1, 2, 3)
    a = ctypes.addressof(buf)
    d = oomb.OombOffloadDesc(a, a, None, None, ctypes.addressof(pt), 4, 4, 16, 1, 128,
                             oomb.OOMB_BF16, a, a, None, None, 2)
    h = ctypes.c_void_p()
    rc = lib.oomb_offload_create(ctypes.byref(d), ctypes.byref(h))
    assert rc == oomb.OOMB_ERR_INVALID_ARG and "pinned host memory" in oomb.oomb_last_error()
    assert not h.value
    d.cache_slots = 0
    assert lib.oomb_offload_create(ctypes.byref(d), ctypes.byref(h)) == oomb.OOMB_ERR_INVALID_ARG
    d.cache_slots, d.dk = 2, a                     # dk without dv / cache grads
    rc = lib.oomb_offload_create(ctypes.byref(d), ctypes.byref(h))
    assert rc == oomb.OOMB_ERR_INVALID_ARG and "all set or all NULL" in oomb.oomb_last_error()
    d.dk = None
    # fp8 K/V pools: only in front of a bf16 cache, and only with zero-copy moves
    d.backing_kv_dtype, d.dtype = oomb.OOMB_FP8_E4M3, oomb.OOMB_FP32
    rc = lib.oomb_offload_create(ctypes.byref(d), ctypes.byref(h))
    assert rc == oomb.OOMB_ERR_INVALID_ARG and "backing_kv_dtype" in oomb.oomb_last_error()
    d.dtype, d.dev_staging, d.dev_staging_bytes = oomb.OOMB_BF16, a, 1 << 16
    rc = lib.oomb_offload_create(ctypes.byref(d), ctypes.byref(h))
    assert rc == oomb.OOMB_ERR_UNSUPPORTED and "zero-copy" in oomb.oomb_last_error()
    assert not h.value


def _bwd(lib, kv, o_lo=None):
    return lib.oomb_sparse_attn_bwd(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE),
                                    ctypes.c_void_p(o_lo) if o_lo else None,
                                    *(ctypes.c_void_p(FAKE),) * 2, ctypes.byref(kv),
                                    ctypes.c_void_p(FAKE), 0, 28, 256, 3840, 0.0,
                                    ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1 << 30, None)


def test_bwd_requires_grad_buffers(lib):
    rc = _bwd(lib, _kv(dk=0))
    assert rc == oomb.OOMB_ERR_INVALID_ARG and "dk" in oomb.oomb_last_error()


def test_o_residual_checks(lib):
    """The residual of O is a bf16 buffer: misaligned, or given with fp32
    pools, it is refused on the host."""
    rc = _bwd(lib, _kv(), o_lo=FAKE + 2)
    assert rc == oomb.OOMB_ERR_INVALID_ARG and "aligned" in oomb.oomb_last_error()
    kv32 = _kv(head_dim=64, dtype=oomb.OOMB_FP32)
    rc = _bwd(lib, kv32, o_lo=FAKE)
    assert rc == oomb.OOMB_ERR_INVALID_ARG and "o_lo" in oomb.oomb_last_error()
    rc = _fwd(lib, kv32, o_lo=FAKE)
    assert rc == oomb.OOMB_ERR_INVALID_ARG and "o_lo" in oomb.oomb_last_error()


def test_select_rejects_bad_pages(lib):
    kv = _kv()
    rc = lib.oomb_page_reps(ctypes.byref(kv), 60, 8, ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE),
                            256, None)
    assert rc == oomb.OOMB_ERR_INVALID_ARG and "outside" in oomb.oomb_last_error()
    rc = lib.oomb_select_topk(ctypes.c_void_p(FAKE), 28, 256, 3840, ctypes.c_void_p(FAKE),
                              ctypes.byref(kv), -3, ctypes.c_void_p(FAKE), None,
                              ctypes.c_void_p(FAKE), 1 << 20, None)
    assert rc == oomb.OOMB_ERR_INVALID_ARG and "top_k" in oomb.oomb_last_error()


def test_workspace_sizes(lib):
    kv = _kv(num_pages=32768, num_slots=32768, page_size=128)
    bwd = lib.oomb_workspace_bytes(oomb.OOMB_OP_ATTN_BWD, ctypes.byref(kv), 28, 8192, 0)
    # status block + Delta and lse*log2(e) [28][8192] each + fp32 dq accumulator [8192][28][128]
    assert bwd == 256 + 2 * 28 * 8192 * 4 + 8192 * 28 * 128 * 4
    assert lib.oomb_workspace_bytes(oomb.OOMB_OP_ATTN_FWD, ctypes.byref(kv), 28, 8192, 0) == 256
    sel = lib.oomb_workspace_bytes(oomb.OOMB_OP_SELECT_TOPK, ctypes.byref(kv), 28, 8192, 128)
    assert sel >= 256 + 4 * 32768 * 4
    assert lib.oomb_workspace_bytes(99, ctypes.byref(kv), 0, 0, 0) == 0


def test_noalloc_selection_refuses_oversized_shapes_on_the_host(lib):
    kv = _kv(num_pages=1 << 20, num_slots=1 << 20, page_size=16)   # scores alone: 16 MiB
    rc = lib.oomb_select_topk_noalloc(ctypes.c_void_p(FAKE), 28, 256, 4096, ctypes.c_void_p(FAKE),
                                      ctypes.byref(kv), 64, ctypes.c_void_p(FAKE), None, None)
    assert rc == oomb.OOMB_ERR_INVALID_ARG and "fixed scratch" in oomb.oomb_last_error()


@pytest.mark.parametrize("t,chunk_len,start", [(48, 24, 0), (48, 16, 8), (80, 16, 0), (0, 16, 0)])
def test_chunk_recurrent_pass_checks_its_chunks_on_the_host(t, chunk_len, start):
    """Chunks must start on pages inside the cache (chunk_len and start multiples
    of P, the sequence within the pages); refused before anything runs."""
    pool = torch.zeros((4, 1, 16, 64))
    kv = oomb.PagedKV(pool, pool, torch.arange(4, dtype=torch.int32))
    q = torch.zeros((t, 2, 64))
    with pytest.raises(oomb.OombError) as e:
        oomb.chunk_recurrent_pass(q, q, kv, chunk_len, 1, start=start)
    assert e.value.code == oomb.OOMB_ERR_INVALID_ARG
