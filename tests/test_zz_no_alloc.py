"""oomb_select_topk_noalloc -- the Top-K selection for callers that cannot
allocate device memory (its scratch is a fixed array inside the library) --
must return exactly what oomb_select_topk returns with a caller workspace, on
two calls in a row (the second one reuses the scratch the first one left).

Kept in a file of its own that pytest collects last; it passes alone in a
fresh process and after the other tests."""
import pytest
import torch

from paged_sparse_attention_oomb_gb300 import oomb
from paged_sparse_attention_oomb_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oomb.load()


def _select(x, kv, reps, top_k, noalloc):
    wl = x.wl
    n_sel = min(top_k, wl.num_candidates)
    sel = torch.full((wl.num_kv_heads, n_sel), -1, dtype=torch.int32, device=DEV)
    scores = torch.full((wl.num_kv_heads, wl.num_pages), float("nan"), device=DEV)
    if noalloc:
        oomb.oomb_select_topk_noalloc(x.q, wl.start, reps, kv, top_k, sel, scores=scores)
    else:
        ws = oomb.workspace(oomb.OOMB_OP_SELECT_TOPK, kv, wl.num_q_heads, wl.chunk_len, top_k)
        oomb.oomb_select_topk(x.q, wl.start, reps, kv, top_k, sel, ws, scores=scores)
    torch.cuda.synchronize()
    return sel, scores


@pytest.mark.parametrize("wl", [
    Workload("noalloc_ctx256k_k64", "bf16", 28, 4, 128, 262144, 64, 4096, 64),
    Workload("noalloc_shuffled_k37", "bf16", 8, 2, 128, 65536, 128, 1024, 37, shuffled=True),
], ids=lambda w: w.name)
def test_noalloc_matches_workspace_call_twice(wl):
    x = make_inputs(wl, seed=6, device=DEV)
    kv = oomb.PagedKV(x.k_pool, x.v_pool, x.page_table)
    n = wl.num_pages
    reps = torch.empty((n, wl.num_kv_heads, wl.head_dim), dtype=torch.float32, device=DEV)
    oomb.oomb_page_reps(kv, 0, n, reps, oomb.workspace(oomb.OOMB_OP_PAGE_REPS, kv))
    ref_sel, ref_scores = _select(x, kv, reps, wl.top_k, noalloc=False)
    for _ in range(2):
        sel, scores = _select(x, kv, reps, wl.top_k, noalloc=True)
        assert torch.equal(sel, ref_sel)
        assert torch.equal(scores, ref_scores)


def test_noalloc_refuses_shapes_beyond_its_scratch():
    import ctypes
    n_pages, p = 1 << 19, 16                  # scores alone: 4 heads x 2^19 pages x 4 B = 8 MiB
    q = torch.zeros((4096, 28, 128), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((1, 4, p, 128), dtype=torch.bfloat16, device=DEV)
    kv = oomb.PagedKV(k, k, torch.zeros(1, dtype=torch.int32, device=DEV))
    s = kv.struct()
    s.num_pages = s.num_slots = n_pages       # shapes only: the call refuses before any launch
    reps = torch.zeros(16, device=DEV)
    sel = torch.zeros((4, 64), dtype=torch.int32, device=DEV)
    rc = oomb.load().oomb_select_topk_noalloc(
        ctypes.c_void_p(q.data_ptr()), 28, 4096, n_pages * p - 4096,
        ctypes.c_void_p(reps.data_ptr()), ctypes.byref(s), 64, ctypes.c_void_p(sel.data_ptr()),
        None, None)
    assert rc == oomb.OOMB_ERR_INVALID_ARG
    assert "fixed scratch" in oomb.oomb_last_error()
