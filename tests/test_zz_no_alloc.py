"""oomb_select_topk_noalloc -- the Top-K selection for callers that cannot
allocate device memory (its scratch is a fixed array inside the library) --
must return exactly what oomb_select_topk returns with a caller workspace, on
two calls in a row (the second one reuses the scratch the first one left).

Kept in a file of its own that pytest collects last; it passes alone in a
fresh process and after the other tests.  The refusal of shapes larger than
the fixed scratch happens on the host before any CUDA call, so it is tested
without a GPU (tests/test_abi_cpu.py)."""
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

