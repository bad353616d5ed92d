"""Top-K selection with exactly equal scores (GB300 only).

The method picks, per (chunk, KV head), the Top-K past pages by the score of
their representative vectors; when scores are equal the lower page index wins
and the selection is written in ascending page order.  Random keys never tie
in fp32, so these cases build pages whose keys are one constant per page
(every row and column of the page the same value) and a chunk of all-ones
queries: the representative is that constant, the group-mean query is exactly
1, and the score is exactly D times the constant on both the GPU and the
oracle.  Pages that share a constant tie exactly, and different constants
are far apart, so no near-tie can excuse a difference: every case asserts the
GPU selection equal, element for element, to the oracle's.

Cases: (a) groups of identical pages with the K-th page inside a group;
(b) every candidate identical (a degenerate score range); (c) thousands of
candidates whose scores fall in one narrow band between two far outliers,
so that one value bin holds more keys than the exact ranking inside a bin
takes; (d) more candidates than the selection caches on chip.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_sparse_attention_oomb_gb300 import oomb
from paged_sparse_attention_oomb_gb300.workloads import Inputs, Workload, to_numpy64

from parity_util import gpu_kv, gpu_reps, gpu_select, oracle_selection

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oomb.load()


def constant_pages(levels, page_size=16, own_pages=4, num_q_heads=4, seed=0):
    """Inputs whose candidate page l of KV head g holds the constant levels[l, g]
    in every key entry; the chunk (all-ones queries) is the last own_pages
    pages.  Pools are stored by a shuffled page table."""
    levels = np.asarray(levels, np.float64)
    n_cand, hkv = levels.shape
    n = n_cand + own_pages
    p, d = page_size, 128
    c = own_pages * p
    wl = Workload("ties", "bf16", num_q_heads, hkv, d, n * p, p, c, 1, shuffled=True)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    vals = torch.zeros((n, hkv), dtype=torch.float32)
    vals[:n_cand] = torch.as_tensor(levels, dtype=torch.float32)
    k_logical = vals[:, :, None, None].expand(n, hkv, p, d).to(torch.bfloat16)
    assert torch.equal(k_logical[:n_cand, :, 0, 0].double(),
                       torch.as_tensor(levels)), "levels must be bf16 values"
    pt = torch.randperm(n, generator=g).to(torch.int32)
    k_pool = torch.empty_like(k_logical)
    k_pool[pt.long()] = k_logical
    v_pool = torch.zeros_like(k_pool)
    q = torch.ones((c, num_q_heads, d), dtype=torch.bfloat16)
    return Inputs(wl, q.to(DEV), k_pool.to(DEV), v_pool.to(DEV), torch.zeros_like(q).to(DEV),
                  pt.to(DEV))


def check_exact(x, top_k):
    """GPU selection == oracle selection, element for element (no exemption)."""
    kv = gpu_kv(x, with_grads=False)
    reps = gpu_reps(kv)
    reps64 = oracle.page_reps(to_numpy64(x.k_pool), to_numpy64(x.page_table))
    sel_g, scores_g = gpu_select(x, kv, reps, top_k)
    sel_o, scores_o = oracle_selection(x, reps64, top_k)
    nc = x.wl.num_candidates
    assert np.array_equal(scores_g[:, :nc].cpu().numpy(), scores_o), "scores must be exact"
    g = sel_g.cpu().numpy()
    assert g.shape == sel_o.shape
    for h in range(g.shape[0]):
        assert np.array_equal(g[h], sel_o[h]), (h, np.setdiff1d(g[h], sel_o[h])[:8],
                                                np.setdiff1d(sel_o[h], g[h])[:8])
    return sel_o


def _groups(n_cand, hkv, values, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(values, n_cand) for _ in range(hkv)], axis=1)


@pytest.mark.parametrize("boundary", ["first", "inside_group", "last_of_group", "all_but_one"])
def test_identical_pages_tie_to_the_lower_index(boundary):
    values = np.array([-1.5, -1.0, -0.5, 0.25, 0.5, 1.0, 1.25, 2.0])
    levels = _groups(509, 2, values, seed=3)
    x = constant_pages(levels)
    # per head, the count of pages strictly above the 4th-highest value, and of that value
    lv = levels[:, 0]
    above, at = int(np.sum(lv > 0.5)), int(np.sum(lv == 0.5))
    top_k = {"first": 1, "inside_group": above + at // 2, "last_of_group": above + at,
             "all_but_one": levels.shape[0] - 1}[boundary]
    sel = check_exact(x, top_k)
    if boundary == "inside_group":
        # head 0 keeps every page above 0.5 and the lowest-indexed half of the 0.5 pages
        ties = np.flatnonzero(lv == 0.5)
        kept = np.intersect1d(sel[0], ties)
        assert np.array_equal(kept, ties[:at // 2])


@pytest.mark.parametrize("top_k", [1, 37, 500])
def test_every_candidate_identical(top_k):
    """A degenerate score range (smallest == largest score): the K lowest page
    indices win."""
    x = constant_pages(np.full((501, 2), 0.75))
    sel = check_exact(x, top_k)
    assert np.array_equal(sel[0], np.arange(top_k)) and np.array_equal(sel[1], np.arange(top_k))


def test_identical_but_one_outlier():
    levels = np.full((300, 2), -0.25)
    levels[217, 0] = 3.0
    levels[5, 1] = 3.0
    sel = check_exact(constant_pages(levels), 10)
    assert np.array_equal(sel[0], np.r_[0:9, 217]) and np.array_equal(sel[1], np.arange(10))


@pytest.mark.parametrize("top_k", [100, 3000])
def test_overfull_value_bin(top_k):
    """About 6000 candidates in a narrow band (scores 128..255, shared by ~47
    pages each) between two far outliers (+-128000): almost every key lands in
    one of 2048 equal-width bins, more than the exact in-bin ranking takes."""
    rng = np.random.default_rng(7)
    band = 1.0 + rng.integers(0, 128, size=(6000, 2)) / 128.0
    band[11, :] = 1000.0
    band[4000, :] = -1000.0
    check_exact(constant_pages(band), top_k)


def test_more_candidates_than_cached_on_chip():
    """50,000 candidates per KV head (more than the selection keeps in shared
    memory), with ties across the boundary."""
    values = np.array([-0.5, 0.125, 0.25, 0.375, 0.5])
    levels = _groups(50_000, 1, values, seed=9)
    top_k = int(np.sum(levels[:, 0] > 0.375)) + 17
    check_exact(constant_pages(levels, num_q_heads=2), top_k)


def given_reps(levels, own_pages=4):
    """Inputs of constant_pages (all-ones queries, so the group-mean query is
    exactly 1) with representatives given directly: candidate l of KV head g
    is levels[l, g] in every column, signed zeros and NaN included, so its
    score is exactly D times that value on both sides."""
    levels = np.asarray(levels, np.float64)
    n_cand, hkv = levels.shape
    x = constant_pages(np.zeros_like(levels), own_pages=own_pages)
    reps64 = np.zeros((n_cand + own_pages, hkv, 128))
    reps64[:n_cand] = levels[:, :, None]
    reps = torch.as_tensor(reps64, dtype=torch.float32, device=DEV)
    return x, reps, reps64


@pytest.mark.parametrize("n_cand", [300, 700])
@pytest.mark.parametrize("boundary", ["among_zeros", "among_nan"])
def test_signed_zeros_tie_and_nan_ranks_last(n_cand, boundary):
    """Scores of +0 and -0 are equal (the lower page wins between them), +-inf
    rank as the largest and smallest numbers, and a NaN score never outranks
    a number: NaN pages are taken last, lowest index first.  300 candidates
    keep the boundary list short (ranked by counting), 700 make it longer
    (sorted)."""
    rng = np.random.default_rng(13 + n_cand)
    levels = rng.choice(np.array([np.inf, 0.5, -0.5, -np.inf, 0.0, -0.0, np.nan]),
                        size=(n_cand, 2), p=[0.05, 0.3, 0.15, 0.05, 0.15, 0.15, 0.15])
    assert np.any(np.signbit(levels) & (levels == 0)), "the draw holds -0 pages"
    x, reps, reps64 = given_reps(levels)
    lv = levels[:, 0]
    above, zeros, nans = int(np.sum(lv > 0)), int(np.sum(lv == 0)), int(np.sum(np.isnan(lv)))
    top_k = above + zeros // 2 if boundary == "among_zeros" else n_cand - nans // 2
    kv = gpu_kv(x, with_grads=False)
    sel_g, scores_g = gpu_select(x, kv, reps, top_k)
    sel_o, scores_o = oracle_selection(x, reps64, top_k)
    nc = x.wl.num_candidates
    np.testing.assert_array_equal(scores_g[:, :nc].cpu().numpy(), scores_o)   # NaN == NaN, -0 == +0
    g = sel_g.cpu().numpy()
    for h in range(2):
        assert np.array_equal(g[h], sel_o[h]), (h, np.setdiff1d(g[h], sel_o[h])[:8],
                                                np.setdiff1d(sel_o[h], g[h])[:8])
    if boundary == "among_zeros":
        zero_pages = np.flatnonzero(lv == 0)      # +0 and -0 pages in page order
        assert np.array_equal(np.intersect1d(g[0], zero_pages), zero_pages[:zeros // 2])
        assert not np.any(np.isnan(lv[g[0]]))
    else:
        nan_pages = np.flatnonzero(np.isnan(lv))
        taken = top_k - (n_cand - nans)            # every number first, then NaN pages
        assert np.array_equal(np.intersect1d(g[0], nan_pages), nan_pages[:taken])
