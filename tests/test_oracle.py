"""Pins of the CPU oracle against things other than itself (CPU only).

* torch's CPU scaled-dot-product attention + autograd (float64) pins the
  dense causal reference, including the GQA head mapping and the scale;
* the dense reference pins the sparse oracle with K = all pages;
* hand-derived closed forms (tests/golden/) pin selection, attention and
  gradients on worked examples;
* invariants: softmax rows sum to one, central finite differences, cross-chunk
  accumulation equals the single-pass gradient, brute-force pair means equal
  the representative-vector score, Top-K order invariants.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng_case(t=96, hq=4, hkv=2, d=8, p=8, seed=1, shuffle=True):
    rng = np.random.default_rng(seed)
    n = t // p
    k_log = rng.normal(size=(n, hkv, p, d)) + 0.5 * rng.normal(size=(n, hkv, 1, d))
    v_log = rng.normal(size=(n, hkv, p, d))
    pt = rng.permutation(n) if shuffle else np.arange(n)
    k_pool = np.empty_like(k_log); v_pool = np.empty_like(v_log)
    k_pool[pt] = k_log; v_pool[pt] = v_log
    q = rng.normal(size=(t, hq, d))
    do = rng.normal(size=(t, hq, d))
    return dict(q=q, do=do, k_log=k_log, v_log=v_log, k_pool=k_pool, v_pool=v_pool, pt=pt,
                n=n, p=p, hq=hq, hkv=hkv, d=d, t=t)


def _flat(pool_log):
    n, hkv, p, d = pool_log.shape
    return pool_log.transpose(0, 2, 1, 3).reshape(n * p, hkv, d)


# ---------------------------------------------------------------------------
# dense reference vs torch (library routine)
# ---------------------------------------------------------------------------
def test_dense_reference_matches_torch_sdpa():
    c = _rng_case(t=40, hq=6, hkv=2, d=8, p=8)
    k, v = _flat(c["k_log"]), _flat(c["v_log"])
    o, lse, dq, dk, dv = oracle.dense_causal_reference(c["q"], k, v, c["do"])
    grp = c["hq"] // c["hkv"]
    tq = torch.tensor(c["q"]).permute(1, 0, 2).requires_grad_(True)
    tk = torch.tensor(k).permute(1, 0, 2).requires_grad_(True)
    tv = torch.tensor(v).permute(1, 0, 2).requires_grad_(True)
    ko = tk.repeat_interleave(grp, dim=0)
    vo = tv.repeat_interleave(grp, dim=0)
    to = torch.nn.functional.scaled_dot_product_attention(tq, ko, vo, is_causal=True)
    to.backward(torch.tensor(c["do"]).permute(1, 0, 2))
    np.testing.assert_allclose(o, to.detach().permute(1, 0, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.permute(1, 0, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.permute(1, 0, 2).numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.permute(1, 0, 2).numpy(), atol=1e-12)
    s = (tq @ ko.transpose(1, 2)) / math.sqrt(c["d"])
    s = s.masked_fill(~torch.tril(torch.ones(40, 40, dtype=torch.bool)), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).detach().numpy(), atol=1e-12)


# ---------------------------------------------------------------------------
# sparse oracle with K = all equals the dense reference
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("shuffle", [False, True])
def test_sparse_all_pages_equals_dense(shuffle):
    c = _rng_case(t=96, hq=4, hkv=2, d=8, p=8, shuffle=shuffle)
    t0, clen = 48, 48
    n_cand = t0 // c["p"]
    sel = np.tile(np.arange(n_cand, dtype=np.int32), (c["hkv"], 1))
    qc, doc = c["q"][t0:], c["do"][t0:]
    o, lse = oracle.attn_fwd(qc, c["k_pool"], c["v_pool"], c["pt"], sel, t0, c["p"])
    dq, dk_acc, dv_acc = oracle.attn_bwd(qc, c["k_pool"], c["v_pool"], c["pt"], sel, t0, c["p"],
                                         o, lse, doc)
    do_full = np.zeros_like(c["do"]); do_full[t0:] = doc
    od, lsed, dqd, dkd, dvd = oracle.dense_causal_reference(
        c["q"], _flat(c["k_log"]), _flat(c["v_log"]), do_full)
    np.testing.assert_allclose(o, od[t0:], atol=1e-12)
    np.testing.assert_allclose(lse, lsed[:, t0:], atol=1e-12)
    np.testing.assert_allclose(dq, dqd[t0:], atol=1e-12)
    np.testing.assert_allclose(_flat(dk_acc), dkd, atol=1e-12)
    np.testing.assert_allclose(_flat(dv_acc), dvd, atol=1e-12)
    rows = np.array([0, 7, 31, 47])
    dqr = oracle.attn_dq_rows(qc, c["k_pool"], c["v_pool"], c["pt"], sel, t0, c["p"], o[rows],
                              lse[:, rows], doc, rows)
    np.testing.assert_allclose(dqr, dqd[t0 + rows], atol=1e-12)
    kvh = [1]
    o1, lse1 = oracle.attn_fwd(qc, c["k_pool"], c["v_pool"], c["pt"], sel, t0, c["p"], kv_heads=kvh)
    dkp, dvp = oracle.attn_bwd_pages(qc, c["k_pool"], c["v_pool"], c["pt"], sel, t0, c["p"], o1,
                                     lse1, doc, 1, [2, 7, 9])
    np.testing.assert_allclose(dkp, dkd.reshape(-1, 8, 2, 8)[[2, 7, 9], :, 1], atol=1e-12)
    np.testing.assert_allclose(dvp, dvd.reshape(-1, 8, 2, 8)[[2, 7, 9], :, 1], atol=1e-12)


def test_sparse_all_pages_equals_dense_tiny_fp32_workload():
    from paged_sparse_attention_oomb_gb300.workloads import WORKLOADS, make_inputs, to_numpy64
    wl = WORKLOADS["tiny_fp32_ctx1k"]
    x = make_inputs(wl)
    q, kp, vp, do, pt = (to_numpy64(x.q), to_numpy64(x.k_pool), to_numpy64(x.v_pool),
                         to_numpy64(x.do), to_numpy64(x.page_table))
    t0 = wl.start
    sel = np.arange(wl.num_candidates, dtype=np.int32)[None, :]
    o, lse = oracle.attn_fwd(q, kp, vp, pt, sel, t0, wl.page_size)
    kf = np.empty((wl.context, 1, wl.head_dim)); vf = np.empty_like(kf)
    kf[:] = _flat(kp[pt]); vf[:] = _flat(vp[pt])
    qf = np.zeros((wl.context, 2, wl.head_dim)); qf[t0:] = q
    dof = np.zeros_like(qf); dof[t0:] = do
    od, lsed, *_ = oracle.dense_causal_reference(qf, kf, vf, dof)
    np.testing.assert_allclose(o, od[t0:], atol=1e-12)
    np.testing.assert_allclose(lse, lsed[:, t0:], atol=1e-12)


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
def test_softmax_rows_sum_to_one():
    c = _rng_case(t=96, hq=4, hkv=2, d=8, p=8)
    t0 = 64
    sel = np.array([[0, 3, 5], [1, 2, 7]], np.int32)
    qc = c["q"][t0:]
    o, lse = oracle.attn_fwd(qc, c["k_pool"], c["v_pool"], c["pt"], sel, t0, c["p"])
    grp = c["hq"] // c["hkv"]
    for h in range(c["hq"]):
        g = h // grp
        kpos = oracle.key_positions(sel[g], t0, 32, c["p"])
        kk = c["k_log"][kpos // c["p"], g, kpos % c["p"]]
        s = qc[:, h] @ kk.T / math.sqrt(c["d"])
        allowed = kpos[None, :] <= (t0 + np.arange(32))[:, None]
        prob = np.where(allowed, np.exp(s - lse[h][:, None]), 0.0)
        np.testing.assert_allclose(prob.sum(axis=1), 1.0, atol=1e-12)


def test_finite_differences_sparse():
    c = _rng_case(t=96, hq=4, hkv=2, d=8, p=8, seed=3)
    t0, clen = 64, 32
    sel = np.array([[0, 3, 5], [1, 2, 7]], np.int32)
    qc, doc = c["q"][t0:].copy(), c["do"][t0:]
    kp, vp, pt, p = c["k_pool"].copy(), c["v_pool"].copy(), c["pt"], c["p"]

    def loss(qx, kx, vx):
        o, _ = oracle.attn_fwd(qx, kx, vx, pt, sel, t0, p)
        return float((o * doc).sum())

    o, lse = oracle.attn_fwd(qc, kp, vp, pt, sel, t0, p)
    dq, dk_acc, dv_acc = oracle.attn_bwd(qc, kp, vp, pt, sel, t0, p, o, lse, doc)
    rng = np.random.default_rng(7)
    eps = 1e-6
    for _ in range(6):
        i = (rng.integers(clen), rng.integers(c["hq"]), rng.integers(c["d"]))
        qa = qc.copy(); qa[i] += eps
        qb = qc.copy(); qb[i] -= eps
        fd = (loss(qa, kp, vp) - loss(qb, kp, vp)) / (2 * eps)
        assert abs(fd - dq[i]) < 1e-6 * max(1.0, abs(dq[i]))
    # keys/values in a selected page and in an own page, for each KV head
    for g in range(2):
        for lpage in (int(sel[g][1]), t0 // p + 2):
            for _ in range(2):
                off, dd = rng.integers(p), rng.integers(c["d"])
                idx = (pt[lpage], g, off, dd)
                for pool, grad in ((kp, dk_acc), (vp, dv_acc)):
                    orig = pool[idx]
                    pool[idx] = orig + eps; lp = loss(qc, kp, vp)
                    pool[idx] = orig - eps; lm = loss(qc, kp, vp)
                    pool[idx] = orig
                    fd = (lp - lm) / (2 * eps)
                    an = grad[lpage, g, off, dd]
                    assert abs(fd - an) < 1e-6 * max(1.0, abs(an)), (lpage, g, fd, an)
    # a page that is neither selected nor own gets exactly zero
    assert np.all(dk_acc[4] == 0) and np.all(dv_acc[4] == 0)


def test_cross_chunk_accumulation_equals_single_pass():
    c = _rng_case(t=128, hq=4, hkv=2, d=8, p=8, seed=5)
    o, dq, dk_acc, dv_acc, sels = oracle.chunk_recurrent_grads(
        c["q"], c["k_pool"], c["v_pool"], c["pt"], c["do"], chunk_len=32, page_size=8,
        top_k=10 ** 6)
    od, _, dqd, dkd, dvd = oracle.dense_causal_reference(
        c["q"], _flat(c["k_log"]), _flat(c["v_log"]), c["do"])
    np.testing.assert_allclose(o, od, atol=1e-12)
    np.testing.assert_allclose(dq, dqd, atol=1e-12)
    np.testing.assert_allclose(_flat(dk_acc), dkd, atol=1e-12)
    np.testing.assert_allclose(_flat(dv_acc), dvd, atol=1e-12)


def _ragged_case(t, hq=4, hkv=2, d=8, p=8, seed=3, tail=1e3):
    """A sequence of T tokens in ceil(T/P) shuffled pages; the rows of the last
    page past T hold large values that must never be read."""
    rng = np.random.default_rng(seed)
    n = -(-t // p)
    k_log = rng.normal(size=(n, hkv, p, d)) + 0.5 * rng.normal(size=(n, hkv, 1, d))
    v_log = rng.normal(size=(n, hkv, p, d))
    if t % p:
        k_log[-1, :, t % p:] = tail * rng.normal(size=(hkv, p - t % p, d))
        v_log[-1, :, t % p:] = tail * rng.normal(size=(hkv, p - t % p, d))
    pt = rng.permutation(n)
    k_pool = np.empty_like(k_log); v_pool = np.empty_like(v_log)
    k_pool[pt] = k_log; v_pool[pt] = v_log
    return dict(q=rng.normal(size=(t, hq, d)), do=rng.normal(size=(t, hq, d)), k_log=k_log,
                v_log=v_log, k_pool=k_pool, v_pool=v_pool, pt=pt, n=n, p=p, t=t)


@pytest.mark.parametrize("t,chunk_len", [(123, 32), (120, 32), (101, 48), (5, 16)])
def test_cross_chunk_ragged_sequence_equals_single_pass(t, chunk_len):
    # a sequence that is not whole chunks (and, but for t = 120, not whole
    # pages): the shorter last chunk and its partial page give the dense causal
    # gradient over the T tokens; the rows past T get no gradient
    c = _ragged_case(t)
    o, dq, dk_acc, dv_acc, _ = oracle.chunk_recurrent_grads(
        c["q"], c["k_pool"], c["v_pool"], c["pt"], c["do"], chunk_len=chunk_len, page_size=8,
        top_k=10 ** 6)
    kf, vf = _flat(c["k_log"])[:t], _flat(c["v_log"])[:t]
    od, _, dqd, dkd, dvd = oracle.dense_causal_reference(c["q"], kf, vf, c["do"])
    np.testing.assert_allclose(o, od, atol=1e-12)
    np.testing.assert_allclose(dq, dqd, atol=1e-12)
    np.testing.assert_allclose(_flat(dk_acc)[:t], dkd, atol=1e-12)
    np.testing.assert_allclose(_flat(dv_acc)[:t], dvd, atol=1e-12)
    assert np.all(_flat(dk_acc)[t:] == 0) and np.all(_flat(dv_acc)[t:] == 0)


def test_no_selected_pages_is_chunk_local_causal():
    c = _rng_case(t=96, hq=4, hkv=2, d=8, p=8, seed=9)
    t0 = 56
    sel = np.zeros((2, 0), np.int32)
    qc, doc = c["q"][t0:], c["do"][t0:]
    o, lse = oracle.attn_fwd(qc, c["k_pool"], c["v_pool"], c["pt"], sel, t0, c["p"])
    dq, dk_acc, dv_acc = oracle.attn_bwd(qc, c["k_pool"], c["v_pool"], c["pt"], sel, t0, c["p"],
                                         o, lse, doc)
    kf, vf = _flat(c["k_log"])[t0:], _flat(c["v_log"])[t0:]
    od, lsed, dqd, dkd, dvd = oracle.dense_causal_reference(qc, kf, vf, doc)
    np.testing.assert_allclose(o, od, atol=1e-12)
    np.testing.assert_allclose(lse, lsed, atol=1e-12)
    np.testing.assert_allclose(dq, dqd, atol=1e-12)
    np.testing.assert_allclose(_flat(dk_acc)[t0:], dkd, atol=1e-12)
    assert np.all(_flat(dk_acc)[:t0] == 0)


def test_first_query_sees_selected_pages_and_itself():
    c = _rng_case(t=96, hq=4, hkv=2, d=8, p=8, seed=11)
    t0 = 64
    sel = np.array([[2], [5]], np.int32)
    qc = c["q"][t0:t0 + 8]
    o, lse = oracle.attn_fwd(qc, c["k_pool"], c["v_pool"], c["pt"], sel, t0, c["p"])
    h, g = 1, 0
    keys = np.concatenate([c["k_log"][2, g], c["k_log"][t0 // 8, g, :1]])
    vals = np.concatenate([c["v_log"][2, g], c["v_log"][t0 // 8, g, :1]])
    s = keys @ qc[0, h] / math.sqrt(8)
    w = np.exp(s - s.max()); w /= w.sum()
    np.testing.assert_allclose(o[0, h], w @ vals, atol=1e-12)


# ---------------------------------------------------------------------------
# representative vectors, scores, Top-K
# ---------------------------------------------------------------------------
def test_page_reps_closed_forms():
    hkv, p, d, n = 2, 4, 3, 5
    pool = np.zeros((n, hkv, p, d))
    for s in range(n):
        pool[s] = s + 10 * np.arange(hkv)[:, None, None]   # constant page per head
    pt = np.array([3, 0, 4, 1, 2])
    reps = oracle.page_reps(pool, pt)
    for l in range(n):
        for g in range(hkv):
            np.testing.assert_array_equal(reps[l, g], pt[l] + 10 * g)
    rng = np.random.default_rng(0)
    one = rng.normal(size=(n, hkv, 1, d))
    np.testing.assert_array_equal(oracle.page_reps(one, np.arange(n)), one[:, :, 0])
    part = oracle.page_reps(pool, pt, first_page=2, n_pages=2)
    np.testing.assert_array_equal(part, reps[2:4])


def test_page_reps_partial_last_page():
    # the page cut by n_tokens: the mean of its written rows only; whatever the
    # rows after them hold does not matter
    hkv, p, d, n = 2, 8, 3, 4
    rng = np.random.default_rng(4)
    pool = rng.normal(size=(n, hkv, p, d)) * 1e3
    pt = np.array([2, 0, 3, 1])
    for l in range(n):
        pool[pt[l]] = l + 10 * np.arange(hkv)[:, None, None]
    pool[pt[3], :, 5:] = rng.normal(size=(hkv, p - 5, d)) * 1e3
    full = oracle.page_reps(pool, pt, 0, 3)
    reps = oracle.page_reps(pool, pt, 0, 4, n_tokens=3 * p + 5)
    np.testing.assert_array_equal(reps[:3], full)
    for g in range(hkv):
        np.testing.assert_array_equal(reps[3, g], 3 + 10 * g)
    # one written row: the representative is that key
    one = oracle.page_reps(pool, pt, 3, 1, n_tokens=3 * p + 1)
    np.testing.assert_array_equal(one[0], pool[pt[3], :, 0])
    # whole pages: n_tokens changes nothing; a page with no token is refused
    np.testing.assert_array_equal(oracle.page_reps(pool, pt, n_tokens=4 * p),
                                  oracle.page_reps(pool, pt))
    with pytest.raises(ValueError):
        oracle.page_reps(pool, pt, 0, 4, n_tokens=3 * p)


def test_score_is_mean_pair_logit_brute_force():
    c = _rng_case(t=96, hq=6, hkv=2, d=8, p=8, seed=13)
    t0, clen = 64, 32
    qc = c["q"][t0:]
    qbar = oracle.query_summary(qc, c["hkv"])
    reps = oracle.page_reps(c["k_pool"], c["pt"])
    grp = 3
    for g in range(2):
        for l in range(t0 // 8):
            pairs = [qc[t, h] @ c["k_log"][l, g, j] for t in range(clen)
                     for h in range(g * grp, g * grp + grp) for j in range(8)]
            brute = float(np.mean(pairs))
            assert abs(qbar[g] @ reps[l, g] - brute) < 1e-12
    s32 = oracle.page_scores(qbar, reps, t0 // 8)
    exact = np.einsum("gd,lgd->gl", qbar.astype(np.float32).astype(np.float64),
                      reps[:8].astype(np.float32).astype(np.float64))
    assert s32.dtype == np.float32
    assert np.all(np.abs(s32 - exact) <= np.abs(exact) * 2.0 ** -24 + 1e-45)


def _check_topk_order(scores, sel, k):
    n = scores.shape[0]
    assert len(sel) == min(k, n)
    assert np.all(np.diff(sel) > 0)
    chosen = set(sel.tolist())
    for a in chosen:
        for b in range(n):
            if b in chosen:
                continue
            assert scores[a] > scores[b] or (scores[a] == scores[b] and a < b)


@pytest.mark.parametrize("k", [0, 1, 5, 17, 40, 64])
def test_topk_invariants_and_brute_force(k):
    rng = np.random.default_rng(k)
    scores = rng.integers(-4, 5, size=(3, 40)).astype(np.float32)   # many exact ties
    sel = oracle.select_topk(scores, k)
    assert sel.shape == (3, min(k, 40))
    for g in range(3):
        _check_topk_order(scores[g], sel[g], k)
        brute = sorted(sorted(range(40), key=lambda l: (-float(scores[g, l]), l))[:k])
        assert sel[g].tolist() == brute


@pytest.mark.parametrize("k", [1, 5, 17, 29, 40])
def test_topk_signed_zero_and_nan(k):
    """+0 and -0 are the same score (the lower page wins) and a NaN score ranks
    below every number (NaN pages last, lower page first): brute force with a
    key that spells both rules out."""
    rng = np.random.default_rng(100 + k)
    vals = np.array([np.inf, 1.0, -1.0, -np.inf, 0.0, -0.0, np.nan], np.float32)
    scores = rng.choice(vals, size=(2, 40))
    for g in range(2):
        def key(l):
            v = float(scores[g, l])
            return (1, 0.0, l) if math.isnan(v) else (0, -v, l)   # -(-0.0) == -(0.0)
        brute = sorted(sorted(range(40), key=key)[:k])
        assert oracle.select_topk(scores, k)[g].tolist() == brute


def test_golden_tie_break():
    with open(os.path.join(GOLDEN, "tie_break_lowest_page.json")) as f:
        gj = json.load(f)
    inp, exp = gj["inputs"], gj["expected"]
    kl = np.array(inp["logical_keys"], np.float64)[:, None]      # [N, 1, P, D]
    pt = np.array(inp["page_table"])
    pool = np.empty_like(kl); pool[pt] = kl
    reps = oracle.page_reps(pool, pt)
    np.testing.assert_array_equal(reps[:, 0], np.array(exp["reps"], np.float64))
    q = np.array(inp["q"], np.float64)
    qbar = oracle.query_summary(q, 1)
    sc = oracle.page_scores(qbar, reps, inp["chunk_start"] // inp["page_size"])
    assert oracle.select_topk(sc, 2)[0].tolist() == exp["sel_top2"]
    assert oracle.select_topk(sc, 1)[0].tolist() == exp["sel_top1"]


def _ev(x):
    return float(eval(x, {"__builtins__": {}}, {"ln": math.log, "sqrt": math.sqrt}))


def test_golden_worked_example():
    with open(os.path.join(GOLDEN, "worked_example_select_attend.json")) as f:
        gj = json.load(f)
    inp, exp = gj["inputs"], gj["expected"]
    keys = np.array([[_ev(x) for x in r] for r in inp["keys"]])
    vals = np.array([[_ev(x) for x in r] for r in inp["values"]])
    pool_k = keys[:, None, None, :]
    pool_v = vals[:, None, None, :]
    pt = np.array(inp["page_table"])
    q = np.array([_ev(x) for x in inp["q"]])[None, None, :]
    do = np.array([_ev(x) for x in inp["do"]])[None, None, :]
    t0, p = inp["chunk_start"], inp["page_size"]
    reps = oracle.page_reps(pool_k, pt)
    sc = oracle.page_scores(oracle.query_summary(q, 1), reps, t0 // p)
    sel = oracle.select_topk(sc, inp["top_k"])
    assert sel[0].tolist() == exp["sel"]
    o, lse = oracle.attn_fwd(q, pool_k, pool_v, pt, sel, t0, p)
    np.testing.assert_allclose(o[0, 0], [_ev(x) for x in exp["o"]], atol=1e-14)
    assert abs(lse[0, 0] - _ev(exp["lse"])) < 1e-14
    dq, dk, dv = oracle.attn_bwd(q, pool_k, pool_v, pt, sel, t0, p, o, lse, do)
    np.testing.assert_allclose(dq[0, 0], [_ev(x) for x in exp["dq"]], atol=1e-14)
    np.testing.assert_allclose(dk[:, 0, 0], [[_ev(x) for x in r] for r in exp["dk"]], atol=1e-14)
    np.testing.assert_allclose(dv[:, 0, 0], [[_ev(x) for x in r] for r in exp["dv"]], atol=1e-14)


# ---------------------------------------------------------------------------
# fp8 (E4M3) storage of the K/V pools
# ---------------------------------------------------------------------------
def test_fp8_e4m3_decode_worked_values():
    # values worked out by hand from the format (bias 7, 3 mantissa bits)
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x3C: 1.5, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0x30: 0.5,
             0xB8: -1.0, 0xFE: -448.0, 0x81: -(2.0 ** -9)}
    got = oracle.fp8_e4m3_decode(np.array(list(cases), np.uint8))
    np.testing.assert_array_equal(got, np.array(list(cases.values())))
    assert np.isnan(oracle.fp8_e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    neg0 = oracle.fp8_e4m3_decode(np.array([0x80], np.uint8))
    assert neg0[0] == 0.0 and np.signbit(neg0[0])


def test_fp8_e4m3_decode_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.fp8_e4m3_decode(codes.numpy())
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    # the 254 finite values are distinct up to the sign of zero, and monotone
    pos = got[:127]
    assert np.all(np.diff(pos) > 0)
