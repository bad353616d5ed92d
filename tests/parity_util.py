"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding and compare with the oracle using the tolerances of the method's
evaluation (bf16: max-abs 2e-2 and relative L2 1e-2; fp32: max-abs 1e-4;
selection bit-exact except pairs whose fp32 score gap is below 1e-4)."""
import numpy as np
import torch

import oracle
from paged_sparse_attention_oomb_gb300 import oomb
from paged_sparse_attention_oomb_gb300.workloads import to_numpy64

BF16_ATOL, BF16_REL_L2 = 2e-2, 1e-2
FP32_ATOL = 1e-4
TIE_GAP = 1e-4


def compare(gpu, ref, dtype, what=""):
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - r)
    mx = float(err.max()) if err.size else 0.0
    if dtype == "fp32":
        assert mx <= FP32_ATOL, f"{what}: max-abs {mx:.3e} > {FP32_ATOL}"
        return mx, 0.0
    rl2 = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    assert mx <= BF16_ATOL, f"{what}: max-abs {mx:.3e} > {BF16_ATOL}"
    assert rl2 <= BF16_REL_L2, f"{what}: rel-L2 {rl2:.3e} > {BF16_REL_L2}"
    return mx, rl2


def check_selection(gpu_sel, ora_sel, ora_scores):
    """Bit-exact selection, except swaps between candidates whose oracle fp32
    scores differ by less than TIE_GAP.  Returns the number of flagged pairs."""
    flagged = 0
    gpu_sel = np.asarray(gpu_sel)
    ora_sel = np.asarray(ora_sel)
    assert gpu_sel.shape == ora_sel.shape
    for g in range(gpu_sel.shape[0]):
        assert np.all(np.diff(gpu_sel[g]) > 0), "selection must be ascending and unique"
        a = sorted(set(gpu_sel[g].tolist()) - set(ora_sel[g].tolist()))
        b = sorted(set(ora_sel[g].tolist()) - set(gpu_sel[g].tolist()))
        assert len(a) == len(b)
        sa = sorted(float(ora_scores[g][i]) for i in a)
        sb = sorted(float(ora_scores[g][i]) for i in b)
        for x, y in zip(sa, sb):
            assert abs(x - y) < TIE_GAP, f"head {g}: selection differs beyond a near-tie"
        flagged += len(a)
    return flagged


def oracle_reps_blocked(k_pool_t, page_table_t, block=512):
    """Oracle representatives of every page, page block by page block from a
    torch pool (so a multi-GB pool is never widened to float64 all at once)."""
    pt = page_table_t.cpu().long()
    k_host = k_pool_t.cpu()
    n = pt.numel()
    out = []
    for b0 in range(0, n, block):
        sub = k_host[pt[b0:b0 + block]].float().numpy()
        out.append(oracle.page_reps(sub, np.arange(sub.shape[0])))
    return np.concatenate(out, axis=0)


def oracle_selection(x, reps64, top_k):
    wl = x.wl
    qbar = oracle.query_summary(to_numpy64(x.q), wl.num_kv_heads)
    n_cand = wl.num_candidates
    scores = oracle.page_scores(qbar, reps64, n_cand)
    sel = oracle.select_topk(scores, top_k)
    return sel, scores


def gpu_kv(x, with_grads=True, grad_init=None):
    dk = dv = None
    if with_grads:
        if grad_init is None:
            dk = torch.zeros_like(x.k_pool)
            dv = torch.zeros_like(x.v_pool)
        else:
            dk, dv = grad_init[0].clone(), grad_init[1].clone()
    return oomb.PagedKV(x.k_pool, x.v_pool, x.page_table, dk, dv)


def gpu_reps(kv):
    n = kv.page_table.numel()
    _, hkv, _, d = kv.k.shape
    reps = torch.empty((n, hkv, d), dtype=torch.float32, device=kv.k.device)
    ws = oomb.workspace(oomb.OOMB_OP_PAGE_REPS, kv)
    oomb.oomb_page_reps(kv, 0, n, reps, ws)
    assert_status_ok(ws)
    return reps


def gpu_select(x, kv, reps, top_k):
    wl = x.wl
    n_sel = min(top_k, wl.num_candidates)
    sel = torch.full((wl.num_kv_heads, max(n_sel, 1)), -1, dtype=torch.int32, device=x.q.device)
    scores = torch.empty((wl.num_kv_heads, wl.num_pages), dtype=torch.float32, device=x.q.device)
    ws = oomb.workspace(oomb.OOMB_OP_SELECT_TOPK, kv, wl.num_q_heads, wl.chunk_len, top_k)
    oomb.oomb_select_topk(x.q, wl.start, reps, kv, top_k, sel, ws, scores=scores)
    assert_status_ok(ws)
    return sel[:, :n_sel], scores


def gpu_fwd(x, kv, sel_t, n_sel, with_lo=False):
    """O and LSE (and, with ``with_lo``, the bf16 rounding residual of O that
    the backward takes for its Delta)."""
    wl = x.wl
    o = torch.empty_like(x.q)
    o_lo = oomb.o_residual_like(o)
    lse = torch.empty((wl.num_q_heads, wl.chunk_len), dtype=torch.float32, device=x.q.device)
    ws = oomb.workspace(oomb.OOMB_OP_ATTN_FWD, kv, wl.num_q_heads, wl.chunk_len)
    oomb.oomb_sparse_attn_fwd(x.q, kv, sel_t, n_sel, wl.start, o, lse, ws, o_lo=o_lo)
    assert_status_ok(ws)
    return (o, lse, o_lo) if with_lo else (o, lse)


def gpu_bwd(x, kv, sel_t, n_sel, o, lse, dout=None, o_lo=None):
    wl = x.wl
    dq = torch.empty_like(x.q)
    ws = oomb.workspace(oomb.OOMB_OP_ATTN_BWD, kv, wl.num_q_heads, wl.chunk_len)
    oomb.oomb_sparse_attn_bwd(x.q, o, x.do if dout is None else dout, lse, kv, sel_t, n_sel,
                              wl.start, dq, ws, o_lo=o_lo)
    assert_status_ok(ws)
    return dq


def assert_status_ok(ws):
    code, where, blk = oomb.oomb_device_status(ws)
    assert code == oomb.OOMB_OK, f"device status {oomb.oomb_status_string(code)} where={where} block={blk}"


def sel_tensor(sel_np, device):
    n = max(sel_np.shape[1], 1)
    t = torch.zeros((sel_np.shape[0], n), dtype=torch.int32, device=device)
    if sel_np.shape[1]:
        t[:, :sel_np.shape[1]] = torch.as_tensor(sel_np, dtype=torch.int32)
    return t
