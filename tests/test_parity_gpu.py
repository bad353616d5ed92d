"""CUDA path vs the CPU oracle, through the C ABI (GB300 only).

Small cases are compared element by element (several tiles, ragged tails,
every page size, K = 0 / some / all, first chunk, shuffled page tables).  The
five named workloads run at full size: selection in full, outputs on sampled
rows and gradients on sampled pages, each computed exactly by the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_sparse_attention_oomb_gb300 import oomb
from paged_sparse_attention_oomb_gb300.workloads import WORKLOADS, Workload, make_inputs, to_numpy64

from parity_util import (check_selection, compare, gpu_bwd, gpu_fwd, gpu_kv, gpu_reps,
                         gpu_select, oracle_reps_blocked, oracle_selection, sel_tensor)

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oomb.load()
    oomb.oomb_set_wait_limit_ns(0)


def W(name, dtype, hq, hkv, ctx, p, c, k, shuffled=True, start=-1):
    return Workload(name, dtype, hq, hkv, 128 if dtype == "bf16" else 64, ctx, p, c, k, shuffled,
                    start)


SMALL = [
    W("bf16_p64_ragged_c576_k13", "bf16", 4, 2, 4096, 64, 576, 13),
    W("bf16_p128_g8_c384_k5", "bf16", 8, 1, 2048, 128, 384, 5, shuffled=False),
    W("bf16_p16_g1_c208_k37", "bf16", 2, 2, 1024, 16, 208, 37),
    W("bf16_p32_k0", "bf16", 4, 4, 1536, 32, 256, 0),
    W("bf16_first_chunk", "bf16", 4, 2, 2048, 64, 1024, 8, start=0),
    W("bf16_dense_all", "bf16", 4, 2, 2048, 64, 512, 1 << 20),
    W("bf16_mid_chunk_k20", "bf16", 14, 2, 4096, 64, 640, 20, start=1920),
    W("fp32_ragged_c176_k7", "fp32", 4, 2, 512, 16, 176, 7),
    W("fp32_p32_k3", "fp32", 2, 1, 1024, 32, 320, 3),
]


def _run_small(wl, seed=0):
    x = make_inputs(wl, seed=seed, device=DEV)
    kv = gpu_kv(x)
    q, kp, vp, do, pt = (to_numpy64(x.q), to_numpy64(x.k_pool), to_numpy64(x.v_pool),
                         to_numpy64(x.do), to_numpy64(x.page_table))
    # step 1: representative vectors
    reps = gpu_reps(kv)
    reps64 = oracle.page_reps(kp, pt)
    compare(reps.cpu().numpy(), reps64, "fp32", f"{wl.name} reps")
    # step 2: selection (bit-exact up to flagged near-ties)
    sel_g, scores_g = gpu_select(x, kv, reps, wl.top_k)
    sel_o, scores_o = oracle_selection(x, reps64, wl.top_k)
    check_selection(sel_g.cpu().numpy(), sel_o, scores_o)
    nc = wl.num_candidates
    if nc:
        np.testing.assert_allclose(scores_g[:, :nc].cpu().numpy(), scores_o, rtol=1e-5, atol=1e-6)
    assert torch.all(torch.isinf(scores_g[:, nc:]))
    # steps 3-4 on the oracle's selection (its output may feed the GPU, never the reverse)
    n_sel = sel_o.shape[1]
    st = sel_tensor(sel_o, DEV)
    o_g, lse_g, o_lo = gpu_fwd(x, kv, st, n_sel, with_lo=True)
    dq_g = gpu_bwd(x, kv, st, n_sel, o_g, lse_g, o_lo=o_lo)
    o_o, lse_o = oracle.attn_fwd(q, kp, vp, pt, sel_o, wl.start, wl.page_size)
    dq_o, dk_o, dv_o = oracle.attn_bwd(q, kp, vp, pt, sel_o, wl.start, wl.page_size, o_o, lse_o, do)
    dt = wl.dtype
    compare(o_g.float().cpu().numpy(), o_o, dt, f"{wl.name} O")
    compare(lse_g.cpu().numpy(), lse_o, "fp32" if dt == "fp32" else "bf16", f"{wl.name} LSE")
    np.testing.assert_allclose(lse_g.cpu().numpy(), lse_o, atol=2e-3 if dt == "bf16" else 1e-4)
    compare(dq_g.float().cpu().numpy(), dq_o, dt, f"{wl.name} dQ")
    ptl = x.page_table.long().cpu()
    dk_g = to_numpy64(kv.dk)[ptl.numpy()]           # logical page order
    dv_g = to_numpy64(kv.dv)[ptl.numpy()]
    compare(dk_g, dk_o, dt, f"{wl.name} dK")
    compare(dv_g, dv_o, dt, f"{wl.name} dV")
    # untouched pages stay exactly zero
    untouched = np.all(dk_o == 0, axis=(2, 3))
    assert np.all(dk_g[untouched] == 0) and np.all(dv_g[untouched] == 0)
    return x, kv


@pytest.mark.parametrize("wl", SMALL, ids=[w.name for w in SMALL])
def test_small_parity(wl):
    _run_small(wl)


def test_tiny_fp32_workload_k8_and_all():
    base = WORKLOADS["tiny_fp32_ctx1k"]
    _run_small(base)
    _run_small(base.with_(name="tiny_fp32_all", top_k=1 << 20))


def test_bwd_accumulates_in_place():
    wl = W("acc", "bf16", 4, 2, 2048, 64, 256, 6)
    x = make_inputs(wl, seed=3, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(11)
    init_k = torch.randn(x.k_pool.shape, generator=g, device=DEV).to(torch.bfloat16)
    init_v = torch.randn(x.v_pool.shape, generator=g, device=DEV).to(torch.bfloat16)
    kv = gpu_kv(x, grad_init=(init_k, init_v))
    q, kp, vp, do, pt = (to_numpy64(x.q), to_numpy64(x.k_pool), to_numpy64(x.v_pool),
                         to_numpy64(x.do), to_numpy64(x.page_table))
    sel_o, _ = oracle_selection(x, oracle.page_reps(kp, pt), wl.top_k)
    st = sel_tensor(sel_o, DEV)
    o_g, lse_g, o_lo = gpu_fwd(x, kv, st, sel_o.shape[1], with_lo=True)
    gpu_bwd(x, kv, st, sel_o.shape[1], o_g, lse_g, o_lo=o_lo)
    o_o, lse_o = oracle.attn_fwd(q, kp, vp, pt, sel_o, wl.start, wl.page_size)
    dk_acc = to_numpy64(init_k)[pt]
    dv_acc = to_numpy64(init_v)[pt]
    _, dk_o, dv_o = oracle.attn_bwd(q, kp, vp, pt, sel_o, wl.start, wl.page_size, o_o, lse_o, do,
                                    dk_acc=dk_acc, dv_acc=dv_acc)
    compare(to_numpy64(kv.dk)[pt], dk_o, "bf16", "dK += ")
    compare(to_numpy64(kv.dv)[pt], dv_o, "bf16", "dV += ")


def test_cross_chunk_accumulation():
    """Chunks processed forward in order, backward in reverse, dK/dV accumulated
    across chunks in the same paged buffers (chunk-recurrent pass)."""
    base = W("xchunk", "bf16", 4, 2, 2048, 64, 512, 1 << 20)
    x = make_inputs(base, seed=5, device=DEV)
    kv = gpu_kv(x)
    q_full = torch.randn((2048, 4, 128), device=DEV, generator=torch.Generator(device=DEV).manual_seed(1)).to(torch.bfloat16)
    do_full = torch.randn((2048, 4, 128), device=DEV, generator=torch.Generator(device=DEV).manual_seed(2)).to(torch.bfloat16)
    reps = gpu_reps(kv)
    outs = []
    for c in range(4):
        wl = base.with_(chunk_start=c * 512)
        xc = type(x)(wl, q_full[c * 512:(c + 1) * 512].contiguous(), x.k_pool, x.v_pool,
                     do_full[c * 512:(c + 1) * 512].contiguous(), x.page_table)
        sel, _ = gpu_select(xc, kv, reps, wl.top_k)
        o, lse, o_lo = gpu_fwd(xc, kv, sel.contiguous(), sel.shape[1], with_lo=True)
        outs.append((xc, sel.contiguous(), o, lse, o_lo))
    for xc, sel, o, lse, o_lo in reversed(outs):
        gpu_bwd(xc, kv, sel if sel.numel() else sel_tensor(np.zeros((2, 0), np.int32), DEV),
                sel.shape[1], o, lse, o_lo=o_lo)
    kp, vp, pt = to_numpy64(x.k_pool), to_numpy64(x.v_pool), to_numpy64(x.page_table)
    o_o, dq_o, dk_o, dv_o, _ = oracle.chunk_recurrent_grads(
        to_numpy64(q_full), kp, vp, pt, to_numpy64(do_full), 512, 64, 1 << 20)
    compare(to_numpy64(kv.dk)[pt], dk_o, "bf16", "cross-chunk dK")
    compare(to_numpy64(kv.dv)[pt], dv_o, "bf16", "cross-chunk dV")


@pytest.mark.parametrize("top_k", [3, 1 << 20])
def test_chunk_recurrent_pass(top_k):
    """Forward over chunks in order, backward in reverse, through the driver."""
    wl = W("crp", "bf16", 4, 2, 2048, 64, 512, top_k)
    x = make_inputs(wl, seed=8, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(3)
    q_full = torch.randn((2048, 4, 128), generator=g, device=DEV).to(torch.bfloat16)
    do_full = torch.randn((2048, 4, 128), generator=g, device=DEV).to(torch.bfloat16)
    kv = gpu_kv(x)
    o_g, dq_g, sels = oomb.chunk_recurrent_pass(q_full, do_full, kv, 512, top_k)
    kp, vp, pt = to_numpy64(x.k_pool), to_numpy64(x.v_pool), to_numpy64(x.page_table)
    o_o, dq_o, dk_o, dv_o, sels_o = oracle.chunk_recurrent_grads(
        to_numpy64(q_full), kp, vp, pt, to_numpy64(do_full), 512, 64, top_k)
    for sg, so in zip(sels, sels_o):
        assert sg.cpu().numpy().tolist() == so.tolist()
    compare(o_g.float().cpu().numpy(), o_o, "bf16", "chunk-recurrent O")
    compare(dq_g.float().cpu().numpy(), dq_o, "bf16", "chunk-recurrent dQ")
    compare(to_numpy64(kv.dk)[pt], dk_o, "bf16", "chunk-recurrent dK")
    compare(to_numpy64(kv.dv)[pt], dv_o, "bf16", "chunk-recurrent dV")


@pytest.mark.parametrize("seed,qseed", [(9, 4), (8, 3), (12, 1)])
def test_chunk_recurrent_pass_concentrated_rows(seed, qseed):
    """The first rows of a sequence see a handful of keys, so their attention
    often sits almost wholly on one key.  There dP of that key nearly equals
    Delta = dO . O, and dS = P (dP - Delta) keeps only their difference: an
    O rounded to bf16 before Delta is taken moved dQ by up to 0.0243 on the
    (9, 4) pass.  With the forward's rounding residual of O the backward
    takes Delta from the fp32 O, and dQ stays inside the bf16 bound."""
    wl = W("crp_conc", "bf16", 4, 2, 2048, 64, 512, 3)
    x = make_inputs(wl, seed=seed, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(qseed)
    q_full = torch.randn((2048, 4, 128), generator=g, device=DEV).to(torch.bfloat16)
    do_full = torch.randn((2048, 4, 128), generator=g, device=DEV).to(torch.bfloat16)
    kv = gpu_kv(x)
    o_g, dq_g, _ = oomb.chunk_recurrent_pass(q_full, do_full, kv, 512, 3)
    kp, vp, pt = to_numpy64(x.k_pool), to_numpy64(x.v_pool), to_numpy64(x.page_table)
    o_o, dq_o, dk_o, dv_o, _ = oracle.chunk_recurrent_grads(
        to_numpy64(q_full), kp, vp, pt, to_numpy64(do_full), 512, 64, 3)
    mx, _ = compare(dq_g.float().cpu().numpy(), dq_o, "bf16", "concentrated rows dQ")
    print(f"seed {seed}/{qseed}: dQ max-abs {mx:.4f}")
    compare(o_g.float().cpu().numpy(), o_o, "bf16", "concentrated rows O")
    compare(to_numpy64(kv.dk)[pt], dk_o, "bf16", "concentrated rows dK")
    compare(to_numpy64(kv.dv)[pt], dv_o, "bf16", "concentrated rows dV")


def test_o_residual_is_the_rounding_remainder():
    """o_lo is what rounding the fp32 output to bf16 dropped: at most half a
    bf16 unit of o in the last place, and o + o_lo is nearer the oracle's O
    than o alone."""
    wl = W("olo", "bf16", 8, 2, 4096, 64, 512, 9)
    x = make_inputs(wl, seed=13, device=DEV)
    kv = gpu_kv(x, with_grads=False)
    q, kp, vp, pt = (to_numpy64(x.q), to_numpy64(x.k_pool), to_numpy64(x.v_pool),
                     to_numpy64(x.page_table))
    sel_o, _ = oracle_selection(x, oracle.page_reps(kp, pt), wl.top_k)
    st = sel_tensor(sel_o, DEV)
    o_g, _, o_lo = gpu_fwd(x, kv, st, sel_o.shape[1], with_lo=True)
    o = o_g.float().cpu().numpy().astype(np.float64)
    lo = o_lo.float().cpu().numpy().astype(np.float64)
    # half a unit in the last place of each bf16 value of o (8 significant bits)
    half_ulp = np.where(o != 0, 2.0 ** (np.floor(np.log2(np.abs(np.where(o != 0, o, 1.0)))) - 8),
                        2.0 ** -134)
    assert np.all(np.abs(lo) <= half_ulp)
    o_o, _ = oracle.attn_fwd(q, kp, vp, pt, sel_o, wl.start, wl.page_size)
    err_hi = np.linalg.norm(o - o_o)
    err_hilo = np.linalg.norm(o + lo - o_o)
    assert err_hilo < err_hi, (err_hilo, err_hi)


OWN_REPS = [
    W("bf16_p64_ragged_c576_k13", "bf16", 4, 2, 4096, 64, 576, 13),   # 9 own pages: last tile 1 page
    W("bf16_p128_c384_k5", "bf16", 8, 1, 2048, 128, 384, 5),
    W("bf16_p16_c208_k37", "bf16", 2, 2, 1024, 16, 208, 37),
    W("bf16_first_chunk", "bf16", 4, 2, 2048, 64, 1024, 8, start=0),
    W("fp32_ragged_c176_k7", "fp32", 4, 2, 512, 16, 176, 7),
]


@pytest.mark.parametrize("wl", OWN_REPS, ids=[w.name for w in OWN_REPS])
def test_fwd_own_reps(wl):
    """The forward with the chunk's own representatives fused in: O and LSE
    bit-identical to the plain forward, the own pages' representatives
    bit-identical to the representatives pass (and within fp32 of the
    oracle), every other row untouched."""
    x = make_inputs(wl, seed=4, device=DEV)
    kv = gpu_kv(x)
    reps = gpu_reps(kv)
    sel_g, _ = gpu_select(x, kv, reps, wl.top_k)
    n_sel = min(wl.top_k, wl.num_candidates)
    st = sel_g[:, :max(n_sel, 1)].contiguous()
    o_ref, lse_ref = gpu_fwd(x, kv, st, n_sel)
    o = torch.empty_like(x.q)
    lse = torch.empty_like(lse_ref)
    fused = torch.full_like(reps, float("nan"))
    ws = oomb.workspace(oomb.OOMB_OP_ATTN_FWD, kv, wl.num_q_heads, wl.chunk_len)
    oomb.oomb_sparse_attn_fwd_own_reps(x.q, kv, st, n_sel, wl.start, o, lse, fused, ws)
    code, where, blk = oomb.oomb_device_status(ws)
    assert code == oomb.OOMB_OK, (code, where, blk)
    assert torch.equal(o.view(torch.int16) if o.dtype == torch.bfloat16 else o,
                       o_ref.view(torch.int16) if o_ref.dtype == torch.bfloat16 else o_ref)
    assert torch.equal(lse, lse_ref)
    p0 = wl.start // wl.page_size
    p1 = (wl.start + wl.chunk_len) // wl.page_size
    assert torch.equal(fused[p0:p1], reps[p0:p1])
    assert torch.isnan(fused[:p0]).all() and torch.isnan(fused[p1:]).all()
    reps64 = oracle.page_reps(to_numpy64(x.k_pool), to_numpy64(x.page_table))
    compare(fused[p0:p1].cpu().numpy(), reps64[p0:p1], "fp32", f"{wl.name} own reps")


# Chunks that end inside a page (the last chunk of a sequence that is not whole
# pages): ragged query tiles, a partial last own page, ragged selection tiles.
PARTIAL = [
    W("bf16_p64_c453_k13", "bf16", 4, 2, 4096, 64, 453, 13, start=3584),     # last page: 5 rows
    W("bf16_p128_g8_c300_k5", "bf16", 8, 1, 2048, 128, 300, 5, start=1024),  # 44 rows
    W("bf16_p16_g1_c77_k37", "bf16", 2, 2, 1024, 16, 77, 37, start=512),     # 13 rows
    W("bf16_single_query", "bf16", 4, 2, 2048, 64, 1, 4, start=1024),
    W("bf16_first_chunk_c45", "bf16", 4, 2, 1024, 32, 45, 8, start=0),
    W("fp32_p16_c99_k7", "fp32", 4, 2, 512, 16, 99, 7, start=256),          # 3 rows
    W("fp32_p32_c45_k0", "fp32", 2, 1, 1024, 32, 45, 0, start=0),
]


def _spoil_tail(x, tokens, scale=30.0):
    """Fill the rows of the partial page past ``tokens`` with large values: a
    kernel that reads them as keys or values would show it."""
    wl = x.wl
    p = wl.page_size
    if tokens % p == 0:
        return
    slot = int(x.page_table[tokens // p])
    g = torch.Generator(device=DEV)
    g.manual_seed(99)
    for pool in (x.k_pool, x.v_pool):
        tail = pool[slot, :, tokens % p:]
        tail.copy_((scale * torch.randn(tail.shape, generator=g, device=DEV)).to(pool.dtype))


@pytest.mark.parametrize("wl", PARTIAL, ids=[w.name for w in PARTIAL])
def test_partial_last_page(wl):
    """Forward and backward of a chunk whose last own page is partial, against
    the oracle element by element, starting from nonzero gradients: the rows
    past the chunk are never attended and keep their dK/dV bit for bit; the
    fused forward represents the partial page by the mean of its written keys."""
    x = make_inputs(wl, seed=6, device=DEV)
    end = wl.start + wl.chunk_len
    _spoil_tail(x, end)
    g = torch.Generator(device=DEV)
    g.manual_seed(12)
    init = [torch.randn(x.k_pool.shape, generator=g, device=DEV).to(x.k_pool.dtype)
            for _ in range(2)]
    kv = gpu_kv(x, grad_init=init)
    q, kp, vp, do, pt = (to_numpy64(x.q), to_numpy64(x.k_pool), to_numpy64(x.v_pool),
                         to_numpy64(x.do), to_numpy64(x.page_table))
    p = wl.page_size
    p0, p1 = wl.start // p, -(-end // p)
    reps = gpu_reps(kv)
    reps64 = oracle.page_reps(kp, pt, 0, p1, n_tokens=end)
    sel_g, _ = gpu_select(x, kv, reps, wl.top_k)
    sel_o, scores_o = oracle_selection(x, reps64, wl.top_k)
    check_selection(sel_g.cpu().numpy(), sel_o, scores_o)
    n_sel = sel_o.shape[1]
    st = sel_tensor(sel_o, DEV)
    # forward with the own representatives fused in
    o_g = torch.empty_like(x.q)
    lse_g = torch.empty((wl.num_q_heads, wl.chunk_len), dtype=torch.float32, device=DEV)
    fused = torch.full_like(reps, float("nan"))
    o_lo = oomb.o_residual_like(o_g)
    ws = oomb.workspace(oomb.OOMB_OP_ATTN_FWD, kv, wl.num_q_heads, wl.chunk_len)
    oomb.oomb_sparse_attn_fwd_own_reps(x.q, kv, st, n_sel, wl.start, o_g, lse_g, fused, ws,
                                       o_lo=o_lo)
    code, where, blk = oomb.oomb_device_status(ws)
    assert code == oomb.OOMB_OK, (code, where, blk)
    full_end = p1 if end % p == 0 else p1 - 1
    assert torch.equal(fused[p0:full_end], reps[p0:full_end])
    compare(fused[p0:p1].cpu().numpy(), reps64[p0:p1], "fp32", f"{wl.name} own reps")
    assert torch.isnan(fused[:p0]).all() and torch.isnan(fused[p1:]).all()
    dq_g = gpu_bwd(x, kv, st, n_sel, o_g, lse_g, o_lo=o_lo)
    o_o, lse_o = oracle.attn_fwd(q, kp, vp, pt, sel_o, wl.start, p)
    dk_o, dv_o = to_numpy64(init[0])[pt], to_numpy64(init[1])[pt]
    dq_o, dk_o, dv_o = oracle.attn_bwd(q, kp, vp, pt, sel_o, wl.start, p, o_o, lse_o, do,
                                       dk_acc=dk_o, dv_acc=dv_o)
    dt = wl.dtype
    compare(o_g.float().cpu().numpy(), o_o, dt, f"{wl.name} O")
    np.testing.assert_allclose(lse_g.cpu().numpy(), lse_o, atol=2e-3 if dt == "bf16" else 1e-4)
    compare(dq_g.float().cpu().numpy(), dq_o, dt, f"{wl.name} dQ")
    dk_g, dv_g = to_numpy64(kv.dk)[pt], to_numpy64(kv.dv)[pt]
    compare(dk_g, dk_o, dt, f"{wl.name} dK")
    compare(dv_g, dv_o, dt, f"{wl.name} dV")
    # the rows past the chunk and the pages after it: exactly the initial values
    k0, v0 = to_numpy64(init[0])[pt], to_numpy64(init[1])[pt]
    if end % p:
        assert np.array_equal(dk_g[end // p, :, end % p:], k0[end // p, :, end % p:])
        assert np.array_equal(dv_g[end // p, :, end % p:], v0[end // p, :, end % p:])
    assert np.array_equal(dk_g[p1:], k0[p1:]) and np.array_equal(dv_g[p1:], v0[p1:])


@pytest.mark.parametrize("what", ["k_nan", "v_inf", "finite"])
def test_partial_last_page_non_finite_rows_are_flagged(what):
    """A NaN or inf in an unused row of the partial last page (where a
    torch.empty pool leaves garbage) is recorded as OOMB_ERR_NONFINITE by the
    forward and the backward; finite garbage there is not an error."""
    wl = PARTIAL[0]
    x = make_inputs(wl, seed=6, device=DEV)
    end = wl.start + wl.chunk_len
    p = wl.page_size
    slot = int(x.page_table[end // p])
    _spoil_tail(x, end)
    row = end % p + (p - end % p) // 2                  # a row past the chunk's end
    if what == "k_nan":
        x.k_pool[slot, 1, row, 77] = float("nan")
    elif what == "v_inf":
        x.v_pool[slot, 0, p - 1, 0] = float("-inf")
    kv = gpu_kv(x)
    sel = sel_tensor(np.tile(np.arange(wl.n_sel, dtype=np.int32), (wl.num_kv_heads, 1)), DEV)
    want = oomb.OOMB_OK if what == "finite" else oomb.OOMB_ERR_NONFINITE
    o = torch.empty_like(x.q)
    lse = torch.empty((wl.num_q_heads, wl.chunk_len), dtype=torch.float32, device=DEV)
    ws = oomb.workspace(oomb.OOMB_OP_ATTN_FWD, kv, wl.num_q_heads, wl.chunk_len)
    oomb.oomb_sparse_attn_fwd(x.q, kv, sel, wl.n_sel, wl.start, o, lse, ws)
    assert oomb.oomb_device_status(ws)[0] == want
    dq = torch.empty_like(x.q)
    ws = oomb.workspace(oomb.OOMB_OP_ATTN_BWD, kv, wl.num_q_heads, wl.chunk_len)
    oomb.oomb_sparse_attn_bwd(x.q, o, x.do, lse, kv, sel, wl.n_sel, wl.start, dq, ws)
    assert oomb.oomb_device_status(ws)[0] == want
    if what == "finite":
        assert torch.isfinite(o).all() and torch.isfinite(dq).all()


@pytest.mark.parametrize("top_k", [3, 1 << 20])
def test_chunk_recurrent_pass_ragged_sequence(top_k):
    """The sequence of test_chunk_recurrent_pass cut 19 tokens before its end:
    2029 tokens in chunks of 512, the last chunk has 493 rows and ends 45 rows
    into its last page, whose unwritten rows hold large values.  Selections,
    O, dQ and the paged dK/dV against the oracle's chunk-recurrent pass; the
    rows past the sequence keep zero gradient."""
    t = 2029
    wl = W("crp_ragged", "bf16", 4, 2, 2048, 64, 512, top_k)
    x = make_inputs(wl, seed=8, device=DEV)
    _spoil_tail(x, t)
    g = torch.Generator(device=DEV)
    g.manual_seed(3)
    q_full = torch.randn((2048, 4, 128), generator=g, device=DEV).to(torch.bfloat16)[:t].contiguous()
    do_full = torch.randn((2048, 4, 128), generator=g, device=DEV).to(torch.bfloat16)[:t].contiguous()
    kv = gpu_kv(x)
    o_g, dq_g, sels = oomb.chunk_recurrent_pass(q_full, do_full, kv, 512, top_k)
    kp, vp, pt = to_numpy64(x.k_pool), to_numpy64(x.v_pool), to_numpy64(x.page_table)
    o_o, dq_o, dk_o, dv_o, sels_o = oracle.chunk_recurrent_grads(
        to_numpy64(q_full), kp, vp, pt, to_numpy64(do_full), 512, 64, top_k)
    assert len(sels) == len(sels_o) == 4
    for sg, so in zip(sels, sels_o):
        assert sg.cpu().numpy().tolist() == so.tolist()
    compare(o_g.float().cpu().numpy(), o_o, "bf16", "ragged chunk-recurrent O")
    compare(dq_g.float().cpu().numpy(), dq_o, "bf16", "ragged chunk-recurrent dQ")
    dk_g, dv_g = to_numpy64(kv.dk)[pt], to_numpy64(kv.dv)[pt]
    compare(dk_g, dk_o, "bf16", "ragged chunk-recurrent dK")
    compare(dv_g, dv_o, "bf16", "ragged chunk-recurrent dV")
    assert np.all(dk_g[31, :, 45:] == 0) and np.all(dv_g[31, :, 45:] == 0)


def _offload_case(seed):
    wl = W("offl", "bf16", 4, 2, 4096, 64, 512, 3)     # 64 pages; a chunk needs <= 3 * 2 + 8 pages
    x = make_inputs(wl, seed=seed, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(seed + 1)
    q_full = torch.randn((4096, 4, 128), generator=g, device=DEV).to(torch.bfloat16)
    do_full = torch.randn((4096, 4, 128), generator=g, device=DEV).to(torch.bfloat16)
    dk0 = torch.randn(x.k_pool.shape, generator=g, device=DEV).to(torch.bfloat16)
    dv0 = torch.randn(x.k_pool.shape, generator=g, device=DEV).to(torch.bfloat16)
    return wl, x, q_full, do_full, dk0, dv0


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


@pytest.mark.parametrize("prefetch,staging", [(False, 256 << 20), (True, 256 << 20),
                                              (True, 0), (True, 5 * 64 * 128 * 2)],
                         ids=["serial", "prefetch", "zero_copy", "staging_5_tiles"])
def test_offload_chunk_pass_matches_resident(prefetch, staging):
    """Pools in pinned host memory behind a device cache that must reuse slots
    (28 slots for 64 pages): the chunk-recurrent pass gives bit-identical O,
    selections and host dK/dV to the same pass on resident pools, starting
    from nonzero gradients (in-place accumulation through the cache), and the
    same dQ up to the order of its fp32 atomic sums."""
    wl, x, q_full, do_full, dk0, dv0 = _offload_case(21)
    kv = oomb.PagedKV(x.k_pool, x.v_pool, x.page_table, dk0.clone(), dv0.clone())
    o_r, dq_r, sels_r = oomb.chunk_recurrent_pass(q_full, do_full, kv, 512, 3)
    host = oomb.PagedKV(x.k_pool.cpu().pin_memory(), x.v_pool.cpu().pin_memory(),
                        x.page_table.cpu(), dk0.cpu().pin_memory(), dv0.cpu().pin_memory())
    cache = oomb.OffloadCache(host, 28, DEV, staging_bytes=staging)
    o_o, dq_o, sels_o = oomb.chunk_recurrent_pass_offloaded(q_full, do_full, cache, 512, 3,
                                                            prefetch=prefetch)
    torch.cuda.synchronize()
    for a, b in zip(sels_r, sels_o):
        assert torch.equal(a, b)
    assert torch.equal(_bits(o_r), _bits(o_o))
    # dQ sums the key tiles' contributions with fp32 atomics, in no fixed order:
    # equal up to that rounding, not bit for bit
    a, b = dq_r.float(), dq_o.float()
    assert float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(a)) < 1e-3
    assert float((a - b).abs().max()) <= 2 ** -7 * float(a.abs().max())
    assert torch.equal(_bits(kv.dk.cpu()), _bits(host.dk))
    assert torch.equal(_bits(kv.dv.cpu()), _bits(host.dv))
    st = cache.stats()
    assert st["slots_reused"] > 0 and st["tiles_out"] > 0, st
    assert st["bytes_in"] == st["tiles_in"] * 64 * 128 * 2
    cache.close()


def test_offload_pass_after_a_prefix_matches_resident():
    """The last 4 chunks of a sequence (start > 0, the prefix's representatives
    given): the offloaded pass fetches chunk 0's own pages first and makes
    chunk 1's selection during the rest of chunk 0's acquire.  Bit-identical O,
    selections and host dK/dV to the resident pass -- twice on one cache (the
    second pass reuses the cache's streams, page tables and workspaces)."""
    wl, x, q_full, do_full, dk0, dv0 = _offload_case(31)
    start = 2048
    q, do = q_full[:2048].contiguous(), do_full[:2048].contiguous()
    kv = oomb.PagedKV(x.k_pool, x.v_pool, x.page_table, dk0.clone(), dv0.clone())
    reps = gpu_reps(kv)
    o_r, dq_r, sels_r = oomb.chunk_recurrent_pass(q, do, kv, 512, 3, start=start,
                                                  reps=reps.clone())
    host = oomb.PagedKV(x.k_pool.cpu().pin_memory(), x.v_pool.cpu().pin_memory(),
                        x.page_table.cpu(), dk0.cpu().pin_memory(), dv0.cpu().pin_memory())
    cache = oomb.OffloadCache(host, 28, DEV)
    for _ in range(2):
        host.dk.copy_(dk0.cpu())
        host.dv.copy_(dv0.cpu())
        cache.flush(drop=True)
        torch.cuda.synchronize()
        o_o, dq_o, sels_o = oomb.chunk_recurrent_pass_offloaded(q, do, cache, 512, 3,
                                                                start=start, reps=reps.clone())
        torch.cuda.synchronize()
        for a, b in zip(sels_r, sels_o):
            assert torch.equal(a, b)
        assert torch.equal(_bits(o_r), _bits(o_o))
        a, b = dq_r.float(), dq_o.float()
        assert float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(a)) < 1e-3
        assert torch.equal(_bits(kv.dk.cpu()), _bits(host.dk))
        assert torch.equal(_bits(kv.dv.cpu()), _bits(host.dv))
    cache.close()


def test_offload_chunk_pass_fp32():
    """The same through the fp32 path (head_dim 64, P = 16, fp32 pools): 8 chunks
    of 128 rows, Top-8, 32 cache slots for 64 pages."""
    wl = W("offl32", "fp32", 2, 1, 1024, 16, 128, 8)
    x = make_inputs(wl, seed=23, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(24)
    q_full = torch.randn((1024, 2, 64), generator=g, device=DEV)
    do_full = torch.randn((1024, 2, 64), generator=g, device=DEV)
    dk0 = torch.randn(x.k_pool.shape, generator=g, device=DEV)
    dv0 = torch.randn(x.k_pool.shape, generator=g, device=DEV)
    kv = oomb.PagedKV(x.k_pool, x.v_pool, x.page_table, dk0.clone(), dv0.clone())
    o_r, dq_r, sels_r = oomb.chunk_recurrent_pass(q_full, do_full, kv, 128, 8)
    host = oomb.PagedKV(x.k_pool.cpu().pin_memory(), x.v_pool.cpu().pin_memory(),
                        x.page_table.cpu(), dk0.cpu().pin_memory(), dv0.cpu().pin_memory())
    cache = oomb.OffloadCache(host, 32, DEV)
    o_o, dq_o, sels_o = oomb.chunk_recurrent_pass_offloaded(q_full, do_full, cache, 128, 8)
    torch.cuda.synchronize()
    for a, b in zip(sels_r, sels_o):
        assert torch.equal(a, b)
    assert torch.equal(o_r, o_o) and torch.equal(dq_r, dq_o)
    assert torch.equal(kv.dk.cpu(), host.dk) and torch.equal(kv.dv.cpu(), host.dv)
    assert cache.stats()["slots_reused"] > 0
    cache.close()


def test_offload_ragged_sequence_matches_resident():
    """The offloaded pass over a sequence that ends inside a page (4001 tokens,
    chunks of 512, the last one 417 rows ending 33 rows into its last page):
    bit-identical O, selections and host dK/dV to the resident pass."""
    wl, x, q_full, do_full, dk0, dv0 = _offload_case(25)
    t = 4001
    _spoil_tail(x, t)
    q_full, do_full = q_full[:t].contiguous(), do_full[:t].contiguous()
    kv = oomb.PagedKV(x.k_pool, x.v_pool, x.page_table, dk0.clone(), dv0.clone())
    o_r, dq_r, sels_r = oomb.chunk_recurrent_pass(q_full, do_full, kv, 512, 3)
    host = oomb.PagedKV(x.k_pool.cpu().pin_memory(), x.v_pool.cpu().pin_memory(),
                        x.page_table.cpu(), dk0.cpu().pin_memory(), dv0.cpu().pin_memory())
    cache = oomb.OffloadCache(host, 28, DEV)
    o_o, dq_o, sels_o = oomb.chunk_recurrent_pass_offloaded(q_full, do_full, cache, 512, 3)
    torch.cuda.synchronize()
    assert len(sels_o) == 8
    for a, b in zip(sels_r, sels_o):
        assert torch.equal(a, b)
    assert torch.equal(_bits(o_r), _bits(o_o))
    a, b = dq_r.float(), dq_o.float()
    assert float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(a)) < 1e-3
    assert torch.equal(_bits(kv.dk.cpu()), _bits(host.dk))
    assert torch.equal(_bits(kv.dv.cpu()), _bits(host.dv))
    cache.close()


@pytest.mark.parametrize("staging", [0, 5 * 64 * 128 * 2], ids=["zero_copy", "staging_5_tiles"])
def test_offload_zero_grads_new_pass_matches_resident(staging):
    """Two offloaded passes over the same sequence: the first accumulates into
    nonzero host gradients; then the host dK/dV are zeroed and declared zero
    (a new pass), and the second pass -- whose first-touch gradient tiles are
    zero fills on the device, not copies -- ends with host dK/dV bit-identical
    to a resident pass from zero gradients, and the same O."""
    wl, x, q_full, do_full, dk0, dv0 = _offload_case(28)
    kv = oomb.PagedKV(x.k_pool, x.v_pool, x.page_table, torch.zeros_like(dk0),
                      torch.zeros_like(dv0))
    o_r, _, sels_r = oomb.chunk_recurrent_pass(q_full, do_full, kv, 512, 3)
    host = oomb.PagedKV(x.k_pool.cpu().pin_memory(), x.v_pool.cpu().pin_memory(),
                        x.page_table.cpu(), dk0.cpu().pin_memory(), dv0.cpu().pin_memory())
    cache = oomb.OffloadCache(host, 28, DEV, staging_bytes=staging)
    oomb.chunk_recurrent_pass_offloaded(q_full, do_full, cache, 512, 3)
    torch.cuda.synchronize()
    assert not torch.equal(_bits(host.dk), _bits(dk0.cpu()))      # the first pass wrote sums
    host.dk.zero_()
    host.dv.zero_()
    cache.zero_grads()
    before = cache.stats()
    o_o, _, sels_o = oomb.chunk_recurrent_pass_offloaded(q_full, do_full, cache, 512, 3)
    torch.cuda.synchronize()
    after = cache.stats()
    for a, b in zip(sels_r, sels_o):
        assert torch.equal(a, b)
    assert torch.equal(_bits(o_r), _bits(o_o))
    assert torch.equal(_bits(kv.dk.cpu()), _bits(host.dk))
    assert torch.equal(_bits(kv.dv.cpu()), _bits(host.dv))
    assert after["tiles_zero_filled"] - before["tiles_zero_filled"] > 0
    cache.close()


def _fp8_pools(x):
    """E4M3 copies of the workload's K/V pools and their exact bf16 values."""
    k8, v8 = x.k_pool.to(torch.float8_e4m3fn), x.v_pool.to(torch.float8_e4m3fn)
    return k8, v8, k8.to(torch.bfloat16), v8.to(torch.bfloat16)


@pytest.mark.parametrize("tier", ["host", "device"])
def test_fp8_kv_offload_matches_widened_resident(tier):
    """An fp8 KV cache: E4M3 K/V pools behind a bf16 device cache (pinned host
    memory, or device memory as a compact tier), expanded tile by tile on each
    fetch.  The chunk-recurrent pass gives bit-identical O, selections and
    dK/dV to the resident pass on bf16 pools holding the same values, and the
    same dQ up to the order of its fp32 atomic sums; K/V fetches move one byte
    per element."""
    wl, x, q_full, do_full, dk0, dv0 = _offload_case(26)
    k8, v8, kw, vw = _fp8_pools(x)
    kv = oomb.PagedKV(kw, vw, x.page_table, dk0.clone(), dv0.clone())
    o_r, dq_r, sels_r = oomb.chunk_recurrent_pass(q_full, do_full, kv, 512, 3)
    if tier == "host":
        back = oomb.PagedKV(k8.cpu().pin_memory(), v8.cpu().pin_memory(), x.page_table.cpu(),
                            dk0.cpu().pin_memory(), dv0.cpu().pin_memory())
    else:
        back = oomb.PagedKV(k8.clone(), v8.clone(), x.page_table.cpu(), dk0.clone(), dv0.clone())
    cache = oomb.OffloadCache(back, 28, DEV)
    o_o, dq_o, sels_o = oomb.chunk_recurrent_pass_offloaded(q_full, do_full, cache, 512, 3)
    torch.cuda.synchronize()
    for a, b in zip(sels_r, sels_o):
        assert torch.equal(a, b)
    assert torch.equal(_bits(o_r), _bits(o_o))
    a, b = dq_r.float(), dq_o.float()
    assert float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(a)) < 1e-3
    assert torch.equal(_bits(kv.dk.cpu()), _bits(back.dk.cpu()))
    assert torch.equal(_bits(kv.dv.cpu()), _bits(back.dv.cpu()))
    st = cache.stats()
    tile = 64 * 128
    assert st["slots_reused"] > 0
    assert tile * st["tiles_in"] < st["bytes_in"] < 2 * tile * st["tiles_in"]   # 1 B (K/V), 2 B (grads)
    cache.close()


def test_fp8_kv_offload_vs_oracle():
    """The fp8 KV cache against the oracle reading the E4M3 codes itself: the
    chunk-recurrent pass (8 chunks, Top-3, a cache that reuses slots) gives the
    oracle's selections, and O, dQ and dK/dV within the bf16 bounds."""
    wl, x, q_full, do_full, _, _ = _offload_case(27)
    k8, v8, _, _ = _fp8_pools(x)
    back = oomb.PagedKV(k8.cpu().pin_memory(), v8.cpu().pin_memory(), x.page_table.cpu(),
                        torch.zeros(x.k_pool.shape, dtype=torch.bfloat16).pin_memory(),
                        torch.zeros(x.k_pool.shape, dtype=torch.bfloat16).pin_memory())
    cache = oomb.OffloadCache(back, 28, DEV)
    o_g, dq_g, sels = oomb.chunk_recurrent_pass_offloaded(q_full, do_full, cache, 512, 3)
    torch.cuda.synchronize()
    kp = oracle.fp8_e4m3_decode(k8.view(torch.uint8).cpu().numpy())
    vp = oracle.fp8_e4m3_decode(v8.view(torch.uint8).cpu().numpy())
    pt = to_numpy64(x.page_table)
    o_o, dq_o, dk_o, dv_o, sels_o = oracle.chunk_recurrent_grads(
        to_numpy64(q_full), kp, vp, pt, to_numpy64(do_full), 512, 64, 3)
    for sg, so in zip(sels, sels_o):
        assert sg.cpu().numpy().tolist() == so.tolist()
    compare(o_g.float().cpu().numpy(), o_o, "bf16", "fp8 KV O")
    compare(dq_g.float().cpu().numpy(), dq_o, "bf16", "fp8 KV dQ")
    compare(to_numpy64(back.dk)[pt], dk_o, "bf16", "fp8 KV dK")
    compare(to_numpy64(back.dv)[pt], dv_o, "bf16", "fp8 KV dV")
    cache.close()


def test_step_pipeline_matches_sequential_steps():
    """Three steps with host-resident inputs and outputs through StepPipeline
    (copies overlapped with the neighbouring steps' compute) give the same O,
    LSE and accumulated dK/dV as three sparse_attention_step calls one after
    another, and the same dQ up to the order of its fp32 atomic sums."""
    wl = W("pipe", "bf16", 4, 2, 4096, 64, 512, 5)
    x = make_inputs(wl, seed=31, device=DEV)
    g = torch.Generator(device=DEV)
    g.manual_seed(32)
    qs = [torch.randn(x.q.shape, generator=g, device=DEV).to(torch.bfloat16) for _ in range(3)]
    dos = [torch.randn(x.q.shape, generator=g, device=DEV).to(torch.bfloat16) for _ in range(3)]
    kv_a = oomb.PagedKV(x.k_pool, x.v_pool, x.page_table, torch.zeros_like(x.k_pool),
                        torch.zeros_like(x.v_pool))
    ref = [oomb.sparse_attention_step(q, do, kv_a, wl.start, wl.top_k) for q, do in zip(qs, dos)]
    kv_b = oomb.PagedKV(x.k_pool, x.v_pool, x.page_table, torch.zeros_like(x.k_pool),
                        torch.zeros_like(x.v_pool))
    pipe = oomb.StepPipeline(kv_b, wl.start, wl.chunk_len, wl.num_q_heads, wl.top_k)
    outs = []
    for q, do in zip(qs, dos):
        q_h, do_h = q.cpu().pin_memory(), do.cpu().pin_memory()
        o_h = torch.empty_like(q_h).pin_memory()
        dq_h = torch.empty_like(q_h).pin_memory()
        lse_h = torch.empty((wl.num_q_heads, wl.chunk_len), dtype=torch.float32).pin_memory()
        pipe.step(q_h, do_h, o_h, lse_h, dq_h)
        outs.append((o_h, lse_h, dq_h, q_h, do_h))
    pipe.finish()
    torch.cuda.synchronize()
    for r, (o_h, lse_h, dq_h, _, _) in zip(ref, outs):
        assert torch.equal(_bits(r["o"].cpu()), _bits(o_h))
        assert torch.equal(r["lse"].cpu(), lse_h)
        a, b = r["dq"].float().cpu(), dq_h.float()
        assert float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(a)) < 1e-3
    assert torch.equal(_bits(kv_a.dk), _bits(kv_b.dk)) and torch.equal(_bits(kv_a.dv), _bits(kv_b.dv))


def test_offload_cache_too_small_is_refused():
    wl, x, q_full, do_full, dk0, dv0 = _offload_case(22)
    host = oomb.PagedKV(x.k_pool.cpu().pin_memory(), x.v_pool.cpu().pin_memory(),
                        x.page_table.cpu(), dk0.cpu().pin_memory(), dv0.cpu().pin_memory())
    cache = oomb.OffloadCache(host, 10, DEV)           # the last chunk alone needs 14
    pt = torch.full((wl.num_pages,), -1, dtype=torch.int32, device=DEV)
    with pytest.raises(oomb.OombError) as e:
        cache.acquire(None, 0, 0, 1024, False, pt)     # 16 own pages
    assert e.value.code == oomb.OOMB_ERR_INVALID_ARG and "cache slots" in str(e.value)
    cache.acquire(None, 0, 0, 512, False, pt)          # 8 own pages fit
    torch.cuda.synchronize()
    assert sorted(pt[:8].tolist()) == list(range(8)) and torch.all(pt[8:] == -1)
    cache.close()


def test_deterministic_selection_and_forward():
    wl = W("det", "bf16", 8, 2, 8192, 64, 512, 31)
    x = make_inputs(wl, seed=9, device=DEV)
    kv = gpu_kv(x, with_grads=False)
    reps = gpu_reps(kv)
    s1, sc1 = gpu_select(x, kv, reps, wl.top_k)
    s2, sc2 = gpu_select(x, kv, gpu_reps(kv), wl.top_k)
    assert torch.equal(s1, s2) and torch.equal(sc1, sc2)
    o1, l1 = gpu_fwd(x, kv, s1.contiguous(), s1.shape[1])
    o2, l2 = gpu_fwd(x, kv, s1.contiguous(), s1.shape[1])
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bounded_wait_reports_timeout_and_context_survives():
    kv = gpu_kv(make_inputs(W("t", "bf16", 4, 2, 1024, 64, 128, 2), device=DEV), with_grads=False)
    ws = oomb.workspace(oomb.OOMB_OP_ATTN_FWD, kv)
    oomb.oomb_set_wait_limit_ns(1_000_000)   # 1 ms
    try:
        oomb.oomb_debug_wait_unset_flag(ws)
        code, where, _ = oomb.oomb_device_status(ws)
    finally:
        oomb.oomb_set_wait_limit_ns(0)
    assert code == oomb.OOMB_ERR_TIMEOUT and where == 90
    # the context is still usable: a normal call completes with OK status
    reps = gpu_reps(kv)
    assert torch.isfinite(reps).all()


def test_out_of_range_selection_is_flagged_not_read():
    wl = W("oob", "bf16", 4, 2, 2048, 64, 256, 4)
    x = make_inputs(wl, device=DEV)
    kv = gpu_kv(x)
    bad = torch.tensor([[0, 1, 2, 10_000], [0, 1, 2, 3]], dtype=torch.int32, device=DEV)
    o = torch.empty_like(x.q)
    lse = torch.empty((4, 256), dtype=torch.float32, device=DEV)
    ws = oomb.workspace(oomb.OOMB_OP_ATTN_FWD, kv)
    oomb.oomb_sparse_attn_fwd(x.q, kv, bad, 4, wl.start, o, lse, ws)
    code, _, _ = oomb.oomb_device_status(ws)
    assert code == oomb.OOMB_ERR_DEVICE_BOUNDS


def test_device_page_table_validation():
    wl = W("pt", "bf16", 4, 2, 1024, 64, 128, 2)
    x = make_inputs(wl, device=DEV)
    kv = gpu_kv(x, with_grads=False)
    ws = oomb.workspace(oomb.OOMB_OP_VALIDATE, kv)
    oomb.oomb_validate_page_table(kv, ws)
    bad = x.page_table.clone()
    bad[3] = bad[5]
    with pytest.raises(oomb.OombError, match="two pages"):
        oomb.oomb_validate_page_table(oomb.PagedKV(x.k_pool, x.v_pool, bad), ws)
    bad[3] = 99
    with pytest.raises(oomb.OombError, match="outside"):
        oomb.oomb_validate_page_table(oomb.PagedKV(x.k_pool, x.v_pool, bad), ws)


# ---------------------------------------------------------------------------
# the named workloads at full size
# ---------------------------------------------------------------------------
FULL = ["qwen7b_dense_ctx32k", "qwen7b_ctx256k_k64", "qwen7b_ctx1m_k128", "qwen7b_ctx4m_k128"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    wl = WORKLOADS[name]
    x = make_inputs(wl, seed=0, device=DEV)
    kv = gpu_kv(x)
    reps = gpu_reps(kv)
    reps64 = oracle_reps_blocked(x.k_pool, x.page_table)
    rs = np.random.default_rng(1).choice(wl.num_pages, 256, replace=False)
    compare(reps[rs].cpu().numpy(), reps64[rs], "fp32", f"{name} reps (256 sampled pages)")
    sel_g, _ = gpu_select(x, kv, reps, wl.top_k)
    sel_o, scores_o = oracle_selection(x, reps64, wl.top_k)
    flagged = check_selection(sel_g.cpu().numpy(), sel_o, scores_o)
    print(f"{name}: near-tie swaps flagged: {flagged}")
    n_sel = sel_o.shape[1]
    st = sel_tensor(sel_o, DEV)
    o_g, lse_g, o_lo = gpu_fwd(x, kv, st, n_sel, with_lo=True)
    dq_g = gpu_bwd(x, kv, st, n_sel, o_g, lse_g, o_lo=o_lo)
    # oracle on 512 sampled rows (all heads) and on 8 sampled selected pages
    # plus 4 own pages of every KV head; the oracle's forward runs over every
    # row, because a page's dK/dV sums over all of them (and needs their LSE
    # and O)
    q, do = to_numpy64(x.q), to_numpy64(x.do)
    pt = x.page_table.cpu().numpy().astype(np.int64)
    rng = np.random.default_rng(2)
    inner = rng.choice(np.arange(1, wl.chunk_len - 1), 510, replace=False)
    rows = np.unique(np.concatenate([inner, [0, wl.chunk_len - 1]]))
    assert rows.size == 512
    # gather just the pages the oracle needs into a compact host pool
    own = np.arange(wl.start // wl.page_size, (wl.start + wl.chunk_len) // wl.page_size)
    need = np.unique(np.concatenate([sel_o.reshape(-1), own]))
    slots = torch.as_tensor(pt[need])
    kc = x.k_pool[slots.to(DEV)].float().cpu().numpy()
    vc = x.v_pool[slots.to(DEV)].float().cpu().numpy()
    ptc = np.full(wl.num_pages, -1, np.int64)
    ptc[need] = np.arange(need.size)
    o_all, lse_all = oracle.attn_fwd(q, kc, vc, ptc, sel_o, wl.start, wl.page_size)
    o_o, lse_o = o_all[rows], lse_all[:, rows]
    compare(o_g.float().cpu().numpy()[rows], o_o, "bf16", f"{name} O (512 sampled rows)")
    np.testing.assert_allclose(lse_g.cpu().numpy()[:, rows], lse_o, atol=2e-3)
    dq_o = oracle.attn_dq_rows(q, kc, vc, ptc, sel_o, wl.start, wl.page_size, o_o, lse_o, do, rows)
    compare(dq_g.float().cpu().numpy()[rows], dq_o, "bf16", f"{name} dQ (512 sampled rows)")
    for g in range(wl.num_kv_heads):
        pages = np.concatenate([rng.choice(sel_o[g], min(8, n_sel), replace=False),
                                rng.choice(own, 4, replace=False)])
        dk_o, dv_o = oracle.attn_bwd_pages(q, kc, vc, ptc, sel_o, wl.start, wl.page_size, o_all,
                                           lse_all, do, g, pages)
        dk_g = kv.dk[torch.as_tensor(pt[pages], device=DEV), g].float().cpu().numpy()
        dv_g = kv.dv[torch.as_tensor(pt[pages], device=DEV), g].float().cpu().numpy()
        compare(dk_g, dk_o, "bf16", f"{name} dK (12 sampled pages, KV head {g})")
        compare(dv_g, dv_o, "bf16", f"{name} dV (12 sampled pages, KV head {g})")
    del x, kv
    torch.cuda.empty_cache()
