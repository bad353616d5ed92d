"""CPU float64 oracle for page-level sparse causal attention over a paged KV cache.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  It shares no code with the CUDA path and never imports the package.

Source: "Out of the Memory Barrier: A Highly Memory Efficient Training System
for LLMs with Million-Token Contexts" (gist.science summary of arXiv
2602.02108), technical summary section 2 ("Methodology"), items
"Paged Memory Management" and "Page-level Sparse Attention".  The summary
states the method in words only: KV cache and its gradients live in pages,
gradients are accumulated in place outside autograd, and for dense-attention
models the most relevant key pages are chosen from representative vectors in
the forward pass and the same choice is reused in the backward pass.  Every
quantity it leaves open is fixed below by the plainest reading, listed in the
function that uses it.

Layouts (all arrays are NumPy; the oracle reads stored values exactly, so bf16
tensors are passed in after an exact widening to float32 or float64):

* K/V pools: ``[num_slots, Hkv, P, D]``; one page of one KV head is ``[P, D]``.
* page table: ``int [num_pages]``, logical page -> physical slot.
* queries, outputs, output grads: ``[C, Hq, D]`` for the chunk's C tokens.
* LSE: ``[Hq, C]``, natural log.
* GQA: query head h reads KV head ``h // G`` with ``G = Hq // Hkv``.

Arithmetic is float64 throughout except where the method itself fixes a
narrower precision (the fp32 representative vectors and the fp32 scores on
which the Top-K decision is taken).

Parity pins (tests/test_oracle.py): every function here is pinned against
something other than itself -- torch's CPU scaled-dot-product attention with
autograd (dense equality), closed-form worked examples (tests/golden/),
brute-force pair means, order invariants of the Top-K, rows of the softmax
summing to one, central finite differences, cross-chunk accumulation equal to
the single-pass dense gradient (also over sequences that end inside a page),
closed forms of a partial page's representative, and the E4M3 decoding against
hand-worked codes and torch's float8_e4m3fn conversion.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "page_reps",
    "query_summary",
    "page_scores",
    "select_topk",
    "key_positions",
    "attn_fwd",
    "attn_bwd",
    "attn_bwd_pages",
    "attn_dq_rows",
    "dense_causal_reference",
    "chunk_recurrent_grads",
    "fp8_e4m3_decode",
]


# ---------------------------------------------------------------------------
# Step 1: representative vector of each page
# ---------------------------------------------------------------------------
def page_reps(k_pool, page_table, first_page=0, n_pages=None, block=1024, n_tokens=None):
    """Mean of each page's keys, per KV head.

    Page-level Sparse Attention item: pages are ranked by a representative
    vector whose definition the summary does not give.  Reading: the mean of
    the page's P keys as stored in the cache, one vector per (logical page,
    KV head).  Returns float64 ``[n_pages, Hkv, D]`` (the caller rounds to
    fp32 where the stored representative is fp32).  Pages are processed in
    groups of ``block`` only to bound host memory; each page's mean is
    independent of every other page.

    ``n_tokens`` (optional) is the length of the sequence when its last page
    is only partly written.  Reading: a page holds only the tokens written to
    it, so the page that ``n_tokens`` cuts is represented by the mean of its
    keys at positions below ``n_tokens``; the rows after them hold no token.
    A page wholly at or after ``n_tokens`` has no representative (ValueError).
    """
    pt = np.asarray(page_table)
    if n_pages is None:
        n_pages = pt.shape[0] - first_page
    num_slots, hkv, p, d = k_pool.shape
    out = np.empty((n_pages, hkv, d), np.float64)
    if n_tokens is not None and n_pages > 0 and (first_page + n_pages - 1) * p >= n_tokens:
        raise ValueError("a page with no token before n_tokens has no representative")
    for b0 in range(0, n_pages, block):
        b1 = min(n_pages, b0 + block)
        slots = pt[first_page + b0:first_page + b1]
        out[b0:b1] = k_pool[slots].astype(np.float64).mean(axis=2)
    cut = None if n_tokens is None or n_tokens % p == 0 else n_tokens // p
    if cut is not None and first_page <= cut < first_page + n_pages:
        # the partial page: only its first n_tokens % P rows hold tokens
        out[cut - first_page] = k_pool[pt[cut], :, :n_tokens % p].astype(np.float64).mean(axis=1)
    return out


# ---------------------------------------------------------------------------
# Step 2: Top-K page selection per (chunk, KV head)
# ---------------------------------------------------------------------------
def query_summary(q, num_kv_heads):
    """Mean query of one KV-head group over the chunk.

    Reading of "most relevant key pages for the current chunk": one selection
    per (chunk, KV head), so the chunk is summarised per group as the mean of
    Q over its C tokens and the G query heads that share the KV head.  By
    bilinearity ``qbar . rep`` is then the mean raw logit ``q . k`` over every
    (query of the group, key of the page) pair.  Returns float64 ``[Hkv, D]``.
    """
    c, hq, d = q.shape
    g = hq // num_kv_heads
    return q.astype(np.float64).reshape(c, num_kv_heads, g, d).mean(axis=(0, 2))


def page_scores(qbar, reps, n_cand):
    """fp32 relevance score of each candidate page for each KV head.

    The Top-K decision is an integer decided by floating point, so it is
    taken in the precision the method stores its representative vectors in
    (fp32): the fp32 representative and fp32 group-mean query are formed by
    rounding their float64 means once, their dot product is taken exactly in
    float64 and rounded once to fp32.  No 1/sqrt(D) factor: a positive scale
    cannot change the ranking.  Returns float32 ``[Hkv, n_cand]``.
    """
    q32 = np.asarray(qbar, np.float64).astype(np.float32).astype(np.float64)
    r32 = np.asarray(reps[:n_cand], np.float64).astype(np.float32).astype(np.float64)
    s = np.einsum("gd,lgd->gl", q32, r32)
    return s.astype(np.float32)


def select_topk(scores, top_k):
    """The ``top_k`` best candidates per KV head, returned in ascending order.

    Candidates are ordered by score, higher first; equal scores go to the
    lower logical page index.  If ``top_k`` is at least the number of
    candidates, every candidate is selected.  Returns int32 ``[Hkv, k]`` with
    ``k = min(top_k, n_cand)``.
    """
    scores = np.asarray(scores)
    hkv, n = scores.shape
    k = min(int(top_k), n)
    sel = np.empty((hkv, k), np.int32)
    idx = np.arange(n)
    for g in range(hkv):
        order = np.lexsort((idx, -scores[g].astype(np.float64)))
        sel[g] = np.sort(order[:k])
    return sel


# ---------------------------------------------------------------------------
# Steps 3 and 4: attention over the selected pages plus the chunk's own pages
# ---------------------------------------------------------------------------
def key_positions(sel_g, chunk_start, chunk_len, page_size):
    """Absolute token positions a query of the chunk may look at (KV head g).

    The selected past pages (all tokens) followed by the chunk's own tokens
    ``[chunk_start, chunk_start + chunk_len)``; the causal mask is applied by
    the caller.
    """
    sel_g = np.asarray(sel_g, np.int64)
    sel_pos = (sel_g[:, None] * page_size + np.arange(page_size)[None, :]).reshape(-1)
    own_pos = chunk_start + np.arange(chunk_len, dtype=np.int64)
    return np.concatenate([sel_pos, own_pos])


def _gather(pool, page_table, positions, g, page_size):
    pt = np.asarray(page_table, np.int64)
    pages = positions // page_size
    offs = positions % page_size
    return pool[pt[pages], g, offs].astype(np.float64)


def _scores(qh, kset, key_pos, query_pos, scale):
    s = scale * (qh @ kset.T)
    allowed = key_pos[None, :] <= query_pos[:, None]
    return np.where(allowed, s, -np.inf), allowed


def attn_fwd(q, k_pool, v_pool, page_table, sel, chunk_start, page_size, scale=None,
             rows=None, kv_heads=None, row_block=1024):
    """Forward of page-level sparse causal attention for one query chunk.

    For query head h (KV head g = h // G) and chunk row t (absolute position
    p = chunk_start + t), the keys are every token of the pages in ``sel[g]``
    plus the chunk's own tokens at positions <= p.  Logits are
    ``scale * q . k`` with ``scale = 1/sqrt(D)`` unless given; the softmax is
    the two-pass form (row max, then exponentials).  Returns float64
    ``O [len(rows), Hq, D]`` and ``lse [Hq, len(rows)]`` (natural log).
    Only the heads of ``kv_heads`` (default all) are filled; the others are
    left NaN.  Rows are processed ``row_block`` at a time only to bound host
    memory.
    """
    c, hq, d = q.shape
    hkv = k_pool.shape[1]
    grp = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.arange(c) if rows is None else np.asarray(rows)
    kv_heads = range(hkv) if kv_heads is None else kv_heads
    o = np.full((rows.shape[0], hq, d), np.nan)
    lse = np.full((hq, rows.shape[0]), np.nan)
    for g in kv_heads:
        kpos = key_positions(sel[g], chunk_start, c, page_size)
        kset = _gather(k_pool, page_table, kpos, g, page_size)
        vset = _gather(v_pool, page_table, kpos, g, page_size)
        for r0 in range(0, rows.shape[0], row_block):
            rr = rows[r0:r0 + row_block]
            qpos = chunk_start + rr
            for h in range(g * grp, (g + 1) * grp):
                s, _ = _scores(q[rr, h].astype(np.float64), kset, kpos, qpos, scale)
                m = s.max(axis=1)
                e = np.exp(s - m[:, None])
                l = e.sum(axis=1)
                o[r0:r0 + rr.shape[0], h] = (e @ vset) / l[:, None]
                lse[h, r0:r0 + rr.shape[0]] = m + np.log(l)
    return o, lse


def attn_bwd(q, k_pool, v_pool, page_table, sel, chunk_start, page_size, o, lse, do,
             scale=None, dk_acc=None, dv_acc=None, row_block=1024, acc_rows=None):
    """Backward of the sparse attention with the same selection as the forward.

    Recomputes P = exp(s - lse) from the saved LSE, then with
    Delta_t = sum_d dO_t . O_t (per head):
    dV_k += sum_t P_tk dO_t, dP_tk = dO_t . v_k, dS = P (dP - Delta),
    dQ_t = scale sum_k dS_tk k_k, dK_k += scale sum_t dS_tk q_t, where the
    sums over t also run over the G heads of the group.  The selection is
    not differentiated and the representative vectors get no gradient.

    dK/dV are added in place into ``dk_acc``/``dv_acc`` (float64, indexed by
    LOGICAL page ``[num_pages, Hkv, P, D]``; created if None), which is how
    gradients reach the paged buffers across chunks.  ``acc_rows`` (optional)
    maps a logical page to its row of the accumulators, for callers that keep
    accumulators for the touched pages only.  Returns
    ``(dq [C, Hq, D], dk_acc, dv_acc)``.
    """
    c, hq, d = q.shape
    hkv = k_pool.shape[1]
    grp = hq // hkv
    n_pages = np.asarray(page_table).shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if dk_acc is None:
        dk_acc = np.zeros((n_pages, hkv, page_size, d))
    if dv_acc is None:
        dv_acc = np.zeros((n_pages, hkv, page_size, d))
    dq = np.zeros((c, hq, d))
    for g in range(hkv):
        kpos = key_positions(sel[g], chunk_start, c, page_size)
        kset = _gather(k_pool, page_table, kpos, g, page_size)
        vset = _gather(v_pool, page_table, kpos, g, page_size)
        dks = np.zeros_like(kset)
        dvs = np.zeros_like(vset)
        for r0 in range(0, c, row_block):
            rr = np.arange(r0, min(c, r0 + row_block))
            qpos = chunk_start + rr
            for h in range(g * grp, (g + 1) * grp):
                qh = q[rr, h].astype(np.float64)
                doh = do[rr, h].astype(np.float64)
                oh = o[rr, h].astype(np.float64)
                s, allowed = _scores(qh, kset, kpos, qpos, scale)
                p = np.where(allowed, np.exp(s - lse[h, rr][:, None]), 0.0)
                dvs += p.T @ doh
                dp = doh @ vset.T
                delta = (doh * oh).sum(axis=1)
                ds = p * (dp - delta[:, None])
                dq[rr, h] = scale * (ds @ kset)
                dks += scale * (ds.T @ qh)
        pages = kpos // page_size
        if acc_rows is not None:
            pages = np.asarray(acc_rows)[pages]
        offs = kpos % page_size
        np.add.at(dk_acc, (pages, g, offs), dks)
        np.add.at(dv_acc, (pages, g, offs), dvs)
    return dq, dk_acc, dv_acc


def attn_bwd_pages(q, k_pool, v_pool, page_table, sel, chunk_start, page_size, o, lse, do,
                   g, pages, scale=None, row_block=1024):
    """dK/dV of one call for a few logical pages of KV head ``g`` only.

    Same arithmetic as :func:`attn_bwd` restricted to the key columns of
    ``pages``; every query row of the chunk and every head of the group
    contributes.  Needs ``o``/``lse`` for all rows of the group's heads.
    Returns float64 ``(dk [len(pages), P, D], dv [len(pages), P, D])``.
    """
    c, hq, d = q.shape
    hkv = k_pool.shape[1]
    grp = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    pages = np.asarray(pages, np.int64)
    kpos = (pages[:, None] * page_size + np.arange(page_size)[None, :]).reshape(-1)
    kset = _gather(k_pool, page_table, kpos, g, page_size)
    vset = _gather(v_pool, page_table, kpos, g, page_size)
    dks = np.zeros_like(kset)
    dvs = np.zeros_like(vset)
    for r0 in range(0, c, row_block):
        rr = np.arange(r0, min(c, r0 + row_block))
        qpos = chunk_start + rr
        for h in range(g * grp, (g + 1) * grp):
            qh = q[rr, h].astype(np.float64)
            doh = do[rr, h].astype(np.float64)
            oh = o[rr, h].astype(np.float64)
            s, allowed = _scores(qh, kset, kpos, qpos, scale)
            p = np.where(allowed, np.exp(s - lse[h, rr][:, None]), 0.0)
            dvs += p.T @ doh
            dp = doh @ vset.T
            delta = (doh * oh).sum(axis=1)
            ds = p * (dp - delta[:, None])
            dks += scale * (ds.T @ qh)
    n = pages.shape[0]
    return dks.reshape(n, page_size, d), dvs.reshape(n, page_size, d)


def attn_dq_rows(q, k_pool, v_pool, page_table, sel, chunk_start, page_size, o_rows, lse_rows,
                 do, rows, scale=None):
    """dQ of a few chunk rows only (every head), same arithmetic as :func:`attn_bwd`.

    ``o_rows [len(rows), Hq, D]`` and ``lse_rows [Hq, len(rows)]`` are the
    forward outputs of those rows.  Returns float64 ``[len(rows), Hq, D]``.
    """
    c, hq, d = q.shape
    hkv = k_pool.shape[1]
    grp = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.asarray(rows)
    qpos = chunk_start + rows
    dq = np.zeros((rows.shape[0], hq, d))
    for g in range(hkv):
        kpos = key_positions(sel[g], chunk_start, c, page_size)
        kset = _gather(k_pool, page_table, kpos, g, page_size)
        vset = _gather(v_pool, page_table, kpos, g, page_size)
        for h in range(g * grp, (g + 1) * grp):
            qh = q[rows, h].astype(np.float64)
            doh = do[rows, h].astype(np.float64)
            s, allowed = _scores(qh, kset, kpos, qpos, scale)
            p = np.where(allowed, np.exp(s - lse_rows[h][:, None]), 0.0)
            dp = doh @ vset.T
            delta = (doh * o_rows[:, h]).sum(axis=1)
            dq[:, h] = scale * ((p * (dp - delta[:, None])) @ kset)
    return dq


# ---------------------------------------------------------------------------
# Textbook dense causal attention (no pages, no selection) -- small inputs only
# ---------------------------------------------------------------------------
def dense_causal_reference(q, k, v, do, scale=None):
    """Full-context causal attention and its gradients, written densely.

    ``q, do: [T, Hq, D]``, ``k, v: [T, Hkv, D]`` in logical token order.
    Materialises the [T, T] masked score matrix per head.  Returns float64
    ``(o, lse [Hq, T], dq, dk, dv)`` with dk/dv summed over each group's heads.
    """
    t, hq, d = q.shape
    hkv = k.shape[1]
    grp = hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q = q.astype(np.float64); k = k.astype(np.float64)
    v = v.astype(np.float64); do = do.astype(np.float64)
    o = np.zeros_like(q); dq = np.zeros_like(q)
    dk = np.zeros_like(k); dv = np.zeros_like(v)
    lse = np.zeros((hq, t))
    mask = np.tril(np.ones((t, t), bool))
    for h in range(hq):
        g = h // grp
        s = np.where(mask, scale * q[:, h] @ k[:, g].T, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        p = e / l
        o[:, h] = p @ v[:, g]
        lse[h] = (m + np.log(l))[:, 0]
        dv[:, g] += p.T @ do[:, h]
        dp = do[:, h] @ v[:, g].T
        ds = p * (dp - (do[:, h] * o[:, h]).sum(axis=1, keepdims=True))
        dq[:, h] = scale * ds @ k[:, g]
        dk[:, g] += scale * ds.T @ q[:, h]
    return o, lse, dq, dk, dv


def chunk_recurrent_grads(q_full, k_pool, v_pool, page_table, do_full, chunk_len, page_size,
                          top_k, scale=None):
    """Chunk-recurrent pass: forward chunks in order, backward in reverse.

    Chunk-Recurrent Training Framework item: the sequence is processed as
    chunks; the backward of each chunk recomputes what it needs.  Each chunk
    c scores its past pages, keeps ``top_k`` of them, and attends them plus
    its own causal pages; chunks are then differentiated from last to first,
    every call adding its dK/dV into the same logical-page accumulators.
    ``chunk_len`` is a multiple of P, so every chunk starts on a page; when T
    is not a multiple of ``chunk_len`` the last chunk is shorter, and when T
    is not a multiple of P its last page is partial (its rows past T are
    neither attended nor given gradient).
    Returns ``(o_full, dq_full, dk_acc, dv_acc, sels)``.
    """
    t, hq, d = q_full.shape
    hkv = k_pool.shape[1]
    if chunk_len % page_size:
        raise ValueError("chunks must start on a page boundary")
    n_chunks = -(-t // chunk_len)
    reps = page_reps(k_pool, page_table, 0, -(-t // page_size), n_tokens=t)
    outs, sels = [], []
    for c in range(n_chunks):
        t0 = c * chunk_len
        qc = q_full[t0:t0 + chunk_len]
        n_cand = t0 // page_size
        sc = page_scores(query_summary(qc, hkv), reps, n_cand)
        sel = select_topk(sc, top_k) if n_cand > 0 else np.zeros((hkv, 0), np.int32)
        o, lse = attn_fwd(qc, k_pool, v_pool, page_table, sel, t0, page_size, scale)
        outs.append((o, lse)); sels.append(sel)
    dk_acc = dv_acc = None
    dq_full = np.zeros((t, hq, d))
    for c in reversed(range(n_chunks)):
        t0 = c * chunk_len
        o, lse = outs[c]
        dq, dk_acc, dv_acc = attn_bwd(q_full[t0:t0 + chunk_len], k_pool, v_pool, page_table,
                                      sels[c], t0, page_size, o, lse,
                                      do_full[t0:t0 + chunk_len], scale, dk_acc, dv_acc)
        dq_full[t0:t0 + chunk_len] = dq
    o_full = np.concatenate([o for o, _ in outs], axis=0)
    return o_full, dq_full, dk_acc, dv_acc, sels


# ---------------------------------------------------------------------------
# Storage variant: K/V pools held as 8-bit E4M3 codes
# ---------------------------------------------------------------------------
def fp8_e4m3_decode(codes):
    """Value of each 8-bit E4M3 code (OCP 8-bit floating point specification,
    E4M3 format): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
    Exponent field 0 encodes the subnormals m * 2^-9; the fields (15, 7) encode
    NaN; there are no infinities, so 0x7E = 448 is the largest finite value.

    Reading for an fp8 KV cache: a stored code stands for exactly this value
    (no scale factor), and the path computes on these values as it does on the
    values of a bf16 pool.  Returns float64 with the shape of ``codes``.
    """
    b = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(b >> 7 == 1, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = m * 2.0 ** -9
    val = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & (m == 7), np.nan, val)
