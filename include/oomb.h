/*
 * oomb.h -- C ABI of liboomb: page-level sparse causal attention of one query
 * chunk against a paged KV cache, forward and backward, on one GB300 (sm_103a).
 *
 * Method: "Out of the Memory Barrier: A Highly Memory Efficient Training
 * System for LLMs with Million-Token Contexts" (gist.science summary of arXiv
 * 2602.02108), technical summary section 2 "Methodology":
 *   - "Paged Memory Management": the KV cache AND its gradients are allocated
 *     per page; gradients are accumulated in place, outside autograd.
 *   - "Page-level Sparse Attention": Top-K page retrieval; for dense-attention
 *     models the forward picks the most relevant key pages from
 *     representative vectors and the backward reuses that choice.
 *   - "Specialized Kernels": KV-cache operations are kept out of the autograd
 *     graph (this ABI has no autograd at all).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no device memory; scratch comes from the caller's workspace
 *     `ws` (size from oomb_workspace_bytes, 256-byte aligned, zero-filled
 *     before its first use; the library leaves its counters at zero after
 *     every call that completes).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on it, except oomb_validate_page_table and
 *     oomb_device_status, which synchronise the stream.
 *   - Argument errors are detected on the host and returned before anything
 *     is launched (OOMB_ERR_INVALID_ARG / OOMB_ERR_UNSUPPORTED, with a message
 *     from oomb_last_error()).  Errors found on the device (a bounded wait that
 *     timed out, an index out of range, a non-finite unused row of a partial
 *     last page) are recorded in the status word at the
 *     start of `ws` and read with oomb_device_status.  No call traps or
 *     asserts on the device.
 *   - Tensor layouts (row-major, innermost last):
 *       K/V pools and dK/dV pools  [num_slots][Hkv][P][D]   (one page of one
 *                                   KV head is a contiguous P x D tile)
 *       page_table                 int32 [num_pages], logical page -> slot,
 *                                   injective on the pages a call reads, each
 *                                   of those entries in [0, num_slots); the
 *                                   other entries are not read (a page cache
 *                                   may hold fewer slots than pages and mark
 *                                   absent pages -1).  An entry a kernel reads
 *                                   out of range is recorded as
 *                                   OOMB_ERR_DEVICE_BOUNDS, never followed.
 *       q, o, o_lo, dout, dq       [chunk_len][Hq][D]
 *       lse                        float [Hq][chunk_len], natural log
 *       reps                       float [num_pages][Hkv][D], logical order
 *       sel                        int32 [Hkv][n_sel], ascending, unique
 *   - GQA: query head h uses KV head h / (Hq / Hkv).
 *   - Own pages of a chunk: logical pages [chunk_start/P, ceil((chunk_start +
 *     chunk_len)/P)).  Candidates: logical pages [0, chunk_start/P).
 *   - Supported: bf16 with D = 128 and P in {16, 32, 64, 128}; fp32 with
 *     D = 64 and P in {16, 32, 64, 128}.  chunk_start is a multiple of P and
 *     chunk_len >= 1, chunk_start + chunk_len <= num_pages * P.
 *   - Partial last page (a sequence whose length is not a multiple of P; only
 *     its last chunk can end inside a page, since every chunk starts on one):
 *     the rows of that page past chunk_start + chunk_len hold no token.  They
 *     are never attended and their dK/dV rows are left as they are, but the
 *     tensor-core kernels load them with the page and weight them by zero, so
 *     their K and V values must be finite (a zero-initialised pool is; in fp8
 *     backing pools of an offload cache, codes other than the NaN codes).
 *     On bf16 pools oomb_sparse_attn_fwd(_own_reps) and oomb_sparse_attn_bwd
 *     check those rows first whenever the chunk ends inside a page (one small
 *     launch reading only the unused rows) and record OOMB_ERR_NONFINITE in
 *     the workspace status when any of them holds an inf or a NaN; the
 *     outputs of that call are then not meaningful.
 */
#ifndef OOMB_H
#define OOMB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OOMB_OK = 0,
  OOMB_ERR_INVALID_ARG = 1,   /* bad pointer, shape, alignment or index  */
  OOMB_ERR_UNSUPPORTED = 2,   /* valid request this build does not serve */
  OOMB_ERR_CUDA = 3,          /* a CUDA runtime call failed              */
  OOMB_ERR_TIMEOUT = 4,       /* a device-side bounded wait gave up      */
  OOMB_ERR_DEVICE_BOUNDS = 5, /* a device-side index check failed        */
  OOMB_ERR_NONFINITE = 6      /* inf/NaN in the unused rows of a partial
                                 last page (device check, bf16 pools)     */
} oomb_status;

/* OOMB_FP8_E4M3: 8-bit E4M3 codes (OCP 8-bit floating point specification),
 * a storage format only: the K/V pools of an offload cache's backing tier
 * (oomb_offload_desc.backing_kv_dtype).  Every kernel computes on bf16. */
typedef enum { OOMB_BF16 = 0, OOMB_FP32 = 1, OOMB_FP8_E4M3 = 2 } oomb_dtype;

/* The paged KV cache and its paged gradient buffers (Paged Memory Management
 * item).  dk/dv may be NULL for forward-only use. */
typedef struct {
  void *k, *v;
  void *dk, *dv;
  const int32_t *page_table;
  int32_t num_pages;
  int32_t num_slots;
  int32_t page_size;     /* P */
  int32_t num_kv_heads;  /* Hkv */
  int32_t head_dim;      /* D */
  int32_t dtype;         /* oomb_dtype of k, v, dk, dv, q, o, dout, dq */
} oomb_paged_kv;

typedef enum {
  OOMB_OP_VALIDATE = 0,
  OOMB_OP_PAGE_REPS = 1,
  OOMB_OP_SELECT_TOPK = 2,
  OOMB_OP_ATTN_FWD = 3,
  OOMB_OP_ATTN_BWD = 4
} oomb_op;

/* Bytes of workspace `op` needs for these shapes (>= 256: the status block).
 * top_k is used by OOMB_OP_SELECT_TOPK only.  Returns 0 for an unknown op. */
size_t oomb_workspace_bytes(int op, const oomb_paged_kv *kv, int32_t num_q_heads,
                            int32_t chunk_len, int32_t top_k);

/* Host-only check of a host copy of a page table: every entry in
 * [0, num_slots) and no slot used twice (a shared slot would make two
 * backward tiles update the same gradient page).  Paged Memory Management. */
oomb_status oomb_validate_page_table_host(const int32_t *page_table, int32_t num_pages,
                                          int32_t num_slots);

/* The same check on the device copy kv->page_table, using ws as a slot
 * bitmap.  Synchronises `stream`.  Returns OOMB_ERR_INVALID_ARG if the table
 * is out of range or not injective. */
oomb_status oomb_validate_page_table(const oomb_paged_kv *kv, void *ws, size_t ws_bytes,
                                     void *stream);

/* Step 1 -- representative vector of each page (Page-level Sparse Attention
 * item: "representative vectors"; reading: the fp32 mean of the page's P
 * keys, per KV head).  For logical pages [first_page, first_page + n_pages):
 *   reps[l][g][d] = (1/P) sum_t K[page_table[l]][g][t][d]     (fp32 accumulate)
 * reps points at the row of logical page 0 ([num_pages][Hkv][D]); only the
 * requested rows are written.  ws: oomb_workspace_bytes(PAGE_REPS) (status
 * word only).  Every page is taken as P keys: the representative of a
 * partial last page comes from oomb_sparse_attn_fwd_own_reps, which knows
 * where the chunk ends. */
oomb_status oomb_page_reps(const oomb_paged_kv *kv, int32_t first_page, int32_t n_pages,
                           float *reps, void *ws, size_t ws_bytes, void *stream);

/* Step 2 -- Top-K page selection per (chunk, KV head) (Page-level Sparse
 * Attention item: "Top-K page retrieval").  With qbar[g] the fp32 mean of q
 * over the chunk's tokens and the heads of group g:
 *   score[g][l] = qbar[g] . reps[l][g]      for candidates l < chunk_start/P
 * keeps the n_sel = min(top_k, chunk_start/P) highest scores per KV head;
 * equal scores go to the lower page index; sel[g][0..n_sel) is written in
 * ascending page order.  scores_opt, if not NULL, receives float
 * [Hkv][num_pages] (non-candidates = -inf).  Deterministic: the fp32
 * reductions run in a fixed order.  One cooperative kernel with one CTA per
 * SM (its CTAs wait for one another; each wait is bounded and records
 * OOMB_ERR_TIMEOUT in the status word of ws if it runs out).
 * ws: oomb_workspace_bytes(SELECT_TOPK). */
oomb_status oomb_select_topk(const void *q, int32_t num_q_heads, int32_t chunk_len,
                             int32_t chunk_start, const float *reps, const oomb_paged_kv *kv,
                             int32_t top_k, int32_t *sel, float *scores_opt, void *ws,
                             size_t ws_bytes, void *stream);

/* Top-K page selection exactly as oomb_select_topk, for callers that cannot
 * allocate device memory -- for example code running inside a CUDA graph
 * whose memory is fixed up front, or a host framework that owns every device
 * allocation and hands this library only its input and output buffers.  The
 * paper has no counterpart; it is a property of this library's interface.
 * Instead of a workspace argument the call uses a scratch array inside the
 * library: a file-scope device array of OOMB_NOALLOC_SCRATCH_BYTES (4 MiB),
 * which every GPU that loads the library holds until the process exits.  It
 * must hold oomb_workspace_bytes(OOMB_OP_SELECT_TOPK, ...) for these shapes
 * (about 256 B + 1152 B * Hkv * D + 256 KiB * Hkv + 4 B * Hkv * num_pages,
 * e.g. up to ~159K pages at Hkv = 4, D = 128); larger requests return
 * OOMB_ERR_INVALID_ARG before anything is launched.  The
 * first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  The call
 * never calls cudaMalloc, cudaFree or any allocating routine.  All calls
 * share the one array, which keeps the last call's contents: the call clears
 * the part that must start at zero, and calls that overlap on the GPU (other
 * streams, other host threads) race on it -- serialise them.  The status word
 * where the selection records a bounded wait that ran out is in that array,
 * which a caller of this entry point cannot read. */
#define OOMB_NOALLOC_SCRATCH_BYTES (4u << 20)
oomb_status oomb_select_topk_noalloc(const void *q, int32_t num_q_heads, int32_t chunk_len,
                                     int32_t chunk_start, const float *reps,
                                     const oomb_paged_kv *kv, int32_t top_k, int32_t *sel,
                                     float *scores_opt, void *stream);

/* Step 3 -- sparse attention forward (Page-level Sparse Attention item).
 * For query head h (KV head g) and chunk row t (position p = chunk_start+t)
 * the keys are all tokens of the n_sel pages sel[g][*] plus the chunk's own
 * tokens at positions <= p:
 *   o[t][h] = softmax_k(scale * q[t][h] . k) v,  lse[h][t] = log sum_k exp(...)
 * scale <= 0 selects 1/sqrt(D).  bf16: tcgen05 tensor cores, fp32
 * accumulation, o rounded once to bf16.  fp32: CUDA-core FMA.
 * o_lo (optional, bf16 pools only; NULL to skip): [chunk_len][Hq][D] bf16,
 * the rounding residual of o -- o_lo = bf16(o32 - o) where o32 is the fp32
 * value that o rounds -- so that o + o_lo carries o32 to about 16 bits.
 * Pass it to the backward: its row sums Delta = dout . o are subtracted from
 * dP = dout . v_k, and in a row whose attention concentrates on one key the
 * two nearly cancel, so the bf16 rounding of o alone (2^-9 relative) would
 * leave an error of up to 2^-9 |Delta| in dS and in dQ.
 * sel must be the same array later passed to the backward (the backward
 * reuses the forward's choice). */
oomb_status oomb_sparse_attn_fwd(const void *q, const oomb_paged_kv *kv, const int32_t *sel,
                                 int32_t n_sel, int32_t num_q_heads, int32_t chunk_len,
                                 int32_t chunk_start, float scale, void *o, void *o_lo,
                                 float *lse, void *ws, size_t ws_bytes, void *stream);

/* Step 3 with step 1 of the chunk's own pages fused in (Chunk-Recurrent
 * Training Framework: the pages a chunk writes become candidates for the
 * chunks after it, so their representatives are needed as soon as the
 * chunk's forward is done).  Computes exactly what oomb_sparse_attn_fwd
 * computes and, in addition, reps[l][g][*] for the chunk's own pages
 * l in [chunk_start/P, ceil((chunk_start+chunk_len)/P)) and every KV head g --
 * the same values oomb_page_reps writes for those pages (bf16: bit-identical;
 * the forward kernel sums the K tiles it has already loaded into shared
 * memory in oomb_page_reps's order, so the chunk's keys are not read again).
 * A partial last own page is represented by the mean of its rows that hold
 * the chunk's keys (oomb_page_reps always takes whole pages).
 * reps: float [num_pages][Hkv][D], 16-byte aligned; other rows are not
 * touched.  fp32 pools: the representatives come from the representatives
 * kernel launched after the forward on the same stream (not fused).
 * Arguments, workspace and errors as oomb_sparse_attn_fwd. */
oomb_status oomb_sparse_attn_fwd_own_reps(const void *q, const oomb_paged_kv *kv,
                                          const int32_t *sel, int32_t n_sel,
                                          int32_t num_q_heads, int32_t chunk_len,
                                          int32_t chunk_start, float scale, void *o, void *o_lo,
                                          float *lse, float *reps, void *ws, size_t ws_bytes,
                                          void *stream);

/* Step 4 -- sparse attention backward with in-place paged gradient
 * accumulation (Paged Memory Management: gradients of the KV cache are
 * paged and accumulated in place; Page-level Sparse Attention: the selection
 * of the forward is reused).  Recomputes P = exp(scale q.k - lse); with
 * Delta[t][h] = dout[t][h] . o[t][h]:
 *   dq[t][h]  = scale sum_k P (dP - Delta) k              (written)
 *   dK[slot]  += scale sum_{t,h in group} P (dP - Delta) q   (read-add-write)
 *   dV[slot]  += sum_{t,h in group} P dout                    (read-add-write)
 * for the slots of the selected and own pages only; each of those slots is
 * rounded once per call.  kv->dk and kv->dv must be set.
 * o_lo: the forward's rounding residual of o (bf16 pools; may be NULL): with
 * it, Delta = dout . (o + o_lo), the forward's fp32 output, instead of
 * dout . o -- see oomb_sparse_attn_fwd for why the rows whose attention
 * concentrates on one key need it.  fp32 pools: must be NULL.
 * ws: oomb_workspace_bytes(ATTN_BWD) (holds Delta and an fp32 dq accumulator). */
oomb_status oomb_sparse_attn_bwd(const void *q, const void *o, const void *o_lo,
                                 const void *dout, const float *lse, const oomb_paged_kv *kv,
                                 const int32_t *sel, int32_t n_sel, int32_t num_q_heads,
                                 int32_t chunk_len, int32_t chunk_start, float scale, void *dq,
                                 void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Host-tier pools with a device page cache (the method's fourth optimisation,
 * "Async CPU offloading": the KV cache and its gradients stay in host memory
 * and only the pages a chunk attends are brought to the GPU, ahead of the
 * kernels that read them).
 *
 * The K, V, dK and dV pools of every page live in pinned host memory
 * ([num_host_slots][Hkv][P][D], caller-owned, allocated with cudaHostAlloc or
 * registered; the GPU reads and writes them directly over the CPU-GPU link).
 * With the zero-copy moves (dev_staging NULL) this backing tier may instead be
 * device memory: a compact tier in HBM in front of which the cache holds the
 * working pages.
 *
 * fp8 KV (backing_kv_dtype = OOMB_FP8_E4M3, dtype = OOMB_BF16): the backing K
 * and V pools hold E4M3 codes (one byte per element, P x D bytes per tile) and
 * each fetch expands a tile to bf16 in the cache.  Every E4M3 value is a bf16
 * value, so the expansion is exact and the kernels compute on exactly the
 * stored values; dK/dV stay bf16 in both tiers.  Zero-copy moves only.
 * A cache of cache_slots page slots ([cache_slots][Hkv][P][D] for each of
 * K, V, dK, dV) lives in caller-owned device memory.  The unit moved is one
 * (page, KV head) tile of P x D elements; a cache slot holds one logical page
 * and only the tiles of the KV heads that use it.
 *
 * oomb_offload_acquire(sel_host, chunk_start, chunk_len, with_grads) makes
 * resident every tile the chunk's kernels read: (sel[g][i], g) for every KV
 * head g and i < n_sel, and all heads of the chunk's own pages.  Missing K/V
 * tiles (and, with with_grads, dK/dV tiles) are copied host -> cache; a slot
 * that must be reused first writes its modified dK/dV tiles back to the host
 * pools.  Gradient tiles are write-back: acquire with with_grads marks them
 * modified (the backward that follows adds into them in place) and they
 * return to the host pools on reuse of their slot or on oomb_offload_flush.
 * The host pools therefore end bit-identical to a run with every page in HBM.
 * Then the call writes the device page table `page_table_dev` (int32
 * [num_pages]: cache slot of every resident page, -1 elsewhere).  The chunk's
 * kernels then take an oomb_paged_kv with the cache pools, num_slots =
 * cache_slots and page_table = page_table_dev.
 *
 * Moves are enqueued on `stream` (see dev_staging below for the two ways);
 * the call returns after enqueueing them.  Slots used by this acquire and by
 * the one before it are never reused, so the acquire for chunk c+1 may run on
 * another stream while the kernels of chunk c are in flight; kernels of older
 * acquires must have completed (the caller orders the streams with events),
 * and each in-flight chunk needs its own page_table_dev.  The call blocks the
 * host only until the moves enqueued four calls earlier (acquire, flush or
 * writeback) have completed (four pinned staging buffers).  Errors:
 * OOMB_ERR_INVALID_ARG if a page index is out of range or the chunk's pages
 * do not fit in the cache next to those of the previous acquire (the
 * directory is then unchanged); OOMB_ERR_CUDA if a launch or copy fails.
 * oomb_offload_create rejects a host page table that is out of range or not
 * injective.
 * ------------------------------------------------------------------------- */
typedef struct {
  void *k, *v, *dk, *dv;          /* backing tier (pinned host or device); dk/dv may be NULL (forward only) */
  const int32_t *host_page_table; /* HOST int32 [num_pages]: logical page -> host slot, injective */
  int32_t num_pages, num_host_slots, page_size, num_kv_heads, head_dim;
  oomb_dtype dtype;
  void *cache_k, *cache_v, *cache_dk, *cache_dv;  /* device tier [cache_slots][Hkv][P][D] */
  int32_t cache_slots;
  /* Optional device staging buffer (caller-owned, 16-byte aligned).  If set,
   * tiles move through it and a pinned host staging buffer of the same size
   * that the library allocates: tiles are gathered on the host (a stream
   * callback with a few threads) and cross the CPU-GPU link in one copy-engine
   * transfer per round of dev_staging_bytes, leaving the SMs to the attention
   * kernels; successive calls are ordered on the GPU (they share the staging
   * buffers).  If NULL, a copy kernel reads and writes the host pools
   * directly (zero-copy), which needs SMs. */
  void *dev_staging;
  int64_t dev_staging_bytes;
  /* Element type of the backing K/V pools: dtype, or OOMB_FP8_E4M3 with
   * dtype OOMB_BF16 (see fp8 KV above). */
  oomb_dtype backing_kv_dtype;
} oomb_offload_desc;

typedef struct oomb_offload oomb_offload;   /* opaque; host memory of the library */

/* Checks the description (the backing pools must be pinned host memory, or
 * device memory with zero-copy moves; the cache pools device memory), copies
 * the host page table and allocates the handle's host state and pinned
 * staging buffers.  No device memory.  OOMB_ERR_UNSUPPORTED for fp8 K/V with
 * a staging buffer. */
oomb_status oomb_offload_create(const oomb_offload_desc *desc, oomb_offload **out);
oomb_status oomb_offload_acquire(oomb_offload *h, const int32_t *sel_host, int32_t n_sel,
                                 int32_t chunk_start, int32_t chunk_len, int32_t with_grads,
                                 int32_t *page_table_dev, void *stream);
/* Writes every modified dK/dV tile back to the host pools (enqueued on
 * `stream`, after the kernels that modified them).  drop != 0 also forgets
 * every cached tile (for a caller that rewrites host K/V pages). */
oomb_status oomb_offload_flush(oomb_offload *h, int32_t drop, void *stream);
/* Writes the modified dK/dV tiles of pages [first_page, first_page + n_pages)
 * back to the host pools now (enqueued on `stream`; the caller orders it after
 * the kernels that modified them) and marks them clean.  For pages whose
 * gradients are final before the pass ends -- in a backward over the chunks in
 * reverse order, a chunk's own pages once its backward is done -- so that the
 * final flush has less to move. */
oomb_status oomb_offload_writeback(oomb_offload *h, int32_t first_page, int32_t n_pages,
                                   void *stream);
/* The same for a list of logical pages (pages_host: host int32 [n], each in
 * [0, num_pages), repeats allowed; read before the call returns).  In a
 * backward over the chunks in reverse order, the gradient tiles of a page are
 * final once the backward of the last chunk to touch it (as an own or a
 * selected page) is done.  A page modified again after its write-back is
 * simply written back again.  OOMB_ERR_INVALID_ARG (nothing enqueued) for a
 * page out of range. */
oomb_status oomb_offload_writeback_pages(oomb_offload *h, const int32_t *pages_host, int32_t n,
                                         void *stream);
/* Declares that the caller has set every tile of the host dK/dV pools to zero
 * (the start of a new pass over the sequence).  The cache's gradient tiles are
 * forgotten without being written back (their sums belonged to the previous
 * pass); the K/V tiles stay cached.  From then on, until a gradient tile is
 * written back again, an acquire that needs it fills the cache tile with zeros
 * on the device instead of copying it over the link.  Host-only bookkeeping:
 * nothing is enqueued, so the caller orders it after the kernels and moves of
 * the previous pass (and after its own zeroing of the host pools).
 * OOMB_ERR_INVALID_ARG without gradient pools. */
oomb_status oomb_offload_zero_grads(oomb_offload *h);
/* Counters since create: out[0] tiles copied host -> cache, out[1] tiles
 * written back, out[2] bytes host -> cache, out[3] bytes cache -> host,
 * out[4] acquires, out[5] slots reused, out[6] gradient tiles zero-filled on
 * the device instead of copied.  out: int64_t[7]. */
oomb_status oomb_offload_stats(const oomb_offload *h, int64_t *out);
/* Frees the handle (waits for its staging buffers' last moves). */
void oomb_offload_destroy(oomb_offload *h);

/* Reads and clears the device status word at the start of ws (synchronises
 * `stream`).  Returns OOMB_OK, OOMB_ERR_TIMEOUT, OOMB_ERR_DEVICE_BOUNDS or
 * OOMB_ERR_NONFINITE; info (optional, 2 ints) receives {where, block} of the
 * first error. */
oomb_status oomb_device_status(void *ws, void *stream, int32_t *info);

/* Upper bound, in nanoseconds, of every device-side wait (default 2e9).
 * Process-wide; for tests of the timeout path.  0 restores the default. */
void oomb_set_wait_limit_ns(uint64_t ns);

/* Debug: a one-thread kernel that waits on a flag in ws nothing ever sets,
 * bounded by the wait limit; records OOMB_ERR_TIMEOUT in the status word. */
oomb_status oomb_debug_wait_unset_flag(void *ws, size_t ws_bytes, void *stream);

const char *oomb_status_string(int status);

/* Message of the last host-side error of the calling thread ("" if none). */
const char *oomb_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* OOMB_H */
