// C ABI of liboomb (declared in include/oomb.h): host-side argument checks,
// workspace layout and dispatch to the kernels.  No exception crosses the ABI;
// every error is a status code plus a message for oomb_last_error().
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include "oomb.h"
#include "oomb_internal.h"

namespace {

thread_local char g_err[512] = "";
uint64_t g_wait_ns = 2000000000ull;

oomb_status fail(oomb_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

}  // namespace

oomb_status oomb::report(oomb_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

namespace {

oomb_status cuda_fail(cudaError_t e, const char* what) {
  return fail(OOMB_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

oomb_status check_kv(const oomb_paged_kv* kv) {
  if (!kv) return fail(OOMB_ERR_INVALID_ARG, "kv is NULL");
  if (!kv->k || !kv->v || !kv->page_table)
    return fail(OOMB_ERR_INVALID_ARG, "kv->k, kv->v and kv->page_table must be set");
  if (kv->dtype == OOMB_FP8_E4M3)
    return fail(OOMB_ERR_UNSUPPORTED,
                "kv->dtype OOMB_FP8_E4M3 is a storage format of the offload backing tier; "
                "the kernels read bf16 pools");
  if (kv->dtype != OOMB_BF16 && kv->dtype != OOMB_FP32)
    return fail(OOMB_ERR_INVALID_ARG, "kv->dtype %d is not OOMB_BF16 or OOMB_FP32", kv->dtype);
  if (kv->num_pages <= 0 || kv->num_slots <= 0)
    return fail(OOMB_ERR_INVALID_ARG, "need num_pages > 0 and num_slots > 0 (got %d, %d)",
                kv->num_pages, kv->num_slots);
  const int P = kv->page_size;
  if (P != 16 && P != 32 && P != 64 && P != 128)
    return fail(OOMB_ERR_UNSUPPORTED, "page_size %d not in {16, 32, 64, 128}", P);
  if (kv->num_kv_heads <= 0 || kv->num_kv_heads > 16)
    return fail(OOMB_ERR_UNSUPPORTED, "num_kv_heads %d not in [1, 16]", kv->num_kv_heads);
  const int want_d = kv->dtype == OOMB_BF16 ? 128 : 64;
  if (kv->head_dim != want_d)
    return fail(OOMB_ERR_UNSUPPORTED, "head_dim %d: this build serves %s with head_dim %d",
                kv->head_dim, kv->dtype == OOMB_BF16 ? "bf16" : "fp32", want_d);
  if (static_cast<long long>(kv->num_slots) * kv->num_kv_heads * P >= (1ll << 31))
    return fail(OOMB_ERR_UNSUPPORTED, "num_slots * Hkv * P must stay below 2^31");
  if (!aligned(kv->k, 16) || !aligned(kv->v, 16) || (kv->dk && !aligned(kv->dk, 16)) ||
      (kv->dv && !aligned(kv->dv, 16)))
    return fail(OOMB_ERR_INVALID_ARG, "K/V/dK/dV pools must be 16-byte aligned");
  return OOMB_OK;
}

oomb_status check_chunk(const oomb_paged_kv* kv, int hq, int chunk_len, int chunk_start) {
  const int P = kv->page_size;
  if (hq <= 0 || hq % kv->num_kv_heads != 0)
    return fail(OOMB_ERR_INVALID_ARG, "num_q_heads %d must be a positive multiple of Hkv %d", hq,
                kv->num_kv_heads);
  // the chunk may end inside a page (the last page of a sequence that is not
  // whole pages); it always starts on one
  if (chunk_len <= 0) return fail(OOMB_ERR_INVALID_ARG, "chunk_len %d must be positive", chunk_len);
  if (chunk_start < 0 || chunk_start % P != 0)
    return fail(OOMB_ERR_INVALID_ARG, "chunk_start %d must be a non-negative multiple of P=%d",
                chunk_start, P);
  if (static_cast<long long>(chunk_start) + chunk_len > static_cast<long long>(kv->num_pages) * P)
    return fail(OOMB_ERR_INVALID_ARG, "chunk [%d, %d) runs past the %d pages of the cache",
                chunk_start, chunk_start + chunk_len, kv->num_pages);
  return OOMB_OK;
}

oomb_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return fail(OOMB_ERR_INVALID_ARG, "ws is NULL");
  if (!aligned(ws, 256)) return fail(OOMB_ERR_INVALID_ARG, "ws must be 256-byte aligned");
  if (ws_bytes < need)
    return fail(OOMB_ERR_INVALID_ARG, "ws has %zu bytes, %zu needed", ws_bytes, need);
  return OOMB_OK;
}

oomb::KvDesc desc(const oomb_paged_kv* kv) {
  oomb::KvDesc d;
  d.k = kv->k;
  d.v = kv->v;
  d.dk = kv->dk;
  d.dv = kv->dv;
  d.page_table = kv->page_table;
  d.num_pages = kv->num_pages;
  d.num_slots = kv->num_slots;
  d.page_size = kv->page_size;
  d.hkv = kv->num_kv_heads;
  d.head_dim = kv->head_dim;
  return d;
}

float resolve_scale(float scale, int head_dim) {
  return scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
}

}  // namespace

extern "C" {

const char* oomb_status_string(int s) {
  switch (s) {
    case OOMB_OK: return "OOMB_OK";
    case OOMB_ERR_INVALID_ARG: return "OOMB_ERR_INVALID_ARG";
    case OOMB_ERR_UNSUPPORTED: return "OOMB_ERR_UNSUPPORTED";
    case OOMB_ERR_CUDA: return "OOMB_ERR_CUDA";
    case OOMB_ERR_TIMEOUT: return "OOMB_ERR_TIMEOUT";
    case OOMB_ERR_DEVICE_BOUNDS: return "OOMB_ERR_DEVICE_BOUNDS";
    case OOMB_ERR_NONFINITE: return "OOMB_ERR_NONFINITE";
    default: return "OOMB_ERR_UNKNOWN";
  }
}

const char* oomb_last_error(void) { return g_err; }

void oomb_set_wait_limit_ns(uint64_t ns) { g_wait_ns = ns ? ns : 2000000000ull; }

size_t oomb_workspace_bytes(int op, const oomb_paged_kv* kv, int32_t num_q_heads,
                            int32_t chunk_len, int32_t top_k) {
  (void)top_k;
  if (!kv) return 0;
  switch (op) {
    case OOMB_OP_VALIDATE:
      return oomb::kStatusBytes +
             oomb::align_up(static_cast<size_t>((kv->num_slots + 31) / 32) * 4, 256);
    case OOMB_OP_PAGE_REPS:
    case OOMB_OP_ATTN_FWD:
      return oomb::kStatusBytes;
    case OOMB_OP_SELECT_TOPK:
      return oomb::select_ws_bytes(kv->num_pages, kv->num_kv_heads, kv->head_dim);
    case OOMB_OP_ATTN_BWD:
      return kv->dtype == OOMB_BF16
                 ? oomb::bf16_bwd_ws_bytes(num_q_heads, chunk_len, kv->head_dim)
                 : oomb::fp32_bwd_ws_bytes(num_q_heads, chunk_len);
    default:
      return 0;
  }
}

oomb_status oomb_validate_page_table_host(const int32_t* pt, int32_t num_pages,
                                          int32_t num_slots) {
  if (!pt || num_pages <= 0 || num_slots <= 0)
    return fail(OOMB_ERR_INVALID_ARG, "page table: need a pointer, num_pages > 0, num_slots > 0");
  std::vector<unsigned char> used(static_cast<size_t>(num_slots), 0);
  for (int32_t l = 0; l < num_pages; ++l) {
    const int32_t s = pt[l];
    if (s < 0 || s >= num_slots)
      return fail(OOMB_ERR_INVALID_ARG, "page_table[%d] = %d is outside [0, %d)", l, s, num_slots);
    if (used[static_cast<size_t>(s)])
      return fail(OOMB_ERR_INVALID_ARG, "slot %d is used by more than one page (page %d)", s, l);
    used[static_cast<size_t>(s)] = 1;
  }
  return OOMB_OK;
}

oomb_status oomb_device_status(void* ws, void* stream, int32_t* info) {
  OOMB_NVTX_RANGE("oomb_device_status");
  if (!ws) return fail(OOMB_ERR_INVALID_ARG, "ws is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int h[3] = {0, 0, 0};
  cudaError_t e = cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  e = cudaMemsetAsync(ws, 0, sizeof(h), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
  if (info) {
    info[0] = h[1];
    info[1] = h[2];
  }
  if (h[0] == 0) return OOMB_OK;
  if (h[0] == OOMB_ERR_TIMEOUT)
    return fail(OOMB_ERR_TIMEOUT, "device wait timed out (where %d, block %d)", h[1], h[2]);
  if (h[0] == OOMB_ERR_NONFINITE)
    return fail(OOMB_ERR_NONFINITE, "inf or NaN in the unused rows of a partial last page "
                "(KV head %d)", h[2]);
  return fail(OOMB_ERR_DEVICE_BOUNDS, "device index check failed (where %d, block %d)", h[1],
              h[2]);
}

oomb_status oomb_validate_page_table(const oomb_paged_kv* kv, void* ws, size_t ws_bytes,
                                     void* stream) {
  OOMB_NVTX_RANGE("oomb_validate_page_table");
  oomb_status s = check_kv(kv);
  if (s != OOMB_OK) return s;
  s = check_ws(ws, ws_bytes, oomb_workspace_bytes(OOMB_OP_VALIDATE, kv, 0, 0, 0));
  if (s != OOMB_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  const size_t bm = static_cast<size_t>((kv->num_slots + 31) / 32) * 4;
  cudaError_t e = cudaMemsetAsync(w + oomb::kStatusBytes, 0, bm, st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the slot bitmap");
  e = oomb::launch_validate_page_table(kv->page_table, kv->num_pages, kv->num_slots,
                                       reinterpret_cast<uint32_t*>(w + oomb::kStatusBytes),
                                       reinterpret_cast<int*>(w), st);
  if (e != cudaSuccess) return cuda_fail(e, "launching the page-table check");
  int32_t info[2];
  s = oomb_device_status(ws, stream, info);
  if (s == OOMB_ERR_DEVICE_BOUNDS)
    return fail(OOMB_ERR_INVALID_ARG, info[0] == 1 ? "page table entry outside [0, num_slots)"
                                                   : "page table maps two pages to one slot");
  return s;
}

oomb_status oomb_page_reps(const oomb_paged_kv* kv, int32_t first_page, int32_t n_pages,
                           float* reps, void* ws, size_t ws_bytes, void* stream) {
  OOMB_NVTX_RANGE("oomb_page_reps");
  oomb_status s = check_kv(kv);
  if (s != OOMB_OK) return s;
  if (!reps) return fail(OOMB_ERR_INVALID_ARG, "reps is NULL");
  if (first_page < 0 || n_pages < 0 ||
      static_cast<long long>(first_page) + n_pages > kv->num_pages)
    return fail(OOMB_ERR_INVALID_ARG, "pages [%d, %d) outside [0, %d)", first_page,
                first_page + n_pages, kv->num_pages);
  s = check_ws(ws, ws_bytes, oomb::kStatusBytes);
  if (s != OOMB_OK) return s;
  cudaError_t e = oomb::launch_page_reps(desc(kv), kv->dtype == OOMB_BF16, first_page, n_pages,
                                         kv->page_size, reps, static_cast<int*>(ws),
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? OOMB_OK : cuda_fail(e, "oomb_page_reps launch");
}

oomb_status oomb_select_topk(const void* q, int32_t num_q_heads, int32_t chunk_len,
                             int32_t chunk_start, const float* reps, const oomb_paged_kv* kv,
                             int32_t top_k, int32_t* sel, float* scores_opt, void* ws,
                             size_t ws_bytes, void* stream) {
  OOMB_NVTX_RANGE("oomb_select_topk");
  oomb_status s = check_kv(kv);
  if (s != OOMB_OK) return s;
  s = check_chunk(kv, num_q_heads, chunk_len, chunk_start);
  if (s != OOMB_OK) return s;
  if (!q || !reps) return fail(OOMB_ERR_INVALID_ARG, "q and reps must be set");
  if (!aligned(q, 16) || !aligned(reps, 16) || (scores_opt && !aligned(scores_opt, 16)))
    return fail(OOMB_ERR_INVALID_ARG, "q, reps and scores must be 16-byte aligned");
  if (top_k < 0) return fail(OOMB_ERR_INVALID_ARG, "top_k %d < 0", top_k);
  const int n_cand = chunk_start / kv->page_size;
  const int n_sel = top_k < n_cand ? top_k : n_cand;
  if (n_sel > 0 && !sel) return fail(OOMB_ERR_INVALID_ARG, "sel is NULL");
  const int vec_elems = kv->dtype == OOMB_BF16 ? 8 : 4;
  if (static_cast<long long>(num_q_heads) * kv->head_dim / vec_elems > 896)
    return fail(OOMB_ERR_UNSUPPORTED, "num_q_heads * head_dim too large for the query summary");
  s = check_ws(ws, ws_bytes, oomb::select_ws_bytes(kv->num_pages, kv->num_kv_heads, kv->head_dim));
  if (s != OOMB_OK) return s;
  cudaError_t e = oomb::launch_select_topk(q, kv->dtype == OOMB_BF16, num_q_heads, chunk_len,
                                           n_cand, reps, kv->num_pages, kv->num_kv_heads,
                                           kv->head_dim, n_sel, sel, scores_opt, ws, g_wait_ns,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? OOMB_OK : cuda_fail(e, "oomb_select_topk launch");
}

oomb_status oomb_select_topk_noalloc(const void* q, int32_t num_q_heads, int32_t chunk_len,
                                     int32_t chunk_start, const float* reps,
                                     const oomb_paged_kv* kv, int32_t top_k, int32_t* sel,
                                     float* scores_opt, void* stream) {
  OOMB_NVTX_RANGE("oomb_select_topk_noalloc");
  oomb_status s = check_kv(kv);
  if (s != OOMB_OK) return s;
  s = check_chunk(kv, num_q_heads, chunk_len, chunk_start);
  if (s != OOMB_OK) return s;
  if (!q || !reps) return fail(OOMB_ERR_INVALID_ARG, "q and reps must be set");
  if (!aligned(q, 16) || !aligned(reps, 16) || (scores_opt && !aligned(scores_opt, 16)))
    return fail(OOMB_ERR_INVALID_ARG, "q, reps and scores must be 16-byte aligned");
  if (top_k < 0) return fail(OOMB_ERR_INVALID_ARG, "top_k %d < 0", top_k);
  const int n_cand = chunk_start / kv->page_size;
  const int n_sel = top_k < n_cand ? top_k : n_cand;
  if (n_sel > 0 && !sel) return fail(OOMB_ERR_INVALID_ARG, "sel is NULL");
  const int vec_elems = kv->dtype == OOMB_BF16 ? 8 : 4;
  if (static_cast<long long>(num_q_heads) * kv->head_dim / vec_elems > 896)
    return fail(OOMB_ERR_UNSUPPORTED, "num_q_heads * head_dim too large for the query summary");
  bool too_big = false;
  cudaError_t e = oomb::launch_select_topk_noalloc(
      q, kv->dtype == OOMB_BF16, num_q_heads, chunk_len, n_cand, reps, kv->num_pages,
      kv->num_kv_heads, kv->head_dim, n_sel, sel, scores_opt, &too_big, g_wait_ns,
      static_cast<cudaStream_t>(stream));
  if (too_big)
    return fail(OOMB_ERR_INVALID_ARG,
                "selection needs %zu bytes of scratch; the fixed scratch holds %u bytes "
                "(use oomb_select_topk with a workspace)",
                oomb::select_ws_bytes(kv->num_pages, kv->num_kv_heads, kv->head_dim),
                OOMB_NOALLOC_SCRATCH_BYTES);
  return e == cudaSuccess ? OOMB_OK : cuda_fail(e, "oomb_select_topk_noalloc");
}

// A chunk that ends inside a page: check that the page's unused rows are finite
// (the tensor-core kernels weight them by zero).
static cudaError_t check_tail_rows(const oomb_paged_kv* kv, int chunk_len, int chunk_start,
                                   int* status, cudaStream_t st) {
  const int end = chunk_start + chunk_len;
  const int P = kv->page_size;
  if (end % P == 0) return cudaSuccess;
  return oomb::launch_check_tail_rows(desc(kv), end / P, end % P, status, st);
}

static oomb_status attn_fwd(const char* name, const void* q, const oomb_paged_kv* kv,
                            const int32_t* sel, int32_t n_sel, int32_t num_q_heads,
                            int32_t chunk_len, int32_t chunk_start, float scale, void* o,
                            void* o_lo, float* lse, float* own_reps, void* ws, size_t ws_bytes,
                            void* stream) {
  oomb_status s = check_kv(kv);
  if (s != OOMB_OK) return s;
  s = check_chunk(kv, num_q_heads, chunk_len, chunk_start);
  if (s != OOMB_OK) return s;
  if (!q || !o || !lse) return fail(OOMB_ERR_INVALID_ARG, "q, o and lse must be set");
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(lse, 16) || !aligned(o_lo, 16))
    return fail(OOMB_ERR_INVALID_ARG, "q, o, o_lo and lse must be 16-byte aligned");
  if (o_lo && kv->dtype != OOMB_BF16)
    return fail(OOMB_ERR_INVALID_ARG, "o_lo is for bf16 pools (an fp32 o needs no residual)");
  const int n_cand = chunk_start / kv->page_size;
  if (n_sel < 0 || n_sel > n_cand)
    return fail(OOMB_ERR_INVALID_ARG, "n_sel %d outside [0, %d] (pages before the chunk)", n_sel,
                n_cand);
  if (n_sel > 0 && !sel) return fail(OOMB_ERR_INVALID_ARG, "sel is NULL");
  s = check_ws(ws, ws_bytes, oomb::kStatusBytes);
  if (s != OOMB_OK) return s;
  const float sc = resolve_scale(scale, kv->head_dim);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (kv->dtype == OOMB_BF16) {
    e = check_tail_rows(kv, chunk_len, chunk_start, static_cast<int*>(ws), st);
    if (e == cudaSuccess)
      e = oomb::launch_attn_fwd_bf16(q, desc(kv), sel, n_sel, num_q_heads, chunk_len, chunk_start,
                                     sc, o, o_lo, lse, own_reps, static_cast<int*>(ws),
                                     g_wait_ns, st);
  } else {
    e = oomb::launch_attn_fwd_fp32(static_cast<const float*>(q), desc(kv), sel, n_sel,
                                   num_q_heads, chunk_len, chunk_start, sc,
                                   static_cast<float*>(o), lse, static_cast<int*>(ws), st);
    if (e == cudaSuccess && own_reps != nullptr)
      e = oomb::launch_page_reps(desc(kv), false, chunk_start / kv->page_size,
                                 (chunk_len + kv->page_size - 1) / kv->page_size,
                                 (chunk_len - 1) % kv->page_size + 1, own_reps,
                                 static_cast<int*>(ws), st);
  }
  return e == cudaSuccess ? OOMB_OK : cuda_fail(e, name);
}

oomb_status oomb_sparse_attn_fwd(const void* q, const oomb_paged_kv* kv, const int32_t* sel,
                                 int32_t n_sel, int32_t num_q_heads, int32_t chunk_len,
                                 int32_t chunk_start, float scale, void* o, void* o_lo,
                                 float* lse, void* ws, size_t ws_bytes, void* stream) {
  OOMB_NVTX_RANGE("oomb_sparse_attn_fwd");
  return attn_fwd("oomb_sparse_attn_fwd", q, kv, sel, n_sel, num_q_heads, chunk_len, chunk_start,
                  scale, o, o_lo, lse, nullptr, ws, ws_bytes, stream);
}

oomb_status oomb_sparse_attn_fwd_own_reps(const void* q, const oomb_paged_kv* kv,
                                          const int32_t* sel, int32_t n_sel,
                                          int32_t num_q_heads, int32_t chunk_len,
                                          int32_t chunk_start, float scale, void* o, void* o_lo,
                                          float* lse, float* reps, void* ws, size_t ws_bytes,
                                          void* stream) {
  OOMB_NVTX_RANGE("oomb_sparse_attn_fwd_own_reps");
  if (!reps) return fail(OOMB_ERR_INVALID_ARG, "reps must be set");
  if (!aligned(reps, 16)) return fail(OOMB_ERR_INVALID_ARG, "reps must be 16-byte aligned");
  return attn_fwd("oomb_sparse_attn_fwd_own_reps", q, kv, sel, n_sel, num_q_heads, chunk_len,
                  chunk_start, scale, o, o_lo, lse, reps, ws, ws_bytes, stream);
}

oomb_status oomb_sparse_attn_bwd(const void* q, const void* o, const void* o_lo,
                                 const void* dout, const float* lse, const oomb_paged_kv* kv,
                                 const int32_t* sel, int32_t n_sel, int32_t num_q_heads,
                                 int32_t chunk_len, int32_t chunk_start, float scale, void* dq,
                                 void* ws, size_t ws_bytes, void* stream) {
  OOMB_NVTX_RANGE("oomb_sparse_attn_bwd");
  oomb_status s = check_kv(kv);
  if (s != OOMB_OK) return s;
  s = check_chunk(kv, num_q_heads, chunk_len, chunk_start);
  if (s != OOMB_OK) return s;
  if (!kv->dk || !kv->dv) return fail(OOMB_ERR_INVALID_ARG, "kv->dk and kv->dv must be set");
  if (!q || !o || !dout || !lse || !dq)
    return fail(OOMB_ERR_INVALID_ARG, "q, o, dout, lse and dq must be set");
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(dout, 16) || !aligned(lse, 16) ||
      !aligned(dq, 16) || !aligned(o_lo, 16))
    return fail(OOMB_ERR_INVALID_ARG, "q, o, o_lo, dout, lse and dq must be 16-byte aligned");
  if (o_lo && kv->dtype != OOMB_BF16)
    return fail(OOMB_ERR_INVALID_ARG, "o_lo is for bf16 pools (an fp32 o needs no residual)");
  const int n_cand = chunk_start / kv->page_size;
  if (n_sel < 0 || n_sel > n_cand)
    return fail(OOMB_ERR_INVALID_ARG, "n_sel %d outside [0, %d] (pages before the chunk)", n_sel,
                n_cand);
  if (n_sel > 0 && !sel) return fail(OOMB_ERR_INVALID_ARG, "sel is NULL");
  s = check_ws(ws, ws_bytes,
               oomb_workspace_bytes(OOMB_OP_ATTN_BWD, kv, num_q_heads, chunk_len, 0));
  if (s != OOMB_OK) return s;
  const float sc = resolve_scale(scale, kv->head_dim);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (kv->dtype == OOMB_BF16) {
    e = check_tail_rows(kv, chunk_len, chunk_start, static_cast<int*>(ws), st);
    if (e == cudaSuccess)
      e = oomb::launch_attn_bwd_bf16(q, o, o_lo, dout, lse, desc(kv), sel, n_sel, num_q_heads,
                                     chunk_len, chunk_start, sc, dq, ws, g_wait_ns, st);
  } else
    e = oomb::launch_attn_bwd_fp32(static_cast<const float*>(q), static_cast<const float*>(o),
                                   static_cast<const float*>(dout), lse, desc(kv), sel, n_sel,
                                   num_q_heads, chunk_len, chunk_start, sc,
                                   static_cast<float*>(dq), ws, st);
  return e == cudaSuccess ? OOMB_OK : cuda_fail(e, "oomb_sparse_attn_bwd launch");
}

oomb_status oomb_debug_wait_unset_flag(void* ws, size_t ws_bytes, void* stream) {
  oomb_status s = check_ws(ws, ws_bytes, oomb::kStatusBytes);
  if (s != OOMB_OK) return s;
  cudaError_t e = oomb::launch_debug_wait(static_cast<int*>(ws), g_wait_ns,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? OOMB_OK : cuda_fail(e, "oomb_debug_wait_unset_flag launch");
}

}  // extern "C"
