// Steps 1 and 2 of the path (Page-level Sparse Attention item of the method):
// the representative vector of each page and the Top-K page selection.  Both
// are HBM-bound streams: 16-byte vector loads, many loads in flight per
// thread, every reduction in a fixed order so the selection is deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "oomb.h"
#include "oomb_internal.h"
#include "sm100.cuh"

namespace oomb {
namespace {

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ static void to_float(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};
template <>
struct Vec<float> {
  static constexpr int kElems = 4;
  __device__ static void to_float(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ---------------------------------------------------------------------------
// Step 1: reps[l][g][:] = mean over the P keys of page l, KV head g.
// One CTA of 256 threads per (page, KV head): 16 threads cover one 256-byte
// key row with 16-byte loads, 16 row groups stride over the page's rows.
// Rows are 256 bytes for both supported shapes (bf16 D=128, fp32 D=64).
// The last page of the range may hold keys in its first last_rows rows only
// (the partial last page of a sequence): its mean is over those rows.
// ---------------------------------------------------------------------------
template <typename T, int P>
__global__ void __launch_bounds__(256) page_reps_kernel(const T* __restrict__ k,
                                                        const int32_t* __restrict__ pt,
                                                        int first_page, int last_page,
                                                        int last_rows, int num_slots, int hkv,
                                                        float* __restrict__ reps, int* status) {
  constexpr int E = Vec<T>::kElems;
  constexpr int D = 16 * E;
  constexpr int RG = 16;                          // row groups
  constexpr int RPT = (P + RG - 1) / RG;          // rows per thread
  __shared__ float part[RG][D];
  const int item = blockIdx.x;
  const int l = first_page + item / hkv;
  const int g = item % hkv;
  const int slot = pt[l];
  if (slot < 0 || slot >= num_slots) {
    if (threadIdx.x == 0) raise_status(status, kStatusBounds, kWhereReps);
    return;
  }
  const int rows = l == last_page ? last_rows : P;
  const int col = threadIdx.x & 15, rg = threadIdx.x >> 4;
  const T* base = k + (static_cast<size_t>(slot) * hkv + g) * P * D + col * E;
  uint4 v[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg + RG * i;
    v[i] = (r < rows) ? ldg_stream(base + static_cast<size_t>(r) * D) : make_uint4(0, 0, 0, 0);
  }
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    float f[E];
    Vec<T>::to_float(v[i], f);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] += f[e];
  }
#pragma unroll
  for (int e = 0; e < E; ++e) part[rg][col * E + e] = acc[e];
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < RG; ++r) s += part[r][threadIdx.x];
    const float inv = rows == P ? 1.0f / P : 1.0f / static_cast<float>(rows);
    reps[(static_cast<size_t>(l) * hkv + g) * D + threadIdx.x] = s * inv;
  }
}

template <typename T>
cudaError_t reps_dispatch(const KvDesc& kv, int first_page, int n_pages, int last_rows,
                          float* reps, int* status, cudaStream_t st) {
  const dim3 grid(n_pages * kv.hkv);
  const T* k = static_cast<const T*>(kv.k);
  const int last_page = first_page + n_pages - 1;
#define OOMB_REPS_CASE(PS)                                                                  \
  case PS:                                                                                  \
    page_reps_kernel<T, PS><<<grid, 256, 0, st>>>(k, kv.page_table, first_page, last_page, \
                                                  last_rows, kv.num_slots, kv.hkv, reps,    \
                                                  status);                                  \
    break;
  switch (kv.page_size) {
    OOMB_REPS_CASE(16)
    OOMB_REPS_CASE(32)
    OOMB_REPS_CASE(64)
    OOMB_REPS_CASE(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef OOMB_REPS_CASE
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Step 2a: qbar[g][:] = mean of q over the chunk's tokens and the G heads of
// group g.  kQbarBlocks CTAs each sum a contiguous token slice (two token rows
// per step, 8 rows in flight per thread); the CTA then folds its heads into
// groups and writes a partial.  The last CTA to finish (ticket counter) sums
// the partials in a fixed tree: 7 sub-slices of consecutive partials per
// float4 column, then the 7 sub-sums in order.
// ---------------------------------------------------------------------------
constexpr int kQbarThreads = 896;
constexpr int kTailMax = 12;                      // partials per sub-slice of the tree

template <typename T>
__global__ void __launch_bounds__(kQbarThreads) qbar_kernel(const T* __restrict__ q, int chunk_len,
                                                            int hq, int hkv, int head_dim,
                                                            float* __restrict__ partials,
                                                            float* __restrict__ qbar,
                                                            int* status) {
  constexpr int E = Vec<T>::kElems;
  constexpr int U = 8;                            // token rows in flight per thread
  extern __shared__ float sm[];                   // [R][hq*head_dim], reused by the tree
  __shared__ int is_last;
  const int row_elems = hq * head_dim;
  const int row_vecs = row_elems / E;             // 16-byte vectors per token row
  const int R = blockDim.x / row_vecs;            // token rows per step (>= 1)
  const int nb = gridDim.x;
  const int t_per = (chunk_len + nb - 1) / nb;
  const int t0 = blockIdx.x * t_per;
  const int t1 = min(chunk_len, t0 + t_per);
  const int sub = threadIdx.x / row_vecs;
  const int col = threadIdx.x % row_vecs;
  if (sub < R) {
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    const T* base = q + static_cast<size_t>(col) * E;
    // rounds of U predicated loads, all in flight together (no serial remainder)
    for (int t = t0 + sub; t < t1; t += U * R) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        v[u] = (t + u * R < t1) ? ldg_stream(base + static_cast<size_t>(t + u * R) * row_elems)
                                : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[E];
        Vec<T>::to_float(v[u], f);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += f[e];
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) sm[sub * row_elems + col * E + e] = acc[e];
  }
  __syncthreads();
  const int grp = hq / hkv;
  for (int o = threadIdx.x; o < hkv * head_dim; o += blockDim.x) {
    const int g = o / head_dim, d = o % head_dim;
    float s = 0.f;
    for (int j = 0; j < grp; ++j) {
      const int idx = (g * grp + j) * head_dim + d;
      for (int r = 0; r < R; ++r) s += sm[r * row_elems + idx];
    }
    partials[static_cast<size_t>(blockIdx.x) * hkv * head_dim + o] = s;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int ticket = atomicAdd(&status[kTicketIdx], 1);
    is_last = (ticket == nb - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // Fixed-order tree over the nb partials.
  const int n_out4 = hkv * head_dim / 4;          // float4 columns
  const int n_sub = blockDim.x / n_out4 < 7 ? blockDim.x / n_out4 : 7;
  float4* red = reinterpret_cast<float4*>(sm);    // [n_sub][n_out4]
  if (threadIdx.x < n_sub * n_out4) {
    const int c4 = threadIdx.x % n_out4, s = threadIdx.x / n_out4;
    const int per = (nb + n_sub - 1) / n_sub;
    const int b0 = s * per, b1 = min(nb, b0 + per);
    const float4* p4 = reinterpret_cast<const float4*>(partials);
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = b0; base < b1; base += kTailMax) {   // kTailMax loads in flight
      float4 x[kTailMax];
#pragma unroll
      for (int u = 0; u < kTailMax; ++u)
        x[u] = (base + u < b1) ? __ldcg(p4 + static_cast<size_t>(base + u) * n_out4 + c4)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < kTailMax; ++u) {
        a.x += x[u].x; a.y += x[u].y; a.z += x[u].z; a.w += x[u].w;
      }
    }
    red[s * n_out4 + c4] = a;
  }
  __syncthreads();
  if (threadIdx.x < n_out4) {
    float4 a = red[threadIdx.x];
    for (int s = 1; s < n_sub; ++s) {
      const float4 x = red[s * n_out4 + threadIdx.x];
      a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
    }
    const float inv = 1.0f / (static_cast<float>(chunk_len) * grp);
    a.x *= inv; a.y *= inv; a.z *= inv; a.w *= inv;
    reinterpret_cast<float4*>(qbar)[threadIdx.x] = a;
  }
  if (threadIdx.x == 0) status[kTicketIdx] = 0;   // leave the counter at zero
}

// ---------------------------------------------------------------------------
// Step 2b: score[g][l] = qbar[g] . reps[l][g] for l < n_cand (else -inf).
// A group of D/4 lanes covers one 4*D-byte rep row with float4 loads; each
// warp keeps 4 row-steps in flight; shuffle reduction in a fixed pattern.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) page_scores_kernel(const float* __restrict__ reps,
                                                          const float* __restrict__ qbar,
                                                          int n_cand, int num_pages, int hkv,
                                                          float* __restrict__ scores) {
  constexpr int L = D / 4;                        // lanes per row
  constexpr int RPW = 32 / L;                     // rows per warp-step
  constexpr int U = 8;
  __shared__ float4 qs[16 * L];                   // hkv <= 16
  for (int i = threadIdx.x; i < hkv * L; i += blockDim.x)
    qs[i] = reinterpret_cast<const float4*>(qbar)[i];
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int sub = lane / L, li = lane % L;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  const int wid = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  // rows = (page, KV head) pairs; below 2^31 for every supported pool
  const int rows = num_pages * hkv;
  const int cand_rows = n_cand * hkv;
  for (int r0 = wid * RPW * U; r0 < rows; r0 += warps_total * RPW * U) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = r0 + u * RPW + sub;
      v[u] = (r < cand_rows) ? __ldcs(reinterpret_cast<const float4*>(reps) + static_cast<long>(r) * L + li)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = r0 + u * RPW + sub;
      const int g = r % hkv;
      const float4 qv = qs[g * L + li];
      float s = v[u].x * qv.x;
      s = fmaf(v[u].y, qv.y, s);
      s = fmaf(v[u].z, qv.z, s);
      s = fmaf(v[u].w, qv.w, s);
#pragma unroll
      for (int off = L / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (li == 0 && r < rows) {
        const int l = r / hkv;
        scores[static_cast<long>(g) * num_pages + l] = (r < cand_rows) ? s : -INFINITY;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Step 2c: per KV head, keep the top_k best scores (ties -> lower page),
// written in ascending page order.  One CTA of 1024 threads per KV head.
// Radix select on order-preserving 32-bit keys (11 + 11 + 10 bits) finds the
// k-th key T; then every key > T is kept plus the lowest-indexed keys == T
// until k are kept.  Compaction runs in index order, so the output is sorted.
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 1024;
constexpr int kTopkSmemKeys = 48 * 1024;          // keys cached in shared memory
constexpr int kTopkCand = 2048;                   // keys of one value bin resolved exactly

__device__ __forceinline__ uint32_t order_key(float f) {
  if (f != f) return 0u;                          // NaN never outranks a number
  if (f == 0.f) f = 0.f;                          // -0 == +0
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The float a key stands for (inverse of order_key on numbers).
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 1024).
__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;                           // inclusive
    if (lane == 31) *total = t;
  }
  __syncthreads();
  const int before = (w == 0 ? 0 : warp_tot[w - 1]) + x - v;
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores,
                                                            int num_pages, int n_cand, int top_k,
                                                            int32_t* __restrict__ sel) {
  extern __shared__ uint32_t keys_sm[];           // n_cand keys when they fit
  __shared__ int hist[2048];
  __shared__ int warp_tot[32];
  __shared__ int total;
  __shared__ uint32_t sh_prefix, sh_min, sh_max;
  __shared__ int sh_need;
  const int g = blockIdx.x;
  const float* sc = scores + static_cast<long>(g) * num_pages;
  const int k = top_k < n_cand ? top_k : n_cand;  // n_sel: row stride of sel
  int32_t* out = sel + static_cast<long>(g) * k;
  if (k == n_cand) {                              // every candidate is kept
    for (int i = threadIdx.x; i < n_cand; i += blockDim.x) out[i] = i;
    return;
  }
  const bool cached = n_cand <= kTopkSmemKeys;
  if (threadIdx.x == 0) {
    sh_min = 0xFFFFFFFFu;
    sh_max = 0u;
  }
  __syncthreads();
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
  constexpr int kU = 8;                           // loads in flight per thread
  for (int base = threadIdx.x; base < n_cand; base += kU * blockDim.x) {
    float v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = base + u * blockDim.x;
      v[u] = i < n_cand ? __ldcg(sc + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = base + u * blockDim.x;
      if (i < n_cand) {
        const uint32_t key = order_key(v[u]);
        if (cached) keys_sm[i] = key;
        kmin = min(kmin, key);
        kmax = max(kmax, key);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if ((threadIdx.x & 31) == 0) {
    atomicMin(&sh_min, kmin);
    atomicMax(&sh_max, kmax);
  }
  __syncthreads();
  auto key_at = [&](int i) -> uint32_t { return cached ? keys_sm[i] : order_key(__ldcg(sc + i)); };

  // Fast path: a histogram of the score values in 2048 equal-width bins
  // between the smallest and the largest score.  The scores of a head sit in
  // a narrow range of either sign, where the bits of their encodings put
  // most keys in a few radix bins; equal-width value bins spread them.  The
  // bin is monotone in the score, so every key of a higher bin ranks above
  // every key of a lower one, and the k-th largest key is found exactly among
  // the keys of its own bin (ranked by counting).  Degenerate ranges, or a bin
  // with more than kTopkCand keys, take the radix passes below.
  __shared__ uint32_t cand[kTopkCand];
  __shared__ int sh_nc, sh_bin;
  uint32_t prefix = 0;
  int need = k;                                   // still to take at or below `prefix`
  bool fast = false;
  {
    const float fmin = key_value(sh_min), fmax = key_value(sh_max);
    const float inv_w = 2048.f / (fmax - fmin);
    if (fmax > fmin && isfinite(fmin) && isfinite(fmax) && isfinite(inv_w)) {
      auto vbin = [&](uint32_t key) -> int {
        const int b = static_cast<int>((key_value(key) - fmin) * inv_w);
        return b < 2047 ? b : 2047;
      };
      for (int i = threadIdx.x; i < 2048; i += blockDim.x) hist[i] = 0;
      if (threadIdx.x == 0) sh_nc = 0;
      __syncthreads();
      for (int i = threadIdx.x; i < n_cand; i += blockDim.x) atomicAdd(&hist[vbin(key_at(i))], 1);
      __syncthreads();
      // bin counts from the top: thread t owns bins 2047 - 2t and 2046 - 2t
      const int b_hi = 2047 - 2 * static_cast<int>(threadIdx.x);
      const int c0 = hist[b_hi], c1 = hist[b_hi - 1];
      const int before = block_excl_scan(c0 + c1, warp_tot, &total);
      if (before < k && before + c0 >= k) {
        sh_bin = b_hi;
        sh_need = k - before;
      } else if (before + c0 < k && before + c0 + c1 >= k) {
        sh_bin = b_hi - 1;
        sh_need = k - before - c0;
      }
      __syncthreads();
      const int bin = sh_bin, need_b = sh_need, c_b = hist[bin];
      if (c_b <= kTopkCand) {
        for (int i = threadIdx.x; i < n_cand; i += blockDim.x) {
          const uint32_t key = key_at(i);
          if (vbin(key) == bin) cand[atomicAdd(&sh_nc, 1)] = key;
        }
        __syncthreads();
        // the need_b-th largest key of the bin: gt keys above it, eq equal to it
        for (int c = threadIdx.x; c < c_b; c += blockDim.x) {
          const uint32_t x = cand[c];
          int gt = 0, eq = 0;
          for (int u = 0; u < c_b; ++u) {
            gt += cand[u] > x;
            eq += cand[u] == x;
          }
          if (gt < need_b && need_b <= gt + eq) {  // every writer writes the same values
            sh_prefix = x;
            sh_nc = need_b - gt;
          }
        }
        __syncthreads();
        prefix = sh_prefix;
        need = sh_nc;
        fast = true;
      }
      __syncthreads();
    }
  }
  // Radix passes: every key shares the bits above the highest bit where min
  // and max differ, so the digits start just below that common prefix.
  const uint32_t diff = sh_min ^ sh_max;
  int lo_bit = (fast || !diff) ? 0 : 32 - __clz(diff);   // bits [0, lo_bit) still vary
  if (!fast) {
    const uint32_t low = (lo_bit >= 32) ? 0xFFFFFFFFu : ((1u << lo_bit) - 1u);
    prefix = sh_max & ~low;                       // the common high bits
  }
  uint32_t mask = (lo_bit >= 32) ? 0u : ~((1u << lo_bit) - 1u);
  while (lo_bit > 0) {
    const int width = lo_bit < 11 ? lo_bit : 11;
    const int sh = lo_bit - width, nbins = 1 << width;
    for (int i = threadIdx.x; i < nbins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n_cand; i += blockDim.x) {
      const uint32_t key = key_at(i);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & (nbins - 1)], 1);
    }
    __syncthreads();
    // Bin counts from the top: thread t owns bins [2t, 2t+1] of the reversed order.
    const int b_hi = nbins - 1 - 2 * static_cast<int>(threadIdx.x);
    const int c0 = (2 * static_cast<int>(threadIdx.x) < nbins) ? hist[b_hi] : 0;
    const int c1 = (2 * static_cast<int>(threadIdx.x) + 1 < nbins) ? hist[b_hi - 1] : 0;
    const int before = block_excl_scan(c0 + c1, warp_tot, &total);
    // the bin where the running count from the top first reaches `need`
    if (2 * static_cast<int>(threadIdx.x) < nbins) {
      if (before < need && before + c0 >= need) {
        sh_prefix = prefix | (static_cast<uint32_t>(b_hi) << sh);
        sh_need = need - before;
      } else if (2 * static_cast<int>(threadIdx.x) + 1 < nbins && before + c0 < need &&
                 before + c0 + c1 >= need) {
        sh_prefix = prefix | (static_cast<uint32_t>(b_hi - 1) << sh);
        sh_need = need - before - c0;
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    need = sh_need;
    mask |= static_cast<uint32_t>(nbins - 1) << sh;
    lo_bit = sh;
    __syncthreads();
  }
  // prefix == T (the k-th key), need == how many keys equal to T are kept.
  // Index-ordered compaction: warp w owns the contiguous index range
  // [w * span, (w + 1) * span) and walks it 32 consecutive indices at a time
  // (lane = index within the step: conflict-free shared loads), so ballots
  // give each key's rank in index order.
  const uint32_t T = prefix;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  const int span = ((n_cand + nw - 1) / nw + 31) & ~31;
  const int j0 = w * span, j1 = min(n_cand, j0 + span);
  const uint32_t below = (1u << lane) - 1u;
  int n_eq = 0;
  for (int base = j0; base < j1; base += 32) {
    const int i = base + lane;
    n_eq += __popc(__ballot_sync(0xffffffffu, i < j1 && key_at(i) == T));
  }
  // exclusive scan over warps of the equal-key counts, then of the kept counts
  __shared__ int wsum[32];
  if (lane == 0) wsum[w] = n_eq;
  __syncthreads();
  int eq_before = 0;
  for (int u = 0; u < w; ++u) eq_before += wsum[u];
  __syncthreads();
  int n_keep = 0, eq_rank = eq_before;
  for (int base = j0; base < j1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < j1 ? key_at(i) : 0u;
    const uint32_t eqm = __ballot_sync(0xffffffffu, i < j1 && key == T);
    const bool keep = i < j1 && (key > T || (key == T && eq_rank + __popc(eqm & below) < need));
    n_keep += __popc(__ballot_sync(0xffffffffu, keep));
    eq_rank += __popc(eqm);
  }
  if (lane == 0) wsum[w] = n_keep;
  __syncthreads();
  int pos = 0;
  for (int u = 0; u < w; ++u) pos += wsum[u];
  eq_rank = eq_before;
  for (int base = j0; base < j1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < j1 ? key_at(i) : 0u;
    const uint32_t eqm = __ballot_sync(0xffffffffu, i < j1 && key == T);
    const bool keep = i < j1 && (key > T || (key == T && eq_rank + __popc(eqm & below) < need));
    const uint32_t km = __ballot_sync(0xffffffffu, keep);
    if (keep) out[pos + __popc(km & below)] = i;
    pos += __popc(km);
    eq_rank += __popc(eqm);
  }
}

// ---------------------------------------------------------------------------
// Page-table check: every entry in range, no slot used twice.
// ---------------------------------------------------------------------------
__global__ void validate_pt_kernel(const int32_t* __restrict__ pt, int num_pages, int num_slots,
                                   uint32_t* bitmap, int* status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= num_pages) return;
  const int s = pt[i];
  if (s < 0 || s >= num_slots) {
    raise_status(status, kStatusBounds, 1);
    return;
  }
  const uint32_t bit = 1u << (s & 31);
  if (atomicOr(&bitmap[s >> 5], bit) & bit) raise_status(status, kStatusBounds, 2);
}

// A wait on an mbarrier nothing arrives on: exercises the bounded-wait path.
__global__ void debug_wait_kernel(int* status, uint64_t limit_ns) {
  __shared__ alignas(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    WaitCtl wc{status, &abort_flag, limit_ns};
    mbar_wait(smem_u32(&bar), 0, wc, kWhereDebug);
  }
}

}  // namespace

cudaError_t launch_page_reps(const KvDesc& kv, bool bf16, int first_page, int n_pages,
                             int last_rows, float* reps, int* status, cudaStream_t st) {
  if (n_pages == 0) return cudaSuccess;
  if (last_rows < 1 || last_rows > kv.page_size) return cudaErrorInvalidValue;
  return bf16 ? reps_dispatch<__nv_bfloat16>(kv, first_page, n_pages, last_rows, reps, status, st)
              : reps_dispatch<float>(kv, first_page, n_pages, last_rows, reps, status, st);
}

size_t select_ws_bytes(int num_pages, int hkv, int head_dim) {
  size_t b = kStatusBytes;
  b += align_up(static_cast<size_t>(kQbarBlocks) * hkv * head_dim * 4, 256);  // partials
  b += align_up(static_cast<size_t>(hkv) * head_dim * 4, 256);                // qbar
  b += align_up(static_cast<size_t>(hkv) * num_pages * 4, 256);              // scores
  return b;
}

cudaError_t launch_select_topk(const void* q, bool bf16, int hq, int chunk_len, int n_cand,
                               const float* reps, int num_pages, int hkv, int head_dim, int top_k,
                               int32_t* sel, float* scores_opt, void* ws, cudaStream_t st) {
  char* w = static_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(w);
  float* partials = reinterpret_cast<float*>(w + kStatusBytes);
  float* qbar = reinterpret_cast<float*>(
      w + kStatusBytes + align_up(static_cast<size_t>(kQbarBlocks) * hkv * head_dim * 4, 256));
  float* scores = scores_opt ? scores_opt
                             : reinterpret_cast<float*>(reinterpret_cast<char*>(qbar) +
                                                        align_up(static_cast<size_t>(hkv) *
                                                                     head_dim * 4, 256));
  // R token rows per step of hq*head_dim floats each, or the tree's 7 x hkv*head_dim
  const size_t row_vecs = static_cast<size_t>(hq) * head_dim / (bf16 ? 8 : 4);
  const size_t rows = kQbarThreads / row_vecs;
  const size_t a = rows * hq * head_dim, b = 7 * static_cast<size_t>(hkv) * head_dim;
  const size_t qsm = sizeof(float) * (a > b ? a : b);
  if (bf16)
    qbar_kernel<__nv_bfloat16><<<kQbarBlocks, kQbarThreads, qsm, st>>>(
        static_cast<const __nv_bfloat16*>(q), chunk_len, hq, hkv, head_dim, partials, qbar,
        status);
  else
    qbar_kernel<float><<<kQbarBlocks, kQbarThreads, qsm, st>>>(
        static_cast<const float*>(q), chunk_len, hq, hkv, head_dim, partials, qbar, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int blocks = 152 * 8;
  if (head_dim == 128)
    page_scores_kernel<128><<<blocks, 256, 0, st>>>(reps, qbar, n_cand, num_pages, hkv, scores);
  else
    page_scores_kernel<64><<<blocks, 256, 0, st>>>(reps, qbar, n_cand, num_pages, hkv, scores);
  e = cudaGetLastError();
  if (e != cudaSuccess || top_k == 0 || n_cand == 0) return e;
  const size_t ksm = n_cand <= kTopkSmemKeys ? static_cast<size_t>(n_cand) * 4 : 0;
  static PerDeviceOnce attr;
  e = once_per_device(attr, [] {
    return cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kTopkSmemKeys * 4);
  });
  if (e != cudaSuccess) return e;
  topk_kernel<<<hkv, kTopkThreads, ksm, st>>>(scores, num_pages, n_cand, top_k, sel);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Selection without a caller workspace: the scratch is this file-scope device
// array.  Host code may not pass the symbol itself to a kernel (on the host it
// names a host-side stand-in), so its device address is looked up once per
// device, with that device current, and cached.
// ---------------------------------------------------------------------------
namespace {
__device__ __align__(256) unsigned char g_select_scratch[OOMB_NOALLOC_SCRATCH_BYTES];
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

cudaError_t select_scratch_addr(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_select_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_select_topk_noalloc(const void* q, bool bf16, int hq, int chunk_len,
                                       int n_cand, const float* reps, int num_pages, int hkv,
                                       int head_dim, int top_k, int32_t* sel, float* scores_opt,
                                       bool* too_big, cudaStream_t st) {
  *too_big = select_ws_bytes(num_pages, hkv, head_dim) > OOMB_NOALLOC_SCRATCH_BYTES;
  if (*too_big) return cudaSuccess;
  void* scratch = nullptr;
  cudaError_t e = select_scratch_addr(&scratch);
  if (e != cudaSuccess) return e;
  // the status block (with the query-summary ticket counter) must start at zero
  e = cudaMemsetAsync(scratch, 0, kStatusBytes, st);
  if (e != cudaSuccess) return e;
  return launch_select_topk(q, bf16, hq, chunk_len, n_cand, reps, num_pages, hkv, head_dim,
                            top_k, sel, scores_opt, scratch, st);
}

cudaError_t launch_validate_page_table(const int32_t* pt, int num_pages, int num_slots,
                                       uint32_t* bitmap, int* status, cudaStream_t st) {
  if (num_pages == 0) return cudaSuccess;
  validate_pt_kernel<<<(num_pages + 255) / 256, 256, 0, st>>>(pt, num_pages, num_slots, bitmap,
                                                              status);
  return cudaGetLastError();
}

cudaError_t launch_debug_wait(int* status, uint64_t limit_ns, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace oomb
