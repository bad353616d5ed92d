// Steps 1 and 2 of the path (Page-level Sparse Attention item of the method):
// the representative vector of each page and the Top-K page selection.  Both
// are HBM-bound streams: 16-byte vector loads, many loads in flight per
// thread, every reduction in a fixed order so the selection is deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cooperative_groups.h>

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

// L2 policy for data read exactly once: its lines are the first to be replaced,
// so a stream does not push out lines that are still wanted (the
// representatives just written, the scores) and mostly replaces its own lines
// instead of writing dirty ones back while it streams.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(l2_evict_first()));
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
// Copies of 16 bytes global -> shared that stay in flight without holding
// registers; each thread waits only for its own (commit groups), so a thread
// that reads back exactly the slots it filled needs no barrier.  The query
// rows and the representatives are read once per call: evict-first in L2.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(
                   smem_u32(smem_dst)),
               "l"(gsrc), "l"(l2_evict_first())
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// ---------------------------------------------------------------------------
// Step 2: the Top-K page selection as one cooperative kernel, one CTA per SM
// (every CTA resident at once, so the CTAs can wait for one another: each
// such wait is bounded and records OOMB_ERR_TIMEOUT if it runs out).
//
//  2a  qbar[g][:] = mean of q over the chunk's tokens and the G heads of
//      group g.  Each CTA streams a contiguous slice of token rows: a thread
//      owns one 16-byte column of a row (R rows side by side per step) and
//      keeps kSelDepth row copies in flight through shared memory.  The CTA
//      folds its rows and the heads of each group into a partial; partials
//      are added in two levels, each by whichever CTA finishes last (ticket
//      counters): the last CTA of each group of kSelGroup consecutive CTAs
//      adds the group's partials in CTA order, the last group adds the group
//      sums in group order and publishes qbar (a generation counter).  Every
//      sum runs in a fixed order: the result does not depend on timing.
//  2b  score[g][l] = qbar[g] . reps[l][g] for l < n_cand (else -inf).  A
//      group of D/4 lanes covers one (page, KV head) row, one 16-byte column
//      per lane, with kSelDepth rows in flight; a CTA issues its first row
//      copies before it waits for qbar (the representatives do not depend on
//      it).  Products are summed by a fixed shuffle pattern.  Each score is
//      also counted in a per-head histogram of the top 16 bits of its
//      order-preserving key: the first digit of the radix select below.
//  2c  Once every CTA has counted its scores (an arrival counter), CTA g <
//      Hkv keeps the top_k best scores of KV head g (ties -> lower page),
//      written in ascending page order.  The first digit's bin where the
//      count from the top reaches k comes from the histogram (coalesced warp
//      sums, then the warp holding the bin narrows it down).  Fast path: the
//      keys at or above that bin (k plus the bin's few) go with their indices
//      into shared memory, and the k largest by (key, then lower index) are
//      written in index order -- ranked by counting when there are at most
//      kSelRankMax of them, else sorted.  When more than kSelSortMax keys
//      share the bins (many equal scores), two 8-bit digits from
//      shared-memory histograms of the keys that share the digits found so
//      far give the k-th largest key T and how many keys equal to T are kept
//      (the lowest-indexed ones); an index-ordered compaction writes every
//      key above T and those ties.
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 1024;
constexpr int kSelDepth = 8;                      // 16-byte copies in flight per thread
constexpr int kSelGroup = 8;                      // CTAs per first-level group
constexpr int kSelMaxBlocks = 256;
constexpr int kSelCacheKeys = 40 * 1024;          // keys cached for the radix passes
constexpr int kSelSortMax = 4096;                 // keys sorted on the fast path
constexpr int kSelRankMax = 256;                  // keys ranked by counting instead
constexpr size_t kSelRingBytes = sizeof(uint4) * kSelDepth * kSelThreads;
constexpr size_t kSelCacheBytes =
    kSelRingBytes > 4 * kSelCacheKeys ? kSelRingBytes : 4 * static_cast<size_t>(kSelCacheKeys);
constexpr size_t kSelListBytes = 8 * 4096 + 4 * 4096;   // the fast path's sort buffers
constexpr size_t kSelDynSmem = kSelCacheBytes + kSelListBytes;
static_assert(kSelRingBytes + sizeof(float4) * kSelThreads <= kSelDynSmem,
              "the query summary's partial sums fit past the copy ring");
static_assert(kGroupTicketIdx + (kSelMaxBlocks + kSelGroup - 1) / kSelGroup <= 64,
              "tickets fit the status block");

// Bring `bytes` (a multiple of 16) at `p` into L2, without waiting.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// In-place bitonic sort of n (a power of two) values in shared memory by the
// whole block: descending if `desc`, else ascending.
template <typename V>
__device__ __forceinline__ void block_bitonic_sort(V* a, int n, bool desc) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < (n >> 1); t += blockDim.x) {
        const int i = 2 * t - (t & (stride - 1));
        const int j = i + stride;
        const bool d = ((i & size) == 0) == desc;
        const V x = a[i], y = a[j];
        if ((x < y) == d) {
          a[i] = y;
          a[j] = x;
        }
      }
      __syncthreads();
    }
  }
}

// Where bin b of a head's 65536-bin key histogram is stored: within each
// window of 2048 bins, bin (hi, lo) = (b >> 6 & 31, b & 63) sits at lo * 32 +
// hi, so neighbouring bins (which a narrow score distribution fills most)
// fall in different 128-byte lines and their atomics do not queue on one line.
__device__ __forceinline__ int hist_slot(uint32_t b) {
  return static_cast<int>((b & ~2047u) | ((b & 63u) << 5) | ((b >> 6) & 31u));
}

__device__ __forceinline__ uint32_t order_key(float f) {
  if (f != f) return 0u;                          // NaN never outranks a number
  if (f == 0.f) f = 0.f;                          // -0 == +0
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
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

// Thread 0 waits until `*word - base` (unsigned) reaches `target`, for at
// most limit_ns; returns false (and records a timeout) if it does not.
__device__ __forceinline__ bool wait_counter(const int* word, uint32_t base, uint32_t target,
                                             int* status, uint64_t limit_ns, int where) {
  const uint64_t t0 = global_timer_ns();
  while (static_cast<uint32_t>(*reinterpret_cast<const volatile int*>(word)) - base < target) {
    if (global_timer_ns() - t0 > limit_ns) {
      raise_status(status, kStatusTimeout, where);
      return false;
    }
    __nanosleep(64);
  }
  __threadfence();                                // acquire: what was published before it
  return true;
}

struct SelParams {
  const void* q;
  const float* reps;
  float* scores;                  // [hkv][num_pages]
  int32_t* sel;                   // [hkv][n_sel]
  float* partials;                // [kSelMaxBlocks][hkv * D]
  float* gsums;                   // [groups][hkv * D]
  float* qbar;                    // [hkv * D]
  int* hist;                      // [hkv][65536]
  int* status;
  int chunk_len, hq, hkv, n_cand, num_pages, top_k;
  uint64_t wait_ns;
};

template <typename T, int D>
__global__ void __launch_bounds__(kSelThreads, 1) select_kernel(const SelParams p) {
  constexpr int E = Vec<T>::kElems;
  constexpr int L = D / 4;                        // lanes per (page, head) row
  constexpr int RPW = 32 / L;                     // rows per warp step
  extern __shared__ __align__(16) uint4 ring[];   // copies in flight; the fold; the key cache
  __shared__ float4 qs[16 * L];                   // qbar (hkv <= 16)
  __shared__ int hist[256];
  __shared__ int warp_tot[32];
  __shared__ int total;
  __shared__ int flag;
  __shared__ uint32_t base_q, base_s, sh_digit;
  __shared__ int sh_need;
  const int tid = threadIdx.x, nt = kSelThreads;
  const int nb = gridDim.x, bid = blockIdx.x;
  int* status = p.status;
  if (tid == 0) {
    // generation counters as they stand: nothing changes them before every
    // CTA of this grid has finished its query slice
    base_q = static_cast<uint32_t>(*reinterpret_cast<volatile int*>(&status[kSelQbarGenIdx]));
    base_s = static_cast<uint32_t>(*reinterpret_cast<volatile int*>(&status[kSelScoreCntIdx]));
  }
  // the key histogram starts at zero (counted into only after qbar exists,
  // i.e. after every CTA has passed this point)
  const long hist_words = static_cast<long>(p.hkv) << 16;
  for (long i = static_cast<long>(bid) * nt + tid; i < hist_words; i += static_cast<long>(nb) * nt)
    p.hist[i] = 0;

  // ---------------------------------------------------------------- 2a
  const int hq = p.hq, hkv = p.hkv;
  const int row_elems = hq * D;
  const int row_vecs = row_elems / E;             // 16-byte vectors per token row
  const int R = 896 / row_vecs;                   // token rows per step (>= 1)
  const int t_per = (p.chunk_len + nb - 1) / nb;
  const int t0 = min(p.chunk_len, bid * t_per);
  const int t1 = min(p.chunk_len, t0 + t_per);
  const int sub = tid / row_vecs, col = tid % row_vecs;
  {
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    if (sub < R) {
      const T* base = static_cast<const T*>(p.q) + static_cast<size_t>(col) * E;
      const int n_j = t1 > t0 + sub ? (t1 - t0 - sub + R - 1) / R : 0;
      auto row = [&](int j) { return base + static_cast<size_t>(t0 + sub + j * R) * row_elems; };
#pragma unroll
      for (int j = 0; j < kSelDepth; ++j) {
        if (j < n_j) cp_async16(&ring[j * nt + tid], row(j));
        cp_async_commit();
      }
      for (int j = 0; j < n_j; ++j) {
        cp_async_wait<kSelDepth - 1>();           // row j has landed
        uint4* slot = &ring[(j % kSelDepth) * nt + tid];
        const uint4 v = *slot;
        if (j + kSelDepth < n_j) cp_async16(slot, row(j + kSelDepth));
        cp_async_commit();
        float f[E];
        Vec<T>::to_float(v, f);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += f[e];
      }
    }
    cp_async_wait<0>();
    if (tid == 0) {
      // this CTA's representative rows (2b), into L2 while the query summary
      // is folded and waited for: the loads of 2b then mostly hit L2
      const int cand_rows0 = p.n_cand * p.hkv;
      const int r_per0 = (cand_rows0 + nb - 1) / nb;
      const int a0 = min(cand_rows0, bid * r_per0), a1 = min(cand_rows0, a0 + r_per0);
      const char* base = reinterpret_cast<const char*>(p.reps) + static_cast<size_t>(a0) * D * 4;
      const size_t bytes = static_cast<size_t>(a1 - a0) * D * 4;
      for (size_t off = 0; off < bytes; off += 65536)
        prefetch_l2(base + off, static_cast<uint32_t>(bytes - off < 65536 ? bytes - off : 65536));
    }
    __syncthreads();                              // the ring becomes the fold area
    float* sm = reinterpret_cast<float*>(ring);   // [R][row_elems]
    if (sub < R) {                                // 16-byte stores: no bank conflicts
      float4* dst = reinterpret_cast<float4*>(sm + sub * row_elems + col * E);
#pragma unroll
      for (int e = 0; e < E; e += 4) dst[e / 4] = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
    }
    __syncthreads();
  }
  const int grp = hq / hkv;
  const int n_out = hkv * D;
  {
    const float* sm = reinterpret_cast<const float*>(ring);
    for (int o = tid; o < n_out; o += nt) {
      const int g = o / D, d = o % D;
      float s = 0.f;
      for (int j = 0; j < grp; ++j) {
        const int idx = (g * grp + j) * D + d;
        for (int r = 0; r < R; ++r) s += sm[r * row_elems + idx];
      }
      p.partials[static_cast<size_t>(bid) * n_out + o] = s;
    }
  }
  const int n_groups = (nb + kSelGroup - 1) / kSelGroup;
  const int group = bid / kSelGroup;
  const int in_group = min(kSelGroup, nb - group * kSelGroup);
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    flag = atomicAdd(&status[kGroupTicketIdx + group], 1) == in_group - 1;
  }
  __syncthreads();
  if (flag) {                                     // last of its group
    __threadfence();
    for (int o = tid; o < n_out; o += nt) {
      float s = 0.f;
      for (int c = 0; c < in_group; ++c)
        s += __ldcg(p.partials + static_cast<size_t>(group * kSelGroup + c) * n_out + o);
      p.gsums[static_cast<size_t>(group) * n_out + o] = s;
    }
    __syncthreads();
    if (tid == 0) {
      status[kGroupTicketIdx + group] = 0;        // leave the counter at zero
      __threadfence();
      atomicAdd(&status[kSelQbarGenIdx], 1);      // one more group summed
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- 2b
  // rows = (page, KV head) pairs of the candidates; this CTA's contiguous
  // range, walked by its warps in steps of RPW rows; kSelDepth rows per lane
  // in flight, the first ones requested before qbar exists
  const int cand_rows = p.n_cand * hkv;
  const int r_per = (cand_rows + nb - 1) / nb;
  const int rb0 = min(cand_rows, bid * r_per), rb1 = min(cand_rows, rb0 + r_per);
  const int lane = tid & 31, w = tid >> 5;
  const int rsub = lane / L, li = lane % L;
  const int stride = (nt / 32) * RPW;
  const int r0 = rb0 + w * RPW + rsub;            // this lane's first row
  const int n_j = r0 < rb1 ? (rb1 - r0 + stride - 1) / stride : 0;
  const int w0 = rb0 + w * RPW;                   // the warp steps together
  const int n_w = w0 < rb1 ? (rb1 - w0 + stride - 1) / stride : 0;
  const float4* src = reinterpret_cast<const float4*>(p.reps) + li;
#pragma unroll
  for (int j = 0; j < kSelDepth; ++j) {
    if (j < n_j) cp_async16(&ring[j * nt + tid], src + static_cast<long>(r0 + j * stride) * L);
    cp_async_commit();
  }
  if (tid == 0)
    flag = wait_counter(&status[kSelQbarGenIdx], base_q, static_cast<uint32_t>(n_groups), status,
                        p.wait_ns, kWhereSelect);
  __syncthreads();
  if (!flag) {
    cp_async_wait<0>();
    return;
  }
  // qbar from the group sums, added the same way in every CTA: thread
  // (s, i) adds the groups s, s + S, ... of column i in that order (all its
  // loads in flight at once), then the S partial sums of a column are added
  // in slice order (shared memory past the copies still in flight)
  {
    const float inv = 1.0f / (static_cast<float>(p.chunk_len) * grp);
    const float4* gs4 = reinterpret_cast<const float4*>(p.gsums);
    const int cols = hkv * L;                     // <= 16 * 32
    const int S = nt / cols;                      // >= 2
    float4* qpart = reinterpret_cast<float4*>(reinterpret_cast<char*>(ring) + kSelRingBytes);
    const int i = tid % cols, sl = tid / cols;
    if (sl < S) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c = sl; c < n_groups; c += S) {
        const float4 v = __ldcg(gs4 + static_cast<size_t>(c) * (n_out / 4) + i);
        a.x += v.x;
        a.y += v.y;
        a.z += v.z;
        a.w += v.w;
      }
      qpart[sl * cols + i] = a;
    }
    __syncthreads();
    if (tid < cols) {
      float4 a = qpart[tid];
      for (int u = 1; u < S; ++u) {
        const float4 v = qpart[u * cols + tid];
        a.x += v.x;
        a.y += v.y;
        a.z += v.z;
        a.w += v.w;
      }
      qs[tid] = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
    }
  }
  __syncthreads();
  for (int j = 0; j < n_w; ++j) {
    cp_async_wait<kSelDepth - 1>();
    const bool valid = j < n_j;
    uint4* slot = &ring[(j % kSelDepth) * nt + tid];
    const uint4 raw = valid ? *slot : make_uint4(0, 0, 0, 0);
    const int r = r0 + j * stride;
    if (j + kSelDepth < n_j) cp_async16(slot, src + static_cast<long>(r + kSelDepth * stride) * L);
    cp_async_commit();
    const int g = r % hkv;
    const float4 qv = qs[g * L + li];
    float sc = __uint_as_float(raw.x) * qv.x;
    sc = fmaf(__uint_as_float(raw.y), qv.y, sc);
    sc = fmaf(__uint_as_float(raw.z), qv.z, sc);
    sc = fmaf(__uint_as_float(raw.w), qv.w, sc);
    // lanes of one row reduce among themselves (the row's L lanes are aligned)
#pragma unroll
    for (int off = L / 2; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
    if (valid && li == 0) {
      p.scores[static_cast<long>(g) * p.num_pages + r / hkv] = sc;
      atomicAdd(&p.hist[(static_cast<long>(g) << 16) + hist_slot(order_key(sc) >> 16)], 1);
    }
  }
  cp_async_wait<0>();
  __syncthreads();                                // the ring is free again
  // pages that are not candidates
  const int n_other = (p.num_pages - p.n_cand) * hkv;
  for (int i = bid * nt + tid; i < n_other; i += nb * nt) {
    const int g = i % hkv, l = p.n_cand + i / hkv;
    p.scores[static_cast<long>(g) * p.num_pages + l] = -INFINITY;
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    atomicAdd(&status[kSelScoreCntIdx], 1);       // this CTA's scores are counted
  }
  if (bid >= hkv || p.top_k == 0 || p.n_cand == 0) return;

  // ---------------------------------------------------------------- 2c
  const int g = bid;
  const float* sc = p.scores + static_cast<long>(g) * p.num_pages;
  const int n_cand = p.n_cand;
  const int k = p.top_k < n_cand ? p.top_k : n_cand;   // n_sel: row stride of sel
  int32_t* out = p.sel + static_cast<long>(g) * k;
  if (k == n_cand) {                              // every candidate is kept
    for (int i = tid; i < n_cand; i += nt) out[i] = i;
    return;
  }
  if (tid == 0)
    flag = wait_counter(&status[kSelScoreCntIdx], base_s, static_cast<uint32_t>(nb), status,
                        p.wait_ns, kWhereSelect);
  __syncthreads();
  if (!flag) return;
  uint32_t* keys_sm = reinterpret_cast<uint32_t*>(ring);
  const bool cached = n_cand <= kSelCacheKeys;
  // digit 1: the 16-bit bin where the count from the top reaches k.  Warp w
  // owns bins [2048 w, 2048 w + 2048) and reads them coalesced; the warp
  // holding the bin then narrows it down to a lane's 64 bins, then to the bin.
  __shared__ int wcount[32];
  __shared__ int sh_above;
  {
    const int* hg = p.hist + (static_cast<long>(g) << 16);
    const int4* h4 = reinterpret_cast<const int4*>(hg + 2048 * w);
    int cw = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int4 v = __ldcg(h4 + 32 * j + lane);
      cw += (v.x + v.y) + (v.z + v.w);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cw += __shfl_xor_sync(0xffffffffu, cw, o);
    if (lane == 0) wcount[w] = cw;
    __syncthreads();
    if (w == 0) {                                 // from the top: lane l holds warp 31 - l
      const int c = wcount[31 - lane];
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (x - c < k && x >= k) {
        sh_digit = static_cast<uint32_t>(31 - lane);
        sh_above = x - c;
      }
    }
    __syncthreads();
    const int bw = static_cast<int>(sh_digit & 31u);
    // lane range l: bins [2048 bw + 64 l, +64), counted from the top (lane
    // 31 first).  Bin 64 l + y of the window is stored at 32 y + l: thread
    // (w, lane) reads y = w and w + 32 of range lane, one load each for the
    // whole block, and warp bw adds the 32 warps' counts in warp order.
    int* lsum = reinterpret_cast<int*>(ring);     // [32][32]; the ring is free here
    {
      const int* hw = hg + 2048 * bw + lane;
      lsum[32 * w + lane] = __ldcg(hw + 32 * w) + __ldcg(hw + 32 * (w + 32));
    }
    __syncthreads();
    if (w == bw) {
      int cl = 0;
#pragma unroll 8
      for (int u = 0; u < 32; ++u) cl += lsum[32 * u + lane];
      const int c = __shfl_sync(0xffffffffu, cl, 31 - lane);
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const int above_w = sh_above;
      const int hit = __ballot_sync(0xffffffffu, above_w + x - c < k && above_w + x >= k);
      const int src = __ffs(hit) - 1;             // exactly one lane
      const int bl = 31 - src;                    // the lane range holding the bin
      const int run0 = above_w + __shfl_sync(0xffffffffu, x - c, src);
      // that range's 64 bins, two per lane from the top
      const int* hb = hg + 2048 * bw + bl;
      const int c0 = __ldcg(hb + 32 * (63 - 2 * lane)), c1 = __ldcg(hb + 32 * (62 - 2 * lane));
      int y = c0 + c1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int z = __shfl_up_sync(0xffffffffu, y, o);
        if (lane >= o) y += z;
      }
      const int ex = run0 + y - (c0 + c1);        // keys above this lane's two bins
      if (ex < k && ex + c0 >= k) {
        sh_digit = static_cast<uint32_t>(2048 * bw + 64 * bl + 63 - 2 * lane);
        sh_need = k - ex;
        sh_above = c0;                            // keys in the bin
      } else if (ex + c0 < k && ex + c0 + c1 >= k) {
        sh_digit = static_cast<uint32_t>(2048 * bw + 64 * bl + 62 - 2 * lane);
        sh_need = k - ex - c0;
        sh_above = c1;
      }
    }
    __syncthreads();
  }
  const uint32_t b16 = sh_digit;
  const int in_bin = sh_above;                    // keys in the boundary bin
  const int list_n = k - sh_need + in_bin;        // keys above the bin, and the bin's
  if (list_n <= kSelSortMax) {
    // Fast path: those keys (with their indices) into shared memory, sorted by
    // key descending and index ascending; the first k are kept, then sorted by
    // index for the output.
    unsigned long long* list = reinterpret_cast<unsigned long long*>(
        reinterpret_cast<char*>(ring) + kSelCacheBytes);
    uint32_t* idx = reinterpret_cast<uint32_t*>(list + kSelSortMax);
    __shared__ int n_list;
    if (tid == 0) n_list = 0;
    __syncthreads();
    // Every score whose key has (key >> 16) >= b16 joins the list, in any
    // order (what follows does not depend on it).  Few do, so the scan first
    // tests a superset with two integer operations per score -- the order key
    // without its NaN and -0 cases, against the bin's lowest key minus one --
    // and applies the exact test only to those.
    const uint32_t lo = b16 == 0 ? 0u : (b16 << 16) - 1u;
    auto may_take = [&](float f) {
      const uint32_t b = __float_as_uint(f);
      return (b ^ (static_cast<uint32_t>(static_cast<int32_t>(b) >> 31) | 0x80000000u)) >= lo;
    };
    auto take = [&](float f, int i) {
      const uint32_t key = order_key(f);
      if ((key >> 16) >= b16) {
        const int at = atomicAdd(&n_list, 1);
        if (at < kSelSortMax)
          list[at] = (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(i));
      }
    };
    // 16-byte loads from the first 16-byte boundary; the scores before it and
    // after the last whole vector one by one
    const int h = min(n_cand, static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(sc) & 15u)) & 15u) >> 2));
    const int n4 = (n_cand - h) >> 2;
    const int tail0 = h + 4 * n4;
    if (tid < h) {
      const float f = __ldcg(sc + tid);
      if (may_take(f)) take(f, tid);
    }
    if (tid < n_cand - tail0) {
      const float f = __ldcg(sc + tail0 + tid);
      if (may_take(f)) take(f, tail0 + tid);
    }
    const float4* sc4 = reinterpret_cast<const float4*>(sc + h);
    constexpr int kV = 8;                         // 16-byte loads in flight per thread
    for (int j0 = 0; j0 < n4; j0 += kV * nt) {
      float4 v[kV];
#pragma unroll
      for (int u = 0; u < kV; ++u) {
        const int j = j0 + tid + u * nt;
        v[u] = j < n4 ? __ldcg(sc4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kV; ++u) {
        const int j = j0 + tid + u * nt;
        if (j < n4 && (may_take(v[u].x) || may_take(v[u].y) || may_take(v[u].z) || may_take(v[u].w))) {
          const int i = h + 4 * j;
          if (may_take(v[u].x)) take(v[u].x, i);
          if (may_take(v[u].y)) take(v[u].y, i + 1);
          if (may_take(v[u].z)) take(v[u].z, i + 2);
          if (may_take(v[u].w)) take(v[u].w, i + 3);
        }
      }
    }
    __syncthreads();
    if (list_n <= kSelRankMax) {
      // entry e's place in (key descending, index ascending) order is the
      // number of entries above it (the composites are distinct); the kept
      // ones then take their place in index order the same way.  Four
      // neighbouring threads share an entry, each counting every fourth one.
      static_assert(4 * kSelRankMax <= kSelThreads, "four threads per ranked entry");
      const int e = tid >> 2, part = tid & 3;
      const bool live = e < list_n;
      const unsigned long long mine = live ? list[e] : 0ull;
      const uint32_t my_idx = 0xFFFFFFFFu - static_cast<uint32_t>(mine & 0xFFFFFFFFull);
      int rank = 0;
      if (live) {
#pragma unroll 4
        for (int j = part; j < list_n; j += 4) rank += list[j] > mine ? 1 : 0;
      }
      rank += __shfl_xor_sync(0xffffffffu, rank, 1);
      rank += __shfl_xor_sync(0xffffffffu, rank, 2);
      const bool kept = live && rank < k;
      if (live && part == 0) idx[e] = kept ? my_idx : 0xFFFFFFFFu;
      __syncthreads();
      int pos = 0;
      if (kept) {
#pragma unroll 4
        for (int j = part; j < list_n; j += 4) pos += idx[j] < my_idx ? 1 : 0;
      }
      pos += __shfl_xor_sync(0xffffffffu, pos, 1);
      pos += __shfl_xor_sync(0xffffffffu, pos, 2);
      if (kept && part == 0) out[pos] = static_cast<int32_t>(my_idx);
      return;
    }
    int np = 1;
    while (np < list_n) np <<= 1;
    for (int i = list_n + tid; i < np; i += nt) list[i] = 0ull;   // below every real entry
    __syncthreads();
    int kp = 1;
    while (kp < k) kp <<= 1;
    block_bitonic_sort(list, np, true);
    for (int i = tid; i < kp; i += nt)
      idx[i] = i < k ? 0xFFFFFFFFu - static_cast<uint32_t>(list[i] & 0xFFFFFFFFull) : 0xFFFFFFFFu;
    __syncthreads();
    block_bitonic_sort(idx, kp, false);
    for (int i = tid; i < k; i += nt) out[i] = static_cast<int32_t>(idx[i]);
    return;
  }
  uint32_t prefix = sh_digit << 16;               // the k-th key's bits found so far
  int need = sh_need;                             // keys still to take with that prefix
  // digits 2 and 3: 8 bits each, over the keys that share the prefix
  for (int pass = 0; pass < 2; ++pass) {
    const int shb = 8 - 8 * pass;                 // bits [shb, shb + 8)
    const uint32_t mask = 0xFFFFFFFFu << (shb + 8);
    for (int i = tid; i < 256; i += nt) hist[i] = 0;
    __syncthreads();
    constexpr int kU = 8;                         // loads in flight per thread
    for (int base0 = 0; base0 < n_cand; base0 += kU * nt) {   // warp-uniform steps
      uint32_t key[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base0 + tid + u * nt;
        key[u] = 0u;
        if (i < n_cand) {
          if (pass == 0 || !cached) {
            key[u] = order_key(__ldcg(sc + i));
            if (pass == 0 && cached) keys_sm[i] = key[u];
          } else {
            key[u] = keys_sm[i];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base0 + tid + u * nt;
        const bool in = i < n_cand && (key[u] & mask) == prefix;
        const int b = in ? static_cast<int>((key[u] >> shb) & 255u) : -1;
        // a warp whose 32 keys fall in one bin (many equal keys) adds once
        const int b0 = __shfl_sync(0xffffffffu, b, 0);
        if (__all_sync(0xffffffffu, b == b0)) {
          if (lane == 0 && b0 >= 0) atomicAdd(&hist[b0], 32);
        } else if (in) {
          atomicAdd(&hist[b], 1);
        }
      }
    }
    __syncthreads();
    // bin counts from the top: thread t < 128 owns bins 255 - 2t and 254 - 2t
    const int b_hi = 255 - 2 * tid;
    const int c0 = tid < 128 ? hist[b_hi] : 0;
    const int c1 = tid < 128 ? hist[b_hi - 1] : 0;
    const int before = block_excl_scan(c0 + c1, warp_tot, &total);
    if (tid < 128) {
      if (before < need && before + c0 >= need) {
        sh_digit = static_cast<uint32_t>(b_hi);
        sh_need = need - before;
      } else if (before + c0 < need && before + c0 + c1 >= need) {
        sh_digit = static_cast<uint32_t>(b_hi - 1);
        sh_need = need - before - c0;
      }
    }
    __syncthreads();
    prefix |= sh_digit << shb;
    need = sh_need;
    __syncthreads();
  }
  // prefix is the k-th key, need == how many keys equal to it are kept.
  // Index-ordered compaction: warp w owns the contiguous index range
  // [w span, (w + 1) span) and walks it 32 consecutive indices at a time
  // (lane = index within the step: conflict-free shared loads), so ballots
  // give each key's rank in index order.
  const uint32_t kth = prefix;
  auto key_at = [&](int i) -> uint32_t { return cached ? keys_sm[i] : order_key(__ldcg(sc + i)); };
  const int nw = nt >> 5;
  const int span = ((n_cand + nw - 1) / nw + 31) & ~31;
  const int j0 = min(n_cand, w * span), j1 = min(n_cand, j0 + span);
  const uint32_t below = (1u << lane) - 1u;
  int n_gt = 0, n_eq = 0;
  for (int base = j0; base < j1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < j1 ? key_at(i) : 0u;
    n_gt += __popc(__ballot_sync(0xffffffffu, i < j1 && key > kth));
    n_eq += __popc(__ballot_sync(0xffffffffu, i < j1 && key == kth));
  }
  int* wsum_gt = reinterpret_cast<int*>(hist);          // the digit histogram is done
  int* wsum_eq = wsum_gt + 32;
  if (lane == 0) {
    wsum_gt[w] = n_gt;
    wsum_eq[w] = n_eq;
  }
  __syncthreads();
  int eq_rank = 0, pos = 0;
  for (int u = 0; u < w; ++u) {
    const int e = wsum_eq[u];
    pos += wsum_gt[u] + max(0, min(e, need - eq_rank));
    eq_rank += e;
  }
  for (int base = j0; base < j1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < j1 ? key_at(i) : 0u;
    const uint32_t eqm = __ballot_sync(0xffffffffu, i < j1 && key == kth);
    const bool keep = i < j1 && (key > kth || (key == kth && eq_rank + __popc(eqm & below) < need));
    const uint32_t km = __ballot_sync(0xffffffffu, keep);
    const int at = pos + __popc(km & below);
    if (keep && at < k) out[at] = i;              // k writes in all, by the counts above
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

// The rows of a partial last page past the chunk's end hold no token.  The
// tensor-core attention kernels still load them with the page and weight them
// by zero, so an inf or NaN there would reach O and dQ (0 * inf); this reads
// only those rows, one CTA per KV head, and records kStatusNonFinite.
__global__ void __launch_bounds__(256) tail_rows_kernel(const uint16_t* __restrict__ k,
                                                        const uint16_t* __restrict__ v,
                                                        const int32_t* __restrict__ pt, int page,
                                                        int valid_rows, int page_size, int hkv,
                                                        int d, int num_slots, int* status) {
  const int slot = pt[page];
  if (slot < 0 || slot >= num_slots) {
    if (threadIdx.x == 0) raise_status(status, kStatusBounds, kWhereTailRows);
    return;
  }
  const int g = blockIdx.x;
  const size_t base = ((static_cast<size_t>(slot) * hkv + g) * page_size + valid_rows) * d;
  const int n = (page_size - valid_rows) * d;
  bool bad = false;
  for (int i = threadIdx.x; i < n; i += blockDim.x)   // bf16 inf/NaN: all exponent bits set
    bad |= ((k[base + i] & 0x7f80u) == 0x7f80u) | ((v[base + i] & 0x7f80u) == 0x7f80u);
  if (__syncthreads_or(bad) && threadIdx.x == 0)
    raise_status(status, kStatusNonFinite, kWhereTailRows);
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
  const size_t row = static_cast<size_t>(hkv) * head_dim * 4;
  size_t b = kStatusBytes;
  b += align_up(kSelMaxBlocks * row, 256);                                    // partials
  b += align_up((kSelMaxBlocks / kSelGroup) * row, 256);                      // group sums
  b += align_up(row, 256);                                                    // qbar
  b += align_up(static_cast<size_t>(hkv) * num_pages * 4, 256);              // scores
  b += static_cast<size_t>(hkv) * 65536 * 4;                                  // key histogram
  return b;
}

namespace {
// The grid of the selection kernel on the current device: every CTA must be
// resident at once (cooperative launch), one per SM.
template <typename T, int D>
cudaError_t sel_grid(int* blocks) {
  static PerDeviceOnce once;
  static int cached[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = once_per_device(once, [&] {
    cudaError_t r = cudaFuncSetAttribute(select_kernel<T, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSelDynSmem));
    if (r != cudaSuccess) return r;
    int sms = 0, per_sm = 0;
    r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (r != cudaSuccess) return r;
    r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, select_kernel<T, D>, kSelThreads,
                                                      kSelDynSmem);
    if (r != cudaSuccess) return r;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    cached[dev & 127] = sms < kSelMaxBlocks ? sms : kSelMaxBlocks;
    return cudaSuccess;
  });
  if (e != cudaSuccess) return e;
  *blocks = cached[dev & 127];
  return cudaSuccess;
}

template <typename T, int D>
cudaError_t launch_select(const SelParams& prm, cudaStream_t st) {
  int blocks = 0;
  cudaError_t e = sel_grid<T, D>(&blocks);
  if (e != cudaSuccess) return e;
  if (blocks < prm.hkv) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = kSelDynSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: they wait for one another
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, select_kernel<T, D>, prm);
}
}  // namespace

cudaError_t launch_select_topk(const void* q, bool bf16, int hq, int chunk_len, int n_cand,
                               const float* reps, int num_pages, int hkv, int head_dim, int top_k,
                               int32_t* sel, float* scores_opt, void* ws, uint64_t wait_ns,
                               cudaStream_t st) {
  const size_t row = static_cast<size_t>(hkv) * head_dim * 4;
  char* w = static_cast<char*>(ws);
  SelParams prm;
  prm.status = reinterpret_cast<int*>(w);
  w += kStatusBytes;
  prm.partials = reinterpret_cast<float*>(w);
  w += align_up(kSelMaxBlocks * row, 256);
  prm.gsums = reinterpret_cast<float*>(w);
  w += align_up((kSelMaxBlocks / kSelGroup) * row, 256);
  prm.qbar = reinterpret_cast<float*>(w);
  w += align_up(row, 256);
  float* scores_ws = reinterpret_cast<float*>(w);
  w += align_up(static_cast<size_t>(hkv) * num_pages * 4, 256);
  prm.hist = reinterpret_cast<int*>(w);
  prm.scores = scores_opt ? scores_opt : scores_ws;
  prm.q = q;
  prm.reps = reps;
  prm.sel = sel;
  prm.chunk_len = chunk_len;
  prm.hq = hq;
  prm.hkv = hkv;
  prm.n_cand = n_cand;
  prm.num_pages = num_pages;
  prm.top_k = top_k;
  prm.wait_ns = wait_ns;
  return bf16 ? launch_select<__nv_bfloat16, 128>(prm, st) : launch_select<float, 64>(prm, st);
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
                                       bool* too_big, uint64_t wait_ns, cudaStream_t st) {
  *too_big = select_ws_bytes(num_pages, hkv, head_dim) > OOMB_NOALLOC_SCRATCH_BYTES;
  if (*too_big) return cudaSuccess;
  void* scratch = nullptr;
  cudaError_t e = select_scratch_addr(&scratch);
  if (e != cudaSuccess) return e;
  // the status block (with the query-summary ticket counter) must start at zero
  e = cudaMemsetAsync(scratch, 0, kStatusBytes, st);
  if (e != cudaSuccess) return e;
  return launch_select_topk(q, bf16, hq, chunk_len, n_cand, reps, num_pages, hkv, head_dim,
                            top_k, sel, scores_opt, scratch, wait_ns, st);
}

cudaError_t launch_validate_page_table(const int32_t* pt, int num_pages, int num_slots,
                                       uint32_t* bitmap, int* status, cudaStream_t st) {
  if (num_pages == 0) return cudaSuccess;
  validate_pt_kernel<<<(num_pages + 255) / 256, 256, 0, st>>>(pt, num_pages, num_slots, bitmap,
                                                              status);
  return cudaGetLastError();
}

cudaError_t launch_check_tail_rows(const KvDesc& kv, int page, int valid_rows, int* status,
                                   cudaStream_t st) {
  if (valid_rows <= 0 || valid_rows >= kv.page_size) return cudaSuccess;
  tail_rows_kernel<<<kv.hkv, 256, 0, st>>>(static_cast<const uint16_t*>(kv.k),
                                           static_cast<const uint16_t*>(kv.v), kv.page_table, page,
                                           valid_rows, kv.page_size, kv.hkv, kv.head_dim,
                                           kv.num_slots, status);
  return cudaGetLastError();
}

cudaError_t launch_debug_wait(int* status, uint64_t limit_ns, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace oomb
