// Host-tier page pools with a device page cache: the C-ABI calls
// oomb_offload_* declared in include/oomb.h.
// Method: "Out of the Memory Barrier" technical summary, section 2, the
// fourth optimisation ("Async CPU offloading"): the KV cache and its
// gradients need not all sit in GPU memory; pages move between host and GPU
// asynchronously, ahead of the kernels that use them.
//
// Design (one GB300 with its Grace host): the pools of every page are pinned
// host memory, which the GPU reads and writes directly over the CPU-GPU link.
// A chunk's tiles -- (page, KV head) blocks of P x D elements -- are moved by
// one kernel per direction (at most one CTA per SM, each looping over tiles)
// from a task list the host writes into a pinned staging buffer; no per-tile
// copy call.  The host keeps
// the cache directory: which logical page sits in which cache slot, which KV
// heads of it are loaded (K/V, gradients), which gradient tiles are modified,
// and when the slot was last used.  Slots used by the current and the
// previous acquire are never reused, so the next chunk's tiles can be brought
// in on another stream while the current chunk computes.
// The backing pools may also be device memory (a compact tier in HBM), and
// the backing K/V pools may hold 8-bit E4M3 codes that each fetch expands to
// bf16 in the cache (an fp8 KV cache; E4M3 values are bf16 values, so the
// kernels see exactly the stored values).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <condition_variable>
#include <cstring>
#include <mutex>
#include <new>
#include <thread>
#include <utility>
#include <vector>

#include "oomb.h"
#include "oomb_internal.h"
#include "page_cache_directory.h"

namespace {

enum CopyMode : int32_t {
  kCopy = 0,        // dst = src
  kExpand = 1,      // src holds E4M3 codes, dst receives their bf16 values
  kZeroFill = 2,    // dst = 0 (src unused)
};

struct TileCopy {
  const uint4* src;
  uint4* dst;
  int32_t mode;
  int32_t pad;
};

// bf16 pair of the two E4M3 codes in the 16 bits `c2` (low code -> low half):
// the hardware conversion to an f16 pair is exact (every E4M3 value is an f16
// value), and so is each f16 -> f32 step, whose low 16 bits are then zero.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t c2) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c2));
  float lo, hi;
  asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"(static_cast<uint16_t>(h2 & 0xFFFFu)));
  asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"(static_cast<uint16_t>(h2 >> 16)));
  return (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
}

__device__ __forceinline__ uint4 expand8(uint32_t w0, uint32_t w1) {   // 8 codes -> 8 bf16
  return make_uint4(e4m3x2_to_bf16x2(static_cast<uint16_t>(w0)),
                    e4m3x2_to_bf16x2(static_cast<uint16_t>(w0 >> 16)),
                    e4m3x2_to_bf16x2(static_cast<uint16_t>(w1)),
                    e4m3x2_to_bf16x2(static_cast<uint16_t>(w1 >> 16)));
}

// Tiles of n16 16-byte words (of the destination), tile blockIdx.x,
// blockIdx.x + gridDim.x, ...: 8 loads in flight per thread, then the stores.
// Either side may be pinned host memory (zero-copy) or device memory.  An
// expanding task reads n16 / 2 words of codes and writes two words per word
// read; a zero fill only writes.  64 threads (80 registers each): small
// enough to share an SM with a running forward-attention CTA.  The grid is at
// most one CTA per SM whatever the number of tiles: moves over the CPU-GPU
// link are latency-bound, so a grid of one CTA per tile would take every SM
// that an attention kernel frees for the whole length of the move, where a
// bounded grid takes a few SMs' worth and keeps the link as busy.
constexpr int kCopyThreads = 64;
__device__ __forceinline__ void copy_tile(const TileCopy& t, int n16) {
  if (t.mode == kZeroFill) {
    for (int k = threadIdx.x; k < n16; k += kCopyThreads) t.dst[k] = make_uint4(0, 0, 0, 0);
    return;
  }
  if (t.mode == kExpand) {
    const int n_src = n16 / 2;
    for (int base = threadIdx.x; base < n_src; base += kCopyThreads * 8) {
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = base + i * kCopyThreads;
        if (k < n_src) v[i] = t.src[k];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = base + i * kCopyThreads;
        if (k < n_src) {
          t.dst[2 * k] = expand8(v[i].x, v[i].y);
          t.dst[2 * k + 1] = expand8(v[i].z, v[i].w);
        }
      }
    }
    return;
  }
  for (int base = threadIdx.x; base < n16; base += kCopyThreads * 8) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int k = base + i * kCopyThreads;
      if (k < n16) v[i] = t.src[k];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int k = base + i * kCopyThreads;
      if (k < n16) t.dst[k] = v[i];
    }
  }
}

__global__ void __launch_bounds__(kCopyThreads) tile_copy_kernel(
    const TileCopy* __restrict__ tasks, int n_tasks, int n16) {
  for (int i = blockIdx.x; i < n_tasks; i += gridDim.x) copy_tile(tasks[i], n16);
}

// Host threads that run the host-side tile copies of the staged path.  A
// stream callback hands a list to the pool and waits for it: the copies happen
// in stream order, on the pool's threads, without blocking the caller.
class CopyPool {
 public:
  explicit CopyPool(size_t n) {
    for (size_t i = 0; i < n; ++i) th_.emplace_back([this, i] { loop(i); });
  }
  ~CopyPool() {
    {
      std::lock_guard<std::mutex> g(mu_);
      stop_ = true;
      ++gen_;
    }
    cv_.notify_all();
    for (auto& t : th_) t.join();
  }
  size_t size() const { return th_.size(); }
  // Copy list[0, n) (tile_bytes each) with every thread of the pool; returns
  // when all copies are done.  Called from one callback at a time.
  void run(const TileCopy* list, size_t n, size_t tile_bytes) {
    {
      std::lock_guard<std::mutex> g(mu_);
      list_ = list;
      n_ = n;
      tb_ = tile_bytes;
      next_.store(0);
      pending_ = th_.size();
      ++gen_;
    }
    cv_.notify_all();
    std::unique_lock<std::mutex> g(mu_);
    done_cv_.wait(g, [this] { return pending_ == 0; });
  }

 private:
  void loop(size_t) {
    uint64_t seen = 0;
    while (true) {
      {
        std::unique_lock<std::mutex> g(mu_);
        cv_.wait(g, [&] { return gen_ != seen; });
        seen = gen_;
        if (stop_) return;
      }
      while (true) {                       // tiles handed out 8 at a time
        const size_t i0 = next_.fetch_add(8);
        if (i0 >= n_) break;
        const size_t i1 = std::min(n_, i0 + 8);
        for (size_t i = i0; i < i1; ++i)
          std::memcpy(reinterpret_cast<void*>(list_[i].dst),
                      reinterpret_cast<const void*>(list_[i].src), tb_);
      }
      {
        std::lock_guard<std::mutex> g(mu_);
        if (--pending_ == 0) done_cv_.notify_one();
      }
    }
  }
  std::vector<std::thread> th_;
  std::mutex mu_;
  std::condition_variable cv_, done_cv_;
  const TileCopy* list_ = nullptr;
  size_t n_ = 0, tb_ = 0, pending_ = 0;
  std::atomic<size_t> next_{0};
  uint64_t gen_ = 0;
  bool stop_ = false;
};

// A list of host-side tile copies for the pool, run by a stream callback.
struct HostMove {
  CopyPool* pool;
  const TileCopy* list;
  size_t n;
  size_t tile_bytes;
};

void CUDART_CB host_copy_cb(void* arg) {
  const HostMove* m = static_cast<const HostMove*>(arg);
  if (m->n) m->pool->run(m->list, m->n, m->tile_bytes);
}

// Pinned staging for one acquire, flush or write-back: its task lists and page
// table mirror, and the event recorded after the moves that read them.
struct Staging {
  TileCopy* tasks = nullptr;       // planned moves: [0, n_wb) write-backs, then fetches
  TileCopy* tasks_dev = nullptr;   // device view of `tasks`
  TileCopy* dev_tasks = nullptr;   // through the device staging buffer: device-side copies
  TileCopy* dev_tasks_dev = nullptr;
  std::vector<TileCopy> host_tasks;  // through the host staging buffer: host-side copies
  std::vector<HostMove> moves;
  int32_t* pt = nullptr;
  cudaEvent_t done = nullptr;
  size_t n_zero = 0;                 // zero fills at the end of `tasks`
  bool used = false;
};

bool is_host_pinned(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

bool is_device(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice;
}

}  // namespace

struct oomb_offload {
  oomb_offload_desc d;
  size_t tile_bytes = 0;                 // P * D * element size (cache; backing dK/dV)
  size_t kv_tile_bytes = 0;              // P * D * element size of the backing K/V pools
  int32_t kv_mode = 0;                   // kExpand: backing K/V hold E4M3 codes
  std::vector<int32_t> host_pt;          // logical page -> host slot
  oomb::PageCacheDirectory* dir = nullptr;
  std::vector<oomb::TileMove> moves;     // the current call's plan
  size_t cap_tasks = 0;
  // copy-engine path: tiles move through a device staging buffer (caller's)
  // and a pinned host staging buffer (the library's) of the same size
  char* dev_staging = nullptr;
  char* host_staging = nullptr;
  size_t stage_tiles = 0;                // tiles per round; 0: zero-copy kernels
  CopyPool* pool = nullptr;              // host copy threads of the staged path
  cudaEvent_t last_done = nullptr;       // moves of the previous call (any stream)
  Staging stage[4];
  int next_stage = 0;
  int64_t stats[7] = {0, 0, 0, 0, 0, 0, 0};
};

namespace {

char* tile_ptr(void* pool, const oomb_offload* h, int slot, int g) {
  return static_cast<char*>(pool) +
         (static_cast<size_t>(slot) * h->d.num_kv_heads + g) * h->tile_bytes;
}

char* backing_kv_ptr(void* pool, const oomb_offload* h, int slot, int g) {
  return static_cast<char*>(pool) +
         (static_cast<size_t>(slot) * h->d.num_kv_heads + g) * h->kv_tile_bytes;
}

oomb_status take_stage(oomb_offload* h, Staging** out) {
  Staging& st = h->stage[h->next_stage];
  h->next_stage = (h->next_stage + 1) % 4;
  if (st.used) {
    cudaError_t e = cudaEventSynchronize(st.done);
    if (e != cudaSuccess) return oomb::report(OOMB_ERR_CUDA, "offload staging wait: %s",
                                              cudaGetErrorString(e));
  }
  *out = &st;
  return OOMB_OK;
}

// Launch the copies list[0, n) (device-readable list) with the copy kernel.
cudaError_t launch_list(const oomb_offload* h, const TileCopy* list, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (n > static_cast<size_t>(INT32_MAX)) return cudaErrorInvalidValue;
  // Same shared-memory carveout as the attention kernels, so that a copy CTA
  // can share an SM with one of theirs instead of waiting for the SM to drain.
  static oomb::PerDeviceOnce carveout;
  {
    cudaError_t e = oomb::once_per_device(carveout, [] {
      return cudaFuncSetAttribute(tile_copy_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared);
    });
    if (e != cudaSuccess) return e;
  }
  static oomb::PerDeviceOnce sm_once;
  static int sms[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = oomb::once_per_device(sm_once, [dev] {
    return cudaDeviceGetAttribute(&sms[dev & 127], cudaDevAttrMultiProcessorCount, dev);
  });
  if (e != cudaSuccess) return e;
  const size_t grid = std::min<size_t>(n, sms[dev & 127] > 0 ? sms[dev & 127] : 1);
  tile_copy_kernel<<<static_cast<unsigned>(grid), kCopyThreads, 0, s>>>(
      list, static_cast<int>(n), static_cast<int>(h->tile_bytes / 16));
  return cudaGetLastError();
}

// Enqueue the planned moves st.tasks[0, n): write-backs [0, n_wb) (cache ->
// host) before fetches [n_wb, n) (host -> cache, which may reuse a slot just
// written back), the last st.n_zero of which are zero fills of cache tiles.
// Zero-copy: the copy kernel reads or writes the host pools directly.
// Staged: per round of at most stage_tiles tiles, write-backs go cache ->
// device staging (kernel) -> host staging (copy engine) -> host pools (host
// callback), fetches the reverse way, so the bulk of the bytes crosses the
// CPU-GPU link on a copy engine instead of occupying SMs; the zero fills,
// which touch only the cache, follow as one kernel launch.
cudaError_t enqueue_moves(oomb_offload* h, Staging& st, size_t n_wb, size_t n, cudaStream_t s) {
  if (h->stage_tiles == 0) {
    cudaError_t e = launch_list(h, st.tasks_dev, n_wb, s);
    if (e == cudaSuccess) e = launch_list(h, st.tasks_dev + n_wb, n - n_wb, s);
    return e;
  }
  if (n == 0) return cudaSuccess;
  const size_t n_zero = st.n_zero;
  n -= n_zero;
  if (h->last_done) {
    cudaError_t e = cudaStreamWaitEvent(s, h->last_done, 0);   // one set of staging buffers
    if (e != cudaSuccess) return e;
  }
  const size_t cap = h->stage_tiles, tb = h->tile_bytes;
  st.host_tasks.resize(n);
  st.moves.clear();
  st.moves.reserve((n_wb + cap - 1) / cap + (n - n_wb + cap - 1) / cap);
  for (size_t r0 = 0; r0 < n_wb; r0 += cap) {
    const size_t k = std::min(cap, n_wb - r0);
    for (size_t i = 0; i < k; ++i) {
      st.dev_tasks[r0 + i] = {st.tasks[r0 + i].src,
                              reinterpret_cast<uint4*>(h->dev_staging + i * tb), 0, 0};
      st.host_tasks[r0 + i] = {reinterpret_cast<const uint4*>(h->host_staging + i * tb),
                               st.tasks[r0 + i].dst, 0, 0};
    }
    cudaError_t e = launch_list(h, st.dev_tasks_dev + r0, k, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h->host_staging, h->dev_staging, k * tb, cudaMemcpyDeviceToHost, s);
    st.moves.push_back({h->pool, st.host_tasks.data() + r0, k, tb});
    if (e == cudaSuccess) e = cudaLaunchHostFunc(s, host_copy_cb, &st.moves.back());
    if (e != cudaSuccess) return e;
  }
  for (size_t r0 = n_wb; r0 < n; r0 += cap) {
    const size_t k = std::min(cap, n - r0);
    for (size_t i = 0; i < k; ++i) {
      st.host_tasks[r0 + i] = {st.tasks[r0 + i].src,
                               reinterpret_cast<uint4*>(h->host_staging + i * tb), 0, 0};
      st.dev_tasks[r0 + i] = {reinterpret_cast<const uint4*>(h->dev_staging + i * tb),
                              st.tasks[r0 + i].dst, 0, 0};
    }
    st.moves.push_back({h->pool, st.host_tasks.data() + r0, k, tb});
    cudaError_t e = cudaLaunchHostFunc(s, host_copy_cb, &st.moves.back());
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h->dev_staging, h->host_staging, k * tb, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = launch_list(h, st.dev_tasks_dev + r0, k, s);
    if (e != cudaSuccess) return e;
  }
  return launch_list(h, st.tasks_dev + n, n_zero, s);
}

// The copies of a plan's tile moves: two per move (K and V, or dK and dV), in
// the plan's order, then the zero fills (st.n_zero of them).
size_t plan_to_tasks(oomb_offload* h, Staging& st) {
  const oomb_offload_desc& d = h->d;
  size_t n = 0;
  for (const oomb::TileMove& m : h->moves) {
    const int hs = h->host_pt[m.page];
    switch (m.kind) {
      case oomb::TileMove::kZeroGrad:
        break;                                     // below, after every copy
      case oomb::TileMove::kWriteGrad:
        st.tasks[n++] = {reinterpret_cast<const uint4*>(tile_ptr(d.cache_dk, h, m.slot, m.head)),
                         reinterpret_cast<uint4*>(tile_ptr(d.dk, h, hs, m.head)), 0, 0};
        st.tasks[n++] = {reinterpret_cast<const uint4*>(tile_ptr(d.cache_dv, h, m.slot, m.head)),
                         reinterpret_cast<uint4*>(tile_ptr(d.dv, h, hs, m.head)), 0, 0};
        h->stats[1] += 2;
        h->stats[3] += 2 * static_cast<int64_t>(h->tile_bytes);
        break;
      case oomb::TileMove::kFetchKV:
        st.tasks[n++] = {reinterpret_cast<const uint4*>(backing_kv_ptr(d.k, h, hs, m.head)),
                         reinterpret_cast<uint4*>(tile_ptr(d.cache_k, h, m.slot, m.head)),
                         h->kv_mode, 0};
        st.tasks[n++] = {reinterpret_cast<const uint4*>(backing_kv_ptr(d.v, h, hs, m.head)),
                         reinterpret_cast<uint4*>(tile_ptr(d.cache_v, h, m.slot, m.head)),
                         h->kv_mode, 0};
        h->stats[0] += 2;
        h->stats[2] += 2 * static_cast<int64_t>(h->kv_tile_bytes);
        break;
      case oomb::TileMove::kFetchGrad:
        st.tasks[n++] = {reinterpret_cast<const uint4*>(tile_ptr(d.dk, h, hs, m.head)),
                         reinterpret_cast<uint4*>(tile_ptr(d.cache_dk, h, m.slot, m.head)), 0, 0};
        st.tasks[n++] = {reinterpret_cast<const uint4*>(tile_ptr(d.dv, h, hs, m.head)),
                         reinterpret_cast<uint4*>(tile_ptr(d.cache_dv, h, m.slot, m.head)), 0, 0};
        h->stats[0] += 2;
        h->stats[2] += 2 * static_cast<int64_t>(h->tile_bytes);
        break;
    }
  }
  st.n_zero = 0;
  for (const oomb::TileMove& m : h->moves) {
    if (m.kind != oomb::TileMove::kZeroGrad) continue;
    st.tasks[n++] = {nullptr, reinterpret_cast<uint4*>(tile_ptr(d.cache_dk, h, m.slot, m.head)),
                     kZeroFill, 0};
    st.tasks[n++] = {nullptr, reinterpret_cast<uint4*>(tile_ptr(d.cache_dv, h, m.slot, m.head)),
                     kZeroFill, 0};
    st.n_zero += 2;
    h->stats[6] += 2;
  }
  return n;
}

// Enqueue st.tasks (write-backs [0, n_wb) first) and record the call's event.
oomb_status finish_call(oomb_offload* h, Staging& st, size_t n_wb, size_t n, cudaStream_t s,
                        int32_t* page_table_dev, const char* what) {
  cudaError_t e = enqueue_moves(h, st, n_wb, n, s);
  if (e == cudaSuccess && page_table_dev) {
    std::memcpy(st.pt, h->dir->slot_of_page().data(),
                static_cast<size_t>(h->d.num_pages) * sizeof(int32_t));
    e = cudaMemcpyAsync(page_table_dev, st.pt,
                        static_cast<size_t>(h->d.num_pages) * sizeof(int32_t),
                        cudaMemcpyHostToDevice, s);
  }
  if (e == cudaSuccess) e = cudaEventRecord(st.done, s);
  if (e == cudaSuccess && h->last_done) e = cudaEventRecord(h->last_done, s);
  st.used = true;
  if (e != cudaSuccess) return oomb::report(OOMB_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return OOMB_OK;
}

}  // namespace

extern "C" {

oomb_status oomb_offload_create(const oomb_offload_desc* d, oomb_offload** out) {
  OOMB_NVTX_RANGE("oomb_offload_create");
  if (!d || !out) return oomb::report(OOMB_ERR_INVALID_ARG, "desc and out must be set");
  *out = nullptr;
  if (d->dtype != OOMB_BF16 && d->dtype != OOMB_FP32)
    return oomb::report(OOMB_ERR_INVALID_ARG, "dtype %d", static_cast<int>(d->dtype));
  if (d->num_pages <= 0 || d->num_host_slots < d->num_pages || d->cache_slots <= 0)
    return oomb::report(OOMB_ERR_INVALID_ARG,
                        "need num_pages > 0, num_host_slots >= num_pages, cache_slots > 0");
  if (d->num_kv_heads <= 0 || d->num_kv_heads > 32)
    return oomb::report(OOMB_ERR_UNSUPPORTED, "num_kv_heads must be in [1, 32]");
  if (d->page_size <= 0 || d->head_dim <= 0)
    return oomb::report(OOMB_ERR_INVALID_ARG, "page_size and head_dim must be positive");
  const bool fp8_kv = d->backing_kv_dtype == OOMB_FP8_E4M3;
  if (d->backing_kv_dtype != d->dtype && !(fp8_kv && d->dtype == OOMB_BF16))
    return oomb::report(OOMB_ERR_INVALID_ARG,
                        "backing_kv_dtype %d: must equal dtype, or be FP8_E4M3 with BF16",
                        static_cast<int>(d->backing_kv_dtype));
  if (fp8_kv && d->dev_staging)
    return oomb::report(OOMB_ERR_UNSUPPORTED, "fp8 K/V pools move by the zero-copy kernel only");
  const size_t elem = d->dtype == OOMB_BF16 ? 2 : 4;
  const size_t tile = static_cast<size_t>(d->page_size) * d->head_dim * elem;
  const size_t kv_tile = fp8_kv ? tile / 2 : tile;
  if (kv_tile % 16) return oomb::report(OOMB_ERR_UNSUPPORTED, "tile bytes must be a multiple of 16");
  if (!d->k || !d->v || !d->cache_k || !d->cache_v || !d->host_page_table)
    return oomb::report(OOMB_ERR_INVALID_ARG, "k, v, cache_k, cache_v, host_page_table must be set");
  if ((d->dk == nullptr) != (d->cache_dk == nullptr) || (d->dv == nullptr) != (d->cache_dv == nullptr) ||
      (d->dk == nullptr) != (d->dv == nullptr))
    return oomb::report(OOMB_ERR_INVALID_ARG, "dk, dv, cache_dk, cache_dv: all set or all NULL");
  const void* host_pools[4] = {d->k, d->v, d->dk, d->dv};
  const void* dev_pools[4] = {d->cache_k, d->cache_v, d->cache_dk, d->cache_dv};
  for (int i = 0; i < 4; ++i) {
    // the staged path gathers on the host: its backing pools must be host memory
    if (host_pools[i] &&
        (!(is_host_pinned(host_pools[i]) || (!d->dev_staging && is_device(host_pools[i]))) ||
         reinterpret_cast<uintptr_t>(host_pools[i]) % 16))
      return oomb::report(OOMB_ERR_INVALID_ARG,
                          "backing pool %d must be pinned host memory (or device memory "
                          "without dev_staging), 16-byte aligned", i);
    if (dev_pools[i] && (!is_device(dev_pools[i]) ||
                         reinterpret_cast<uintptr_t>(dev_pools[i]) % 16))
      return oomb::report(OOMB_ERR_INVALID_ARG,
                          "cache pool %d must be device memory, 16-byte aligned", i);
  }
  if (d->dev_staging && (!is_device(d->dev_staging) ||
                         reinterpret_cast<uintptr_t>(d->dev_staging) % 16 ||
                         d->dev_staging_bytes < static_cast<int64_t>(tile)))
    return oomb::report(OOMB_ERR_INVALID_ARG,
                        "dev_staging must be device memory, 16-byte aligned, >= one tile");
  oomb_offload* h = new (std::nothrow) oomb_offload();
  if (!h) return oomb::report(OOMB_ERR_INVALID_ARG, "out of host memory");
  h->d = *d;
  h->tile_bytes = tile;
  h->kv_tile_bytes = kv_tile;
  h->kv_mode = fp8_kv ? kExpand : kCopy;
  h->host_pt.assign(d->host_page_table, d->host_page_table + d->num_pages);
  {
    std::vector<char> seen(d->num_host_slots, 0);
    for (int l = 0; l < d->num_pages; ++l) {
      const int s = h->host_pt[l];
      if (s < 0 || s >= d->num_host_slots || seen[s]) {
        delete h;
        return oomb::report(OOMB_ERR_INVALID_ARG,
                            "host page table: page %d -> slot %d is out of range or repeated", l, s);
      }
      seen[s] = 1;
    }
  }
  h->dir = new (std::nothrow) oomb::PageCacheDirectory(d->num_pages, d->cache_slots,
                                                       d->num_kv_heads);
  if (!h->dir) {
    delete h;
    return oomb::report(OOMB_ERR_INVALID_ARG, "out of host memory");
  }
  // per slot and KV head: an acquire writes back at most 2 tiles (dK, dV) and
  // fetches at most 4 (K, V, dK, dV); a flush writes back at most 2
  h->cap_tasks = static_cast<size_t>(d->cache_slots) * d->num_kv_heads * 6 + 16;
  if (d->dev_staging) {
    h->stage_tiles = static_cast<size_t>(d->dev_staging_bytes) / tile;
    h->dev_staging = static_cast<char*>(d->dev_staging);
    const unsigned hw = std::thread::hardware_concurrency();
    h->pool = new (std::nothrow) CopyPool(std::max(1u, std::min(8u, hw ? hw / 2 : 1u)));
    cudaError_t e = h->pool ? cudaHostAlloc(&h->host_staging, h->stage_tiles * tile,
                                            cudaHostAllocDefault)
                            : cudaErrorMemoryAllocation;
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->last_done, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      oomb_offload_destroy(h);
      return oomb::report(OOMB_ERR_CUDA, "offload host staging: %s", cudaGetErrorString(e));
    }
  }
  for (auto& st : h->stage) {
    cudaError_t e = cudaHostAlloc(&st.tasks, h->cap_tasks * sizeof(TileCopy), cudaHostAllocMapped);
    if (e == cudaSuccess)
      e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&st.tasks_dev), st.tasks, 0);
    if (e == cudaSuccess)
      e = cudaHostAlloc(&st.dev_tasks, h->cap_tasks * sizeof(TileCopy), cudaHostAllocMapped);
    if (e == cudaSuccess)
      e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&st.dev_tasks_dev), st.dev_tasks, 0);
    if (e == cudaSuccess)
      e = cudaHostAlloc(&st.pt, static_cast<size_t>(d->num_pages) * sizeof(int32_t),
                        cudaHostAllocDefault);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&st.done, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      oomb_offload_destroy(h);
      return oomb::report(OOMB_ERR_CUDA, "offload staging: %s", cudaGetErrorString(e));
    }
  }
  *out = h;
  return OOMB_OK;
}

oomb_status oomb_offload_acquire(oomb_offload* h, const int32_t* sel_host, int32_t n_sel,
                                 int32_t chunk_start, int32_t chunk_len, int32_t with_grads,
                                 int32_t* page_table_dev, void* stream) {
  OOMB_NVTX_RANGE("oomb_offload_acquire");
  if (!h || !page_table_dev) return oomb::report(OOMB_ERR_INVALID_ARG, "handle and page_table_dev");
  const oomb_offload_desc& d = h->d;
  const int P = d.page_size;
  // the chunk starts on a page; its last page may be partial
  if (chunk_start < 0 || chunk_len <= 0 || chunk_start % P ||
      static_cast<long long>(chunk_start) + chunk_len > static_cast<long long>(d.num_pages) * P)
    return oomb::report(OOMB_ERR_INVALID_ARG,
                        "chunk [%d, %d) does not start on a page or runs past the %d pages",
                        chunk_start, chunk_start + chunk_len, d.num_pages);
  if (n_sel < 0 || (n_sel > 0 && !sel_host))
    return oomb::report(OOMB_ERR_INVALID_ARG, "n_sel %d / sel_host", n_sel);
  if (with_grads && !d.dk)
    return oomb::report(OOMB_ERR_INVALID_ARG, "with_grads needs the dK/dV pools");
  // the staging buffer is taken first: a failed wait leaves the directory as it was
  Staging* st = nullptr;
  oomb_status rs = take_stage(h, &st);
  if (rs != OOMB_OK) return rs;
  h->moves.clear();
  size_t n_wb_moves = 0;
  const std::string err = h->dir->plan(sel_host, n_sel, chunk_start / P,
                                       (chunk_start + chunk_len + P - 1) / P, with_grads != 0,
                                       &h->moves,
                                       &n_wb_moves, &h->stats[5]);
  if (!err.empty()) return oomb::report(OOMB_ERR_INVALID_ARG, "%s", err.c_str());
  const size_t n = plan_to_tasks(h, *st);
  ++h->stats[4];
  return finish_call(h, *st, 2 * n_wb_moves, n, static_cast<cudaStream_t>(stream),
                     page_table_dev, "offload acquire");
}

oomb_status oomb_offload_flush(oomb_offload* h, int32_t drop, void* stream) {
  OOMB_NVTX_RANGE("oomb_offload_flush");
  if (!h) return oomb::report(OOMB_ERR_INVALID_ARG, "handle");
  Staging* st = nullptr;
  oomb_status rs = take_stage(h, &st);
  if (rs != OOMB_OK) return rs;
  h->moves.clear();
  h->dir->collect_writebacks(0, -1, &h->moves);
  if (drop) h->dir->drop();
  const size_t n = plan_to_tasks(h, *st);
  return finish_call(h, *st, n, n, static_cast<cudaStream_t>(stream), nullptr, "offload flush");
}

oomb_status oomb_offload_writeback(oomb_offload* h, int32_t first_page, int32_t n_pages,
                                   void* stream) {
  OOMB_NVTX_RANGE("oomb_offload_writeback");
  if (!h) return oomb::report(OOMB_ERR_INVALID_ARG, "handle");
  if (first_page < 0 || n_pages < 0 || first_page + n_pages > h->d.num_pages)
    return oomb::report(OOMB_ERR_INVALID_ARG, "pages [%d, %d) outside [0, %d)", first_page,
                        first_page + n_pages, h->d.num_pages);
  Staging* st = nullptr;
  oomb_status rs = take_stage(h, &st);
  if (rs != OOMB_OK) return rs;
  h->moves.clear();
  h->dir->collect_writebacks(first_page, n_pages, &h->moves);
  const size_t n = plan_to_tasks(h, *st);
  return finish_call(h, *st, n, n, static_cast<cudaStream_t>(stream), nullptr,
                     "offload writeback");
}

oomb_status oomb_offload_writeback_pages(oomb_offload* h, const int32_t* pages_host,
                                         int32_t n, void* stream) {
  OOMB_NVTX_RANGE("oomb_offload_writeback_pages");
  if (!h) return oomb::report(OOMB_ERR_INVALID_ARG, "handle");
  if (n < 0 || (n > 0 && !pages_host))
    return oomb::report(OOMB_ERR_INVALID_ARG, "pages_host is NULL or n < 0");
  for (int32_t i = 0; i < n; ++i)
    if (pages_host[i] < 0 || pages_host[i] >= h->d.num_pages)
      return oomb::report(OOMB_ERR_INVALID_ARG, "page %d outside [0, %d)", pages_host[i],
                          h->d.num_pages);
  Staging* st = nullptr;
  oomb_status rs = take_stage(h, &st);
  if (rs != OOMB_OK) return rs;
  h->moves.clear();
  h->dir->collect_writebacks_of(pages_host, n, &h->moves);
  const size_t m = plan_to_tasks(h, *st);
  return finish_call(h, *st, m, m, static_cast<cudaStream_t>(stream), nullptr,
                     "offload writeback of pages");
}

oomb_status oomb_offload_zero_grads(oomb_offload* h) {
  if (!h) return oomb::report(OOMB_ERR_INVALID_ARG, "handle");
  if (!h->d.dk) return oomb::report(OOMB_ERR_INVALID_ARG, "the cache has no gradient pools");
  h->dir->declare_host_grads_zero();
  return OOMB_OK;
}

oomb_status oomb_offload_stats(const oomb_offload* h, int64_t* out) {
  if (!h || !out) return oomb::report(OOMB_ERR_INVALID_ARG, "handle and out");
  for (int i = 0; i < 7; ++i) out[i] = h->stats[i];
  return OOMB_OK;
}

void oomb_offload_destroy(oomb_offload* h) {
  if (!h) return;
  for (auto& st : h->stage) {
    if (st.used && st.done) cudaEventSynchronize(st.done);
    if (st.done) cudaEventDestroy(st.done);
    if (st.tasks) cudaFreeHost(st.tasks);
    if (st.dev_tasks) cudaFreeHost(st.dev_tasks);
    if (st.pt) cudaFreeHost(st.pt);
  }
  if (h->last_done) cudaEventDestroy(h->last_done);
  if (h->host_staging) cudaFreeHost(h->host_staging);
  delete h->pool;
  delete h->dir;
  delete h;
}

}  // extern "C"
