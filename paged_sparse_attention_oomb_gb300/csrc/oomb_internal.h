// Internal interface between the C-ABI host layer (oomb_abi.cu) and the
// kernel translation units.  Host-callable launchers only; plain pointers.
#pragma once
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "oomb.h"

namespace oomb {

// Records a host-side error message for oomb_last_error() and returns `s`
// (defined in oomb_abi.cu).
oomb_status report(oomb_status s, const char* fmt, ...);

// An NVTX range named after the ABI call, open for the call's host-side work
// (checks and launches), so that a profiler's timeline and launch list group
// the kernels by the call that issued them.  Costs nothing unless a tool is
// attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define OOMB_NVTX_RANGE(name) ::oomb::NvtxRange oomb_nvtx_range_(name)

// Workspace: a 256-byte status block first.
//   int[0] status code (0 = ok), int[1] where, int[2] block
//   int[16] query-summary ticket counter of the groups (self-resetting)
//   int[17] debug flag that nothing sets
//   int[18] selection: query summary published (generation, counts up)
//   int[19] selection: CTAs done scoring (counts up)
//   int[32..32+kQbarBlocks/8) query-summary ticket counters within each group
constexpr size_t kStatusBytes = 256;
constexpr int kTicketIdx = 16;
constexpr int kDebugFlagIdx = 17;
constexpr int kSelQbarGenIdx = 18;      // query summary published (generation counter)
constexpr int kSelScoreCntIdx = 19;     // CTAs done scoring (monotonic counter)
constexpr int kGroupTicketIdx = 32;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Runs `fn` (a cudaFuncSetAttribute call) once per device.  Kernel attributes
// belong to a device, so a process-wide flag would leave a second device
// without them; the mutex keeps concurrent first calls from racing.
struct PerDeviceOnce {
  std::mutex mu;
  uint64_t done[2] = {0, 0};            // one bit per device ordinal < 128
};
template <class F>
cudaError_t once_per_device(PerDeviceOnce& once, F&& fn) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return fn();
  std::lock_guard<std::mutex> lock(once.mu);
  const uint64_t bit = 1ull << (dev & 63);
  if (once.done[dev >> 6] & bit) return cudaSuccess;
  e = fn();
  if (e == cudaSuccess) once.done[dev >> 6] |= bit;
  return e;
}

// Where-codes recorded with a device error (status int[1]).
enum Where : int {
  kWhereReps = 10,
  kWhereTopk = 20,
  kWhereSelect = 21,
  kWhereFwdProducer = 30,
  kWhereFwdMma = 31,
  kWhereFwdSoftmax = 32,
  kWhereBwdProducer = 40,
  kWhereBwdMma = 41,
  kWhereBwdCompute = 42,
  kWhereBwdEpilogue = 43,
  kWhereFp32 = 50,
  kWhereTailRows = 60,
  kWhereDebug = 90,
};

struct KvDesc {
  const void* k;
  const void* v;
  void* dk;
  void* dv;
  const int32_t* page_table;
  int num_pages, num_slots, page_size, hkv, head_dim;
};

// --- k_reps_select.cu
// last_rows: rows of the last page of the range that hold keys (P: whole pages)
cudaError_t launch_page_reps(const KvDesc& kv, bool bf16, int first_page, int n_pages,
                             int last_rows, float* reps, int* status, cudaStream_t st);
size_t select_ws_bytes(int num_pages, int hkv, int head_dim);
cudaError_t launch_select_topk(const void* q, bool bf16, int hq, int chunk_len, int n_cand,
                               const float* reps, int num_pages, int hkv, int head_dim, int top_k,
                               int32_t* sel, float* scores_opt, void* ws, uint64_t wait_ns,
                               cudaStream_t st);
// The selection with its scratch in a fixed device array of the library
// (oomb_select_topk_noalloc); sets *too_big when the shapes need more.
cudaError_t launch_select_topk_noalloc(const void* q, bool bf16, int hq, int chunk_len,
                                       int n_cand, const float* reps, int num_pages, int hkv,
                                       int head_dim, int top_k, int32_t* sel, float* scores_opt,
                                       bool* too_big, uint64_t wait_ns, cudaStream_t st);
cudaError_t launch_validate_page_table(const int32_t* pt, int num_pages, int num_slots,
                                       uint32_t* bitmap, int* status, cudaStream_t st);
// bf16 pools: raises kStatusNonFinite when a K or V entry in rows [valid_rows, P)
// of logical page `page` is inf or NaN.
cudaError_t launch_check_tail_rows(const KvDesc& kv, int page, int valid_rows, int* status,
                                   cudaStream_t st);
cudaError_t launch_debug_wait(int* status, uint64_t limit_ns, cudaStream_t st);

// --- k_attn_fp32.cu
size_t fp32_bwd_ws_bytes(int hq, int chunk_len);
cudaError_t launch_attn_fwd_fp32(const float* q, const KvDesc& kv, const int32_t* sel, int n_sel,
                                 int hq, int chunk_len, int chunk_start, float scale, float* o,
                                 float* lse, int* status, cudaStream_t st);
cudaError_t launch_attn_bwd_fp32(const float* q, const float* o, const float* dout,
                                 const float* lse, const KvDesc& kv, const int32_t* sel,
                                 int n_sel, int hq, int chunk_len, int chunk_start, float scale,
                                 float* dq, void* ws, cudaStream_t st);

// --- k_attn_fwd_bf16.cu
// own_reps: if not null, the representatives of the chunk's own pages are
// also written there (rows of the logical pages, [num_pages][hkv][128]).
// o_lo: if not null, the rounding residual of o (bf16(o32 - bf16(o32))).
cudaError_t launch_attn_fwd_bf16(const void* q, const KvDesc& kv, const int32_t* sel, int n_sel,
                                 int hq, int chunk_len, int chunk_start, float scale, void* o,
                                 void* o_lo, float* lse, float* own_reps, int* status,
                                 uint64_t wait_ns, cudaStream_t st);

// --- k_attn_bwd_bf16.cu
size_t bf16_bwd_ws_bytes(int hq, int chunk_len, int head_dim);
// o_lo: the forward's residual of o (or null): Delta = dout . (o + o_lo).
cudaError_t launch_attn_bwd_bf16(const void* q, const void* o, const void* o_lo,
                                 const void* dout, const float* lse, const KvDesc& kv,
                                 const int32_t* sel, int n_sel, int hq, int chunk_len,
                                 int chunk_start, float scale, void* dq, void* ws,
                                 uint64_t wait_ns, cudaStream_t st);

}  // namespace oomb
