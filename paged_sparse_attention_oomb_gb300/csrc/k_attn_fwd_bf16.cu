// Step 3 of the path: forward of page-level sparse causal attention, bf16 in,
// fp32 accumulate, on the 5th-generation tensor cores (tcgen05 + TMEM).
// Method: "Out of the Memory Barrier" technical summary, section 2, item
// "Page-level Sparse Attention": the chunk attends the pages chosen by their
// representative vectors plus its own pages.
//
// One CTA computes one 128-row query tile of one query head over its key
// tiles -- first the selected pages (ceil(n_sel * P / 128) tiles, masked only
// in a ragged last tile), then the chunk's own pages up to the diagonal.  The
// scores of three consecutive key tiles live in three TMEM buffers, so the
// MMA S(j+2) = Q K_{j+2}^T only waits for O += P(j-1) V_{j-1} -- an MMA issued
// one tile earlier -- and the softmax of tile j+1 can follow the softmax of
// tile j without waiting for the O update of tile j.  Roles (352 threads):
//   warp 0      TMA producer: Q once; then K_j, V_j page by page through the
//               page table (one 2-D box per page and 64-column half) into a
//               6-slot shared ring; also allocates TMEM.
//   warp 10     issues S(j) = Q K_j^T into buffer j % 3 (SS), j = 0, 1, ...,
//               each once the O update that last read the buffer is done;
//   warp 1      issues O += P(j) V_j, P(j) in buffer j % 3 (P from TMEM), each
//               once P(j) is ready.  (Each a whole warp in lockstep, one
//               elected lane issues.)  tcgen05.mma blocks its issuing thread
//               while the tensor pipe's queue is full; with two issuing warps
//               an O update waiting on the softmax never holds back the next
//               score MMA, and the reverse.
//   warps 2..9  softmax, two threads per query row (warps w and w + 4 share a
//               TMEM lane quarter and split the 128 key columns): the half row
//               of S is read from TMEM into registers once, the row maximum is
//               completed through shared memory, exponentials in base 2, P
//               written back over S as bf16 pairs.  O is rescaled in TMEM
//               only when a row maximum grows by more than 2^8 (the final
//               normalisation uses the same running maximum, so this is
//               exact); the rescale first waits for the previous O update.
// TMEM (512 columns allocated): S0 [0,128), S1 [128,256), S2 [256,384),
// O [384,512).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "oomb_internal.h"
#include "sm100.cuh"
#include "tmap.h"

namespace oomb {
namespace {

constexpr int kThreads = 352;
constexpr int kSWarp = 10;                      // issues S(j) = Q K_j^T
constexpr int kSoftmaxThreads = 256;
constexpr int kSlots = 6;                         // K/V ring (3 key tiles)
constexpr int kSBufs = 3;                         // score buffers in TMEM
constexpr uint32_t kQOff = 0;
constexpr uint32_t kRingOff = kTileBytes;
constexpr uint32_t kBarOff = kRingOff + kSlots * kTileBytes;
constexpr uint32_t kXchgOff = kBarOff + 256;      // row-max / row-sum exchange [2][4][2][32] floats
constexpr uint32_t kSmemBytes = kXchgOff + 2 * 4 * 2 * 32 * 4;  // base is 1024-aligned
constexpr uint32_t kOCol = 384;
constexpr float kRescaleThreshold = 8.0f;         // log2 units

struct Bars {
  uint64_t q_full;
  uint64_t slot_full[kSlots], slot_empty[kSlots];
  // pv_done[b]: the O update that read buffer b is complete.  One barrier per
  // buffer keeps every waiter at most one phase ahead of the barrier it tests
  // (a single barrier could lag two O updates behind a waiter, and a parity
  // test two phases ahead reads as complete).
  uint64_t s_full[kSBufs], p_ready[kSBufs], pv_done[kSBufs];
  uint64_t pair[4];           // the two softmax warps of a TMEM lane quarter
  uint64_t drain, drain_s;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct FwdParams {
  const int32_t* sel;
  const int32_t* pt;
  __nv_bfloat16* o;
  __nv_bfloat16* o_lo;                 // rounding residual of o, or null
  float* lse;
  float* reps;                         // own-page representatives, or null
  int* status;
  int n_sel, hq, hkv, page_size, chunk_len, chunk_start, num_slots;
  int n_qtiles, t_sel;                 // query tiles, selected key tiles
  float scale_log2;
  uint64_t wait_ns;
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, const uint64_t* field,
                                             const Bars* b) {
  return base + static_cast<uint32_t>(reinterpret_cast<const char*>(field) -
                                      reinterpret_cast<const char*>(b));
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  const uint32_t bbase = sbase + kBarOff;
#define BAR(f) bar_addr(bbase, &bars->f, bars)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (sbase & 1023u) {          // the swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) raise_status(p.status, kStatusBounds, kWhereFwdProducer);
    return;
  }
  // heaviest query tiles (most own key tiles) first
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x) / p.hq;
  const int h = static_cast<int>(blockIdx.x) % p.hq;
  const int g = h / (p.hq / p.hkv);
  const int n_tiles = p.t_sel + qt + 1;            // key tiles of this query tile
  const int ppt = 128 / p.page_size;               // pages per key tile
  const int own_page0 = p.chunk_start / p.page_size;
  // the chunk's own pages; the last one may be partial (rows past the chunk's
  // end hold no token: the causal mask never reaches them)
  const int n_own_pages = (p.chunk_len + p.page_size - 1) / p.page_size;

  if (threadIdx.x == 0) {
    mbar_init(BAR(q_full), 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(BAR(slot_full[i]), 1);
      mbar_init(BAR(slot_empty[i]), 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(BAR(s_full[i]), 1);
      mbar_init(BAR(p_ready[i]), kSoftmaxThreads);
      mbar_init(BAR(pv_done[i]), 1);
    }
    for (int i = 0; i < 4; ++i) mbar_init(BAR(pair[i]), 64);
    mbar_init(BAR(drain), 1);
    mbar_init(BAR(drain_s), 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{p.status, &bars->abort_flag, p.wait_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop in lockstep; one elected lane issues.
    const bool leader = elect_one();
    if (leader) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(BAR(q_full), kTileBytes);
      for (int hf = 0; hf < 2; ++hf)
        tma_load_3d(sbase + kQOff + hf * kHalfBytes, &tm_q, BAR(q_full), hf * 64, h, qt * 128);
    }
    __syncwarp();
    const int32_t* sel_g = p.sel + static_cast<long>(g) * p.n_sel;
    int issued = 0;                                // ring loads issued (K_0, V_0, K_1, ...)
    // Page lookups run ahead of the loads that need them, in three stages one
    // key tile apart: the selection entry of tile j+2, then the page table
    // entry of tile j+1, then the row of tile j -- each load's value is first
    // used a tile later, so its latency hides behind a tile's work.  Lane u
    // (< pages per tile) resolves page u of a tile.  An entry out of range is
    // recorded when its tile is loaded, and never followed (row 0 instead).
    const bool my_page = lane < ppt;
    auto sel_raw = [&](int j) -> int {             // stage A: selection entry
      if (!my_page || j >= n_tiles || j >= p.t_sel) return 0;
      const int pi = j * ppt + lane;
      return sel_g[pi < p.n_sel ? pi : 0];
    };
    auto page_of = [&](int j, int raw, bool* bad) -> int {   // stage B: logical page
      *bad = false;
      if (!my_page || j >= n_tiles) return own_page0;
      if (j < p.t_sel) {
        if (raw < 0 || raw >= own_page0) {
          *bad = true;
          return own_page0;
        }
        return raw;
      }
      const int lp = own_page0 + (j - p.t_sel) * ppt + lane;
      return lp < own_page0 + n_own_pages ? lp : own_page0;
    };
    bool bad_b;
    int slot_b = p.pt[page_of(0, sel_raw(0), &bad_b)];        // tile 0, stages A and B
    int raw_a = sel_raw(1);                                     // tile 1, stage A
    for (int j = 0; j < n_tiles; ++j) {
      const int slot = slot_b;                                  // tile j (stage C)
      const bool bad_lp = bad_b;
      const int lp_next = page_of(j + 1, raw_a, &bad_b);        // tile j+1 (stage B)
      slot_b = (my_page && j + 1 < n_tiles) ? p.pt[lp_next] : 0;
      raw_a = sel_raw(j + 2);                                   // tile j+2 (stage A)
      const bool bad = my_page && (bad_lp || slot < 0 || slot >= p.num_slots);
      if (__any_sync(0xffffffffu, bad)) raise_status(p.status, kStatusBounds, kWhereFwdProducer);
      const int row = (my_page && !bad) ? (slot * p.hkv + g) * p.page_size : 0;
      int rows[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) rows[u] = __shfl_sync(0xffffffffu, row, u);
      bool ok = true;
      for (int kv = 0; kv < 2 && ok; ++kv) {
        const int q = 2 * j + kv;
        const int sl = q % kSlots;
        const uint32_t phe = ((q / kSlots) & 1) ^ 1;
        if (!(ok = mbar_wait(BAR(slot_empty[sl]), phe, wc, kWhereFwdProducer))) break;
        const uint32_t dst = sbase + kRingOff + sl * kTileBytes;
        if (leader) {
          mbar_arrive_expect_tx(BAR(slot_full[sl]), kTileBytes);
          for (int u = 0; u < ppt; ++u)
            for (int hf = 0; hf < 2; ++hf)
              tma_load_2d(dst + hf * kHalfBytes + u * p.page_size * 128, kv ? &tm_v : &tm_k,
                          BAR(slot_full[sl]), hf * 64, rows[u]);
        }
        __syncwarp();
        ++issued;
      }
      if (!ok) break;
    }
    if (p.reps != nullptr && h % (p.hq / p.hkv) == 0 && !bars->abort_flag) {
      // Step 1 for the chunk's own pages, from the K tile already in shared
      // memory: the last key tile of this CTA is own tile qt, and the first
      // query head of each group writes the representatives of its pages.
      // Same summation order as page_reps_kernel (16 row groups, rows
      // rg, rg + 16, ... in order, then the groups in order), so the values
      // are bit-identical to a separate representatives pass.
      const int q = 2 * (n_tiles - 1);
      const int sl = q % kSlots;
      if (mbar_wait(BAR(slot_full[sl]), (q / kSlots) & 1, wc, kWhereFwdProducer)) {
        const uint32_t tile = sbase + kRingOff + sl * kTileBytes;
        // this lane's 4 columns [4 lane, 4 lane + 4): half, 16-byte chunk, offset in chunk
        const uint32_t col_off = (lane >> 4) * kHalfBytes + (lane & 1) * 8;
        const int chunk = (lane & 15) >> 1;
        for (int u = 0; u < ppt; ++u) {
          const int op = qt * ppt + u;                 // own page index in the chunk
          if (op >= n_own_pages) break;
          // rows of the page that hold the chunk's keys (fewer on a partial page)
          const int n_rows = min(p.page_size, p.chunk_len - op * p.page_size);
          const float inv = 1.0f / static_cast<float>(n_rows);
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
          for (int rg = 0; rg < 16; ++rg) {
            float a4[4] = {0.f, 0.f, 0.f, 0.f};
            for (int rr = rg; rr < n_rows; rr += 16) {
              const int row = u * p.page_size + rr;
              const uint32_t addr = tile + col_off + row * 128 + ((chunk ^ (row & 7)) << 4);
              uint32_t w0, w1;
              asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(addr));
              a4[0] += __uint_as_float(w0 << 16);
              a4[1] += __uint_as_float(w0 & 0xFFFF0000u);
              a4[2] += __uint_as_float(w1 << 16);
              a4[3] += __uint_as_float(w1 & 0xFFFF0000u);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) s4[e] += a4[e];
          }
          float4* dst = reinterpret_cast<float4*>(
              p.reps + (static_cast<long>(own_page0 + op) * p.hkv + g) * 128) + lane;
          *dst = make_float4(s4[0] * inv, s4[1] * inv, s4[2] * inv, s4[3] * inv);
        }
      }
    }
    if (bars->abort_flag) {
      // unwinding: let every copy this warp issued land before the CTA exits
      mbar_drain_wait(BAR(q_full), 0);
      for (int sl = 0; sl < kSlots; ++sl) {
        int last = -1;
        for (int q = sl; q < issued; q += kSlots) last = q;
        if (last >= 0) mbar_drain_wait(BAR(slot_full[sl]), (last / kSlots) & 1);
      }
    }
  } else if (warp == 1 || warp == kSWarp) {
    // ------------------------------------------------------------ MMA issuers
    // Each issuing warp runs its loop in lockstep (its decisions are
    // warp-uniform); one elected lane issues the MMAs and their commits.  A
    // commit tracks the MMAs of its own thread, so s_full is committed by the
    // S warp and pv_done by the O-update warp.
    constexpr uint32_t kIdQK = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdPV = idesc_bf16_f32(128, 128, false, true);
    const uint64_t d0 = desc_kmajor0(sbase);
    const uint64_t dQ = d0 + desc_off(kQOff);
    const uint64_t dRing_k = d0 + desc_off(kRingOff), dRing_mn = d0 + kDescMn + desc_off(kRingOff);
    const bool s_role = warp == kSWarp;
    bool ok = !s_role || mbar_wait_spin(BAR(q_full), 0, wc, kWhereFwdMma);
    // S(j) = Q K_j^T into buffer j % 3.  The buffer last held P(j-3), read by
    // the O update of tile j-3, which must be complete.
    auto issue_s = [&](int j) -> bool {
      const int sk = (2 * j) % kSlots, b = j % kSBufs;
      if (!mbar_wait_spin(BAR(slot_full[sk]), ((2 * j) / kSlots) & 1, wc, kWhereFwdMma))
        return false;
      if (j >= kSBufs && !mbar_wait_spin(BAR(pv_done[b]), ((j - kSBufs) / kSBufs) & 1, wc,
                                         kWhereFwdMma))
        return false;
      tc_fence_after();
      const uint64_t qa = opaque(dQ), ka = opaque(dRing_k + sk * kTileDesc);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + b * 128, qa + kstep_kmajor(kk), ka + kstep_kmajor(kk), kIdQK, kk > 0);
        umma_commit(BAR(s_full[b]));
        umma_commit(BAR(slot_empty[sk]));
      }
      __syncwarp();
      return true;
    };
    // O += P(j) V_j  (P(j) in buffer j % 3 as bf16 pairs, 8 columns per k-step;
    // keys [64 c, 64 c + 64) sit at buffer columns [64 c, 64 c + 32))
    auto issue_pv = [&](int j) -> bool {
      const int sv = (2 * j + 1) % kSlots, b = j % kSBufs;
      if (!mbar_wait_spin(BAR(slot_full[sv]), ((2 * j + 1) / kSlots) & 1, wc, kWhereFwdMma))
        return false;
      if (!mbar_wait_spin(BAR(p_ready[b]), (j / kSBufs) & 1, wc, kWhereFwdMma)) return false;
      tc_fence_after();
      const uint64_t va = opaque(dRing_mn + sv * kTileDesc);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tmem + kOCol, tmem + b * 128 + 64 * (kk >> 2) + 8 * (kk & 3),
                  va + kstep_mnmajor(kk), kIdPV, (j > 0 || kk > 0));
        umma_commit(BAR(pv_done[b]));
        umma_commit(BAR(slot_empty[sv]));
      }
      __syncwarp();
      return true;
    };
    if (s_role) {
      for (int j = 0; ok && j < n_tiles; ++j) ok = issue_s(j);
    } else {
      for (int j = 0; ok && j < n_tiles; ++j) ok = issue_pv(j);
    }
    if (!ok) {
      if (elect_one()) umma_commit(s_role ? BAR(drain_s) : BAR(drain));
      __syncwarp();
      mbar_drain_wait(s_role ? BAR(drain_s) : BAR(drain), 0);
    }
  } else if (warp < kSWarp) {
    // ------------------------------------------------------------ softmax
    // Two warps per TMEM lane quarter (the same 32 query rows): warp half
    // ch = 0 takes key columns [0, 64), ch = 1 columns [64, 128).  Their
    // partial row maxima (and at the end their partial row sums) meet in
    // shared memory behind a per-quarter mbarrier (bounded waits).
    const int q4 = warp & 3;
    const int ch = (warp - 2) >> 2;
    const int r = q4 * 32 + lane;                  // row of the query tile
    const int t = qt * 128 + r;                    // chunk row
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t t_o = tmem + lane_base + kOCol + 64 * ch;   // this warp's O columns
    float* xchg = reinterpret_cast<float*>(smem + kXchgOff);  // [2][4][2][32]
    auto slot = [&](int par, int c) -> float* { return xchg + ((par * 4 + q4) * 2 + c) * 32 + lane; };
    float m = -INFINITY, l = 0.f;                  // l: this warp's partial row sum
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j % kSBufs;
      const uint32_t t_s = tmem + lane_base + b * 128 + 64 * ch;
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(s_full[b]), (j / kSBufs) & 1, wc, kWhereFwdSoftmax));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld64(t_s, sr);
      // valid key columns are [0, lim); `masked` is uniform over the warp
      int lim = 128;
      bool masked = false;
      if (j < p.t_sel) {
        const int rem = (p.n_sel - j * ppt) * p.page_size;
        if (rem < 128) {
          lim = rem;
          masked = true;
        }
      } else if (j - p.t_sel == qt) {
        lim = r + 1;
        masked = true;
      }
      if (masked) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (64 * ch + c >= lim) sr[c] = __float_as_uint(-INFINITY);
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        mx[i] = fmax3(__uint_as_float(sr[i]), __uint_as_float(sr[8 + i]),
                      __uint_as_float(sr[16 + i]));
#pragma unroll
      for (int c = 24; c < 56; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          mx[i] = fmax3(mx[i], __uint_as_float(sr[c + i]), __uint_as_float(sr[c + 8 + i]));
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = fmaxf(mx[i], __uint_as_float(sr[56 + i]));
      const float mp = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                             fmaxf(mx[6], mx[7]));
      // exchange the partial maxima of the row with the other half
      *slot(j & 1, ch) = mp;
      mbar_arrive(BAR(pair[q4]));
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(pair[q4]), j & 1, wc, kWhereFwdSoftmax));
      if (!ok) break;
      const float mt = fmaxf(mp, *slot(j & 1, ch ^ 1)) * p.scale_log2;
      // lazy rescale: m moves only when the row maximum grows by more than 2^8
      // (both halves take the same decision from the same row maximum)
      float alpha = 1.f;
      bool any_need = false;
      if (j == 0) {
        m = mt;
      } else {
        const float m_new = fmaxf(m, mt);
        const bool need = m_new > m + kRescaleThreshold;
        any_need = __any_sync(0xffffffffu, need);
        if (need) {
          alpha = ex2(m - m_new);
          m = m_new;
        }
      }
      // P = exp2(s * scale_log2 - m) -> bf16 pairs into this warp's first 32
      // columns (S is already in registers); the scaling and the 8 partial row
      // sums on packed FP32 pairs
      const float neg_m = -m;
      const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nm2 = f2_pack(neg_m, neg_m);
      uint64_t rs2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) rs2[i] = 0ull;
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), sc2, nm2),
                  x0, x1);
        const float e0 = ex2(x0), e1 = ex2(x1);
        rs2[(i >> 1) & 3] = f2_add(rs2[(i >> 1) & 3], f2_pack(e0, e1));
        pk[i >> 1] = pack_bf16(e0, e1);
      }
      float rs[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) f2_unpack(rs2[i], rs[2 * i], rs[2 * i + 1]);
      tmem_st32(t_s, pk);
      if (any_need) {
        // O must be stable: wait for the O update of tile j-1 (the one of tile j
        // waits for this thread's p_ready)
        const int jp = j - 1;
        ok = __all_sync(0xffffffffu, mbar_wait(BAR(pv_done[jp % kSBufs]), (jp / kSBufs) & 1, wc,
                                               kWhereFwdSoftmax));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t rr[32];
          tmem_ld32(t_o + c2 * 32, rr);
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
          tmem_st32(t_o + c2 * 32, rr);
        }
      }
      tmem_st_wait();
      l = l * alpha + (((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7])));
      tc_fence_before();
      mbar_arrive(BAR(p_ready[b]));
    }
    if (ok && n_tiles > 0) {
      const int jl = n_tiles - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(pv_done[jl % kSBufs]), (jl / kSBufs) & 1, wc,
                                             kWhereFwdSoftmax));
    }
    if (ok && n_tiles > 0) {
      // full row sum from the two halves (one more phase of the pair barrier)
      *slot(n_tiles & 1, ch) = l;
      mbar_arrive(BAR(pair[q4]));
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(pair[q4]), n_tiles & 1, wc, kWhereFwdSoftmax));
    }
    if (ok && n_tiles > 0) {
      tc_fence_after();
      const float lt = l + *slot(n_tiles & 1, ch ^ 1);
      const float inv = 1.f / lt;
      const bool row_ok = t < p.chunk_len;
      const long row_off = (static_cast<long>(t) * p.hq + h) * 128 + 64 * ch;
      uint4* orow = reinterpret_cast<uint4*>(p.o + row_off);
      uint4* lrow = p.o_lo ? reinterpret_cast<uint4*>(p.o_lo + row_off) : nullptr;
#pragma unroll 1
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t rr[32];
        tmem_ld32(t_o + c2 * 32, rr);
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float a = __uint_as_float(rr[8 * i + 2 * k]) * inv;
              const float b = __uint_as_float(rr[8 * i + 2 * k + 1]) * inv;
              hi[k] = pack_bf16(a, b);
              // what the rounding dropped (exact in fp32), itself rounded to bf16
              lo[k] = pack_bf16(a - __uint_as_float(hi[k] << 16),
                                b - __uint_as_float(hi[k] & 0xFFFF0000u));
            }
            orow[c2 * 4 + i] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            if (lrow) lrow[c2 * 4 + i] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
      }
      if (row_ok && ch == 0)
        p.lse[static_cast<long>(h) * p.chunk_len + t] = (m + __log2f(lt)) * 0.69314718055994530942f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
#undef BAR
}

}  // namespace

cudaError_t launch_attn_fwd_bf16(const void* q, const KvDesc& kv, const int32_t* sel, int n_sel,
                                 int hq, int chunk_len, int chunk_start, float scale, void* o,
                                 void* o_lo, float* lse, float* own_reps, int* status,
                                 uint64_t wait_ns, cudaStream_t st) {
  CUtensorMap tq, tk, tv;
  {
    const uint64_t dims[3] = {128, static_cast<uint64_t>(hq), static_cast<uint64_t>(chunk_len)};
    const uint64_t strides[2] = {128 * 2, static_cast<uint64_t>(hq) * 128 * 2};
    const uint32_t box[3] = {64, 1, 128};
    if (!make_tmap_bf16(&tq, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t rows = static_cast<uint64_t>(kv.num_slots) * kv.hkv * kv.page_size;
    const uint64_t dims[2] = {128, rows};
    const uint64_t strides[1] = {128 * 2};
    const uint32_t box[2] = {64, static_cast<uint32_t>(kv.page_size)};
    if (!make_tmap_bf16(&tk, kv.k, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tv, kv.v, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  FwdParams p;
  p.sel = sel;
  p.pt = kv.page_table;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.o_lo = static_cast<__nv_bfloat16*>(o_lo);
  p.lse = lse;
  p.reps = own_reps;
  p.status = status;
  p.n_sel = n_sel;
  p.hq = hq;
  p.hkv = kv.hkv;
  p.page_size = kv.page_size;
  p.chunk_len = chunk_len;
  p.chunk_start = chunk_start;
  p.num_slots = kv.num_slots;
  p.n_qtiles = (chunk_len + 127) / 128;
  p.t_sel = (n_sel * kv.page_size + 127) / 128;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_ns = wait_ns;
  static PerDeviceOnce attr;
  {
    cudaError_t e = once_per_device(attr, [] {
      return cudaFuncSetAttribute(sparse_attn_fwd_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (e != cudaSuccess) return e;
  }
  sparse_attn_fwd_kernel<<<p.n_qtiles * hq, kThreads, kSmemBytes, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace oomb
