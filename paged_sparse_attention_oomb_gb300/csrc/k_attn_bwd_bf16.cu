// Step 4 of the path: backward of page-level sparse causal attention on the
// tcgen05 tensor cores, with the dK/dV accumulation into the paged gradient
// buffers fused into the tile loop.
// Method: "Out of the Memory Barrier" technical summary, section 2: "Paged
// Memory Management" (KV gradients live in pages and are accumulated in place
// outside autograd), "Page-level Sparse Attention" (the backward reuses the
// forward's page choice), "Chunk-Recurrent Training Framework" (the backward
// recomputes what the forward discarded).
//
// One CTA owns one 128-key tile of one KV head: a tile of selected pages
// (attended by every query tile of the chunk) or of the chunk's own pages
// (attended by the query tiles at or after it).  It loops over the G query
// heads of the group x the query tiles that see it.  Iteration n:
//   MMA1  S^T  = K Q^T                 TMEM R0 (keys on lanes, queries on columns)
//   MMA2  dP^T = V dO^T                TMEM R1
//   P^T = exp2(S^T * scale*log2e - lse2)   -> bf16 pairs, back into R0 (TMEM)
//   MMA3  dV  += P^T dO                A from TMEM (R0), B = dO (shared)
//   dS^T = P^T (dP^T - Delta)           -> bf16 into a swizzled shared tile
//                                      (the softmax scale is applied to dK in the
//                                      epilogue and to dQ when it is converted)
//   MMA4  dK  += dS^T Q                TMEM R3
//   MMA5  dQ^T = K^T dS^T              TMEM R1 (head dim on lanes), drained with
//                                      coalesced fp32 reductions
// Q (+ its lse2/Delta rows) and dO tiles stream through a 2-stage TMA ring.
// The compute warps keep P^T in registers for the dS pass, so R0 is free as
// soon as MMA3 has read it: the issue order is dP^T(n), dV(n), S^T(n+1),
// dK(n), dQ^T(n), and the exponentials of n+1 follow the dS pass of n without
// waiting for dK/dQ of n.
// At the end the CTA adds dK and dV to the bf16 gradient pages of its slots:
// one read-add-write and one rounding per slot per call, no atomics, because
// each (slot, KV head) has exactly one owner CTA.
// Roles (512 threads, four warpgroups): warp 0 TMA producer + TMEM allocator,
// warp 1 MMA issuer (polls its barriers: its wake-up latency is on the
// critical path), warps 2..3 idle; warps 4..11 compute P^T and dS^T (TMEM lane
// quarter = warp % 4; the two warps of a quarter split the 128 columns); warps
// 12..15 drain dQ^T: each thread copies its whole TMEM lane (128 columns) into
// registers, releases R1 for the next dP^T at once, and only then issues the
// fp32 reductions, so neither the tensor pipe nor the compute warps wait on
// them.  The drain warpgroup takes the registers this needs from the
// producer/MMA warpgroup (setmaxnreg: 72 + 2 x 128 + 184 per thread = the
// 128 per thread the block is launched with).
// TMEM: R0 [0,128) S^T / P^T, R1 [128,256) dP^T / dQ, R2 [256,384) dV,
// R3 [384,512) dK.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "oomb_internal.h"
#include "sm100.cuh"
#include "tmap.h"

namespace oomb {
namespace {

constexpr int kThreads = 512;
constexpr int kComputeThreads = 256;              // warps 4..11: P^T and dS^T
constexpr int kDrainThreads = 128;                // warps 12..15: dQ^T out of TMEM
constexpr uint32_t kKOff = 0;
constexpr uint32_t kVOff = kTileBytes;
constexpr uint32_t kQOff = 2 * kTileBytes;        // 2 stages
constexpr uint32_t kDOOff = 4 * kTileBytes;       // 2 stages
constexpr uint32_t kDSOff = 6 * kTileBytes;
constexpr uint32_t kVecOff = 7 * kTileBytes;      // per stage: lse2[128], delta[128]
constexpr uint32_t kBarOff = kVecOff + 2 * 1024;
constexpr uint32_t kSmemBytes = kBarOff + 256;    // base is 1024-aligned by declaration

struct Bars {
  uint64_t kv_full;
  uint64_t q_full[2], q_empty[2];
  uint64_t do_full[2], do_empty[2];
  uint64_t s_full, dp_full, dq_full;
  uint64_t p_ready, ds_ready, r1_free;
  uint64_t pt_consumed, ds_free;
  uint64_t acc_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct BwdParams {
  const int32_t* sel;
  const int32_t* pt;
  const float* lse2;       // [hq][n_qtiles*128]  lse * log2(e); +inf on padding rows
  const float* delta;      // [hq][n_qtiles*128]  0 on padding rows
  float* dq_acc;           // [chunk_len][hq][128]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* status;
  int n_sel, hq, hkv, page_size, chunk_len, chunk_start, num_slots;
  int n_qtiles, t_sel;
  float scale, scale_log2;
  uint64_t wait_ns;
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t base, const uint64_t* field,
                                             const Bars* b) {
  return base + static_cast<uint32_t>(reinterpret_cast<const char*>(field) -
                                      reinterpret_cast<const char*>(b));
}

__device__ __forceinline__ uint32_t bf16x2_add(uint32_t old2, float a, float b) {
  const float lo = __uint_as_float(old2 << 16) + a;
  const float hi = __uint_as_float(old2 & 0xFFFF0000u) + b;
  return pack_bf16(lo, hi);
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_do,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  const uint32_t bbase = sbase + kBarOff;
  const float* vec = reinterpret_cast<const float*>(smem + kVecOff);
#define BAR(f) bar_addr(bbase, &bars->f, bars)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (sbase & 1023u) {          // the swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) raise_status(p.status, kStatusBounds, kWhereBwdProducer);
    return;
  }
  const int g = static_cast<int>(blockIdx.x) % p.hkv;
  const int kt = static_cast<int>(blockIdx.x) / p.hkv;     // selected tiles first
  const bool is_sel = kt < p.t_sel;
  const int own_t = kt - p.t_sel;                          // own key tile index
  const int grp = p.hq / p.hkv;
  const int i0 = is_sel ? 0 : own_t;                       // first query tile that sees it
  const int nq = p.n_qtiles - i0;
  const int n_iter = grp * nq;
  const int ppt = 128 / p.page_size;
  const int own_page0 = p.chunk_start / p.page_size;
  // the last own page may be partial: its rows past the chunk are masked as keys
  // (key_valid) and their gradient rows are left as they are
  const int n_own_pages = (p.chunk_len + p.page_size - 1) / p.page_size;
  const int padded = p.n_qtiles * 128;
  const int32_t* sel_g = p.sel + static_cast<long>(g) * p.n_sel;

  if (threadIdx.x == 0) {
    mbar_init(BAR(kv_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(q_full[i]), 1);
      mbar_init(BAR(q_empty[i]), 1);
      mbar_init(BAR(do_full[i]), 1);
      mbar_init(BAR(do_empty[i]), 1);
    }
    mbar_init(BAR(s_full), 1);
    mbar_init(BAR(dp_full), 1);
    mbar_init(BAR(dq_full), 1);
    mbar_init(BAR(p_ready), kComputeThreads);
    mbar_init(BAR(ds_ready), kComputeThreads);
    mbar_init(BAR(r1_free), kDrainThreads);
    mbar_init(BAR(pt_consumed), 1);
    mbar_init(BAR(ds_free), 1);
    mbar_init(BAR(acc_done), 1);
    mbar_init(BAR(drain), 1);
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

  // Logical page of page-slot u of this key tile, and whether its keys are real.
  auto tile_page = [&](int u, bool* valid) -> int {
    if (is_sel) {
      const int pi = kt * ppt + u;
      *valid = pi < p.n_sel;
      return sel_g[pi < p.n_sel ? pi : 0];
    }
    const int lp = own_page0 + own_t * ppt + u;
    *valid = lp < own_page0 + n_own_pages;
    return *valid ? lp : own_page0;
  };

  if (warp < 4) {
    regs_decrease<72>();            // producer / MMA warpgroup gives registers to the drain
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop in lockstep; one elected lane issues.
    {
      const bool leader = elect_one();
      if (leader) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_arrive_expect_tx(BAR(kv_full), 2 * kTileBytes);
      }
      for (int u = 0; u < ppt; ++u) {
        bool valid;
        int lp = tile_page(u, &valid);
        if (lp < 0 || (is_sel && lp >= own_page0)) {
          raise_status(p.status, kStatusBounds, kWhereBwdProducer);
          lp = own_page0;
        }
        int slot = p.pt[lp];
        if (slot < 0 || slot >= p.num_slots) {
          raise_status(p.status, kStatusBounds, kWhereBwdProducer);
          slot = 0;
        }
        const int row = (slot * p.hkv + g) * p.page_size;
        if (leader) {
          for (int hf = 0; hf < 2; ++hf) {
            const uint32_t off = hf * kHalfBytes + u * p.page_size * 128;
            tma_load_2d(sbase + kKOff + off, &tm_k, BAR(kv_full), hf * 64, row);
            tma_load_2d(sbase + kVOff + off, &tm_v, BAR(kv_full), hf * 64, row);
          }
        }
        __syncwarp();
      }
      int nq_issued = 0, ndo_issued = 0;
      for (int n = 0; n < n_iter; ++n) {
        const int h = g * grp + n / nq;
        const int qi = i0 + n % nq;
        const int s = n & 1;
        const uint32_t phe = ((n >> 1) & 1) ^ 1;
        // Q with its lse2 and Delta rows (read by the P and dS passes; the stage
        // is released after dK, which follows the dS pass)
        if (!mbar_wait(BAR(q_empty[s]), phe, wc, kWhereBwdProducer)) break;
        const uint32_t vb = sbase + kVecOff + s * 1024;
        const long voff = static_cast<long>(h) * padded + qi * 128;
        if (leader) {
          mbar_arrive_expect_tx(BAR(q_full[s]), kTileBytes + 1024);
          tma_load_3d(sbase + kQOff + s * kTileBytes, &tm_q, BAR(q_full[s]), 0, h, qi * 128);
          tma_load_3d(sbase + kQOff + s * kTileBytes + kHalfBytes, &tm_q, BAR(q_full[s]), 64, h,
                      qi * 128);
          bulk_load(vb, p.lse2 + voff, 512, BAR(q_full[s]));
          bulk_load(vb + 512, p.delta + voff, 512, BAR(q_full[s]));
        }
        __syncwarp();
        ++nq_issued;
        if (!mbar_wait(BAR(do_empty[s]), phe, wc, kWhereBwdProducer)) break;
        if (leader) {
          mbar_arrive_expect_tx(BAR(do_full[s]), kTileBytes);
          tma_load_3d(sbase + kDOOff + s * kTileBytes, &tm_do, BAR(do_full[s]), 0, h, qi * 128);
          tma_load_3d(sbase + kDOOff + s * kTileBytes + kHalfBytes, &tm_do, BAR(do_full[s]), 64,
                      h, qi * 128);
        }
        __syncwarp();
        ++ndo_issued;
      }
      if (bars->abort_flag) {
        // unwinding: let every copy this warp issued land before the CTA exits
        mbar_drain_wait(BAR(kv_full), 0);
        for (int s = 0; s < 2; ++s) {
          const int lq = (nq_issued - 1 - s) >= 0 ? ((nq_issued - 1 - s) / 2) * 2 + s : -1;
          if (lq >= 0) mbar_drain_wait(BAR(q_full[s]), (lq >> 1) & 1);
          const int ld = (ndo_issued - 1 - s) >= 0 ? ((ndo_issued - 1 - s) / 2) * 2 + s : -1;
          if (ld >= 0) mbar_drain_wait(BAR(do_full[s]), (ld >> 1) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop in lockstep (its decisions are
    // warp-uniform); one elected lane issues the MMAs and their commits.
    {
      constexpr uint32_t kIdKQ = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, 128, false, true);  // dV, dK
      constexpr uint32_t kIdDQ = idesc_bf16_f32(128, 128, true, true);    // dQ^T
      const uint32_t t_r0 = tmem, t_r1 = tmem + 128, t_dv = tmem + 256, t_dk = tmem + 384;
      bool ok = mbar_wait_spin(BAR(kv_full), 0, wc, kWhereBwdMma);
      // every operand descriptor = one base + compile-time constants
      const uint64_t d0 = desc_kmajor0(sbase);
      const uint64_t dK_k = d0 + desc_off(kKOff), dK_mn = d0 + kDescMn + desc_off(kKOff);
      const uint64_t dV_k = d0 + desc_off(kVOff);
      const uint64_t dDS_k = d0 + desc_off(kDSOff), dDS_mn = d0 + kDescMn + desc_off(kDSOff);
      const uint64_t dQ_k = d0 + desc_off(kQOff), dQ_mn = d0 + kDescMn + desc_off(kQOff);
      const uint64_t dDO_k = d0 + desc_off(kDOOff), dDO_mn = d0 + kDescMn + desc_off(kDOOff);
      // S^T(n) = K Q^T into R0: R0 is free once MMA3 of n-1 has read P^T (the
      // compute warps keep their own copy of P(n-1) in registers for the dS pass)
      auto issue_s = [&](int n) -> bool {
        const int s = n & 1;
        if (!mbar_wait_spin(BAR(q_full[s]), (n >> 1) & 1, wc, kWhereBwdMma)) return false;
        if (n > 0 && !mbar_wait_spin(BAR(pt_consumed), (n - 1) & 1, wc, kWhereBwdMma)) return false;
        tc_fence_after();
        const uint64_t a = opaque(dK_k), qa = opaque(dQ_k + s * kTileDesc);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ss(t_r0, a + kstep_kmajor(kk), qa + kstep_kmajor(kk), kIdKQ, kk > 0);
          umma_commit(BAR(s_full));
        }
        __syncwarp();
        return true;
      };
      // Issue order: S^T(0); then per n: dP^T(n), dV(n), S^T(n+1), dK(n), dQ^T(n).
      // S^T(n+1) goes before dK/dQ(n) so that the exponentials of n+1 can start
      // as soon as the dS pass of n is over.
      if (ok && n_iter > 0) ok = issue_s(0);
      for (int n = 0; ok && n < n_iter; ++n) {
        const int s = n & 1;
        const uint32_t phs = (n >> 1) & 1;       // stage phase
        const uint32_t ph = n & 1, ph1 = ph ^ 1; // per-iteration phase
        // MMA2: dP^T = V dO^T  (R1 must be free: dQ^T of n-1 copied out by the drain)
        if (!(ok = mbar_wait_spin(BAR(do_full[s]), phs, wc, kWhereBwdMma))) break;
        if (!(ok = mbar_wait_spin(BAR(r1_free), ph1, wc, kWhereBwdMma))) break;
        tc_fence_after();
        {
          const uint64_t a = opaque(dV_k), da = opaque(dDO_k + s * kTileDesc);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_ss(t_r1, a + kstep_kmajor(kk), da + kstep_kmajor(kk), kIdKQ, kk > 0);
            umma_commit(BAR(dp_full));
          }
          __syncwarp();
        }
        // MMA3: dV += P^T dO  (P^T in TMEM R0 as bf16 pairs, 8 columns per k-step;
        // query columns [64 h, 64 h + 64) sit at R0 columns [64 h, 64 h + 32))
        if (!(ok = mbar_wait_spin(BAR(p_ready), ph, wc, kWhereBwdMma))) break;
        tc_fence_after();
        {
          const uint64_t da = opaque(dDO_mn + s * kTileDesc);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_ts(t_dv, t_r0 + 64 * (kk >> 2) + 8 * (kk & 3), da + kstep_mnmajor(kk), kIdAcc,
                      (n > 0 || kk > 0));
            umma_commit(BAR(pt_consumed));
            umma_commit(BAR(do_empty[s]));
          }
          __syncwarp();
        }
        // MMA1 of the next iteration
        if (n + 1 < n_iter && !(ok = issue_s(n + 1))) break;
        // MMA4: dK += dS^T Q ; MMA5: dQ^T = K^T dS^T
        if (!(ok = mbar_wait_spin(BAR(ds_ready), ph, wc, kWhereBwdMma))) break;
        tc_fence_after();
        {
          const uint64_t a = opaque(dDS_k), qa = opaque(dQ_mn + s * kTileDesc);
          const uint64_t a2 = opaque(dK_mn), b2 = opaque(dDS_mn);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_ss(t_dk, a + kstep_kmajor(kk), qa + kstep_mnmajor(kk), kIdAcc, (n > 0 || kk > 0));
            umma_commit(BAR(q_empty[s]));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              umma_ss(t_r1, a2 + kstep_mnmajor(kk), b2 + kstep_mnmajor(kk), kIdDQ, kk > 0);
            umma_commit(BAR(dq_full));
            umma_commit(BAR(ds_free));
          }
          __syncwarp();
        }
      }
      if (ok) {
        if (elect_one()) umma_commit(BAR(acc_done));
        __syncwarp();
      } else {
        if (elect_one()) umma_commit(BAR(drain));
        __syncwarp();
        mbar_drain_wait(BAR(drain), 0);
      }
    }
  }
  } else {
    // ------------------------------------------------------------ compute / drain
    const int q4 = warp & 3;
    const bool drain_warp = warp >= 12;
    const int ch = (warp - 4) >> 2;                // compute: column half [64 ch, 64 ch + 64)
    const int r = q4 * 32 + lane;                  // key row (S/dP/dK/dV) or d (dQ^T)
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t t_r0 = tmem + lane_base, t_r1 = tmem + lane_base + 128;
    // key row validity: invalid rows (padding of a ragged tile) get P = 0
    bool key_valid;
    tile_page(r / p.page_size, &key_valid);
    if (!is_sel) key_valid = key_valid && (own_t * 128 + r) < p.chunk_len;
    const float row_bias = key_valid ? 0.f : -INFINITY;
    const bool warp_valid = __all_sync(0xffffffffu, key_valid);
    bool ok = true;
    if (drain_warp) {
      regs_increase<184>();
      // ---- dQ^T drain: TMEM lane = head-dim index r, columns = query rows
      for (int n = 0; n < n_iter; ++n) {
        const int qi = i0 + n % nq;
        const int h = g * grp + n / nq;
        ok = __all_sync(0xffffffffu, mbar_wait(BAR(dq_full), n & 1, wc, kWhereBwdCompute));
        if (!ok) break;
        tc_fence_after();
        const int t0 = qi * 128;
        const int rows = min(128, p.chunk_len - t0);
        float* dst = p.dq_acc + (static_cast<long>(t0) * p.hq + h) * 128 + r;
        const long row_stride = static_cast<long>(p.hq) * 128;
        uint32_t v[128];
        tmem_ld128(t_r1, v);
        tc_fence_before();
        mbar_arrive(BAR(r1_free));                 // R1 may now take the next dP^T
        if (rows >= 128) {                         // full query tile: the common case
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            red_add_f32(dst, __uint_as_float(v[c]));
            dst += row_stride;
          }
        } else {
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            if (c < rows) red_add_f32(dst, __uint_as_float(v[c]));
            dst += row_stride;
          }
        }
      }
      regs_decrease<128>();
    } else {
      for (int n = 0; n < n_iter; ++n) {
        const int qi = i0 + n % nq;
        const int s = n & 1;
        const uint32_t phs = (n >> 1) & 1, ph = n & 1, ph1 = ph ^ 1;
        const float4* lse4 = reinterpret_cast<const float4*>(vec + s * 256 + 64 * ch);
        const float4* dl4 = reinterpret_cast<const float4*>(vec + s * 256 + 128 + 64 * ch);
        const bool diag = !is_sel && qi == own_t;   // key r sees query columns c >= r only
        // ---- P^T = exp2(S^T scale log2e - lse2) -> bf16 pairs into R0
        ok = __all_sync(0xffffffffu, mbar_wait(BAR(s_full), ph, wc, kWhereBwdCompute));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(BAR(q_full[s]), phs, wc, kWhereBwdCompute));
        if (!ok) break;
        tc_fence_after();
        uint32_t pk[32];                           // P^T of this warp's 64 columns, kept for dS
        {
          uint32_t rr[64];
          tmem_ld64(t_r0 + 64 * ch, rr);
          if (warp_valid && !diag) {               // no mask: the common case
            const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
            for (int i = 0; i < 64; i += 4) {       // scaling on packed FP32 pairs
              const float4 l = lse4[i >> 2];
              float x0, x1, x2, x3;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1])), sc2,
                               f2_pack(-l.x, -l.y)), x0, x1);
              f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[i + 2]), __uint_as_float(rr[i + 3])),
                               sc2, f2_pack(-l.z, -l.w)), x2, x3);
              pk[i >> 1] = pack_bf16(ex2(x0), ex2(x1));
              pk[(i >> 1) + 1] = pack_bf16(ex2(x2), ex2(x3));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 64; i += 4) {
              const float4 l = lse4[i >> 2];
              const float lv[4] = {l.x, l.y, l.z, l.w};
              float e[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                float x = fmaf(__uint_as_float(rr[i + j]), p.scale_log2, row_bias - lv[j]);
                if (diag && 64 * ch + i + j < r) x = -INFINITY;
                e[j] = ex2(x);
              }
              pk[i >> 1] = pack_bf16(e[0], e[1]);
              pk[(i >> 1) + 1] = pack_bf16(e[2], e[3]);
            }
          }
          // P^T of query columns [64 ch, 64 ch + 64) goes to R0 columns
          // [64 ch, 64 ch + 32): inside the S^T columns this warp has just read,
          // so the other warp of the lane quarter is never overtaken
          tmem_st32(t_r0 + 64 * ch, pk);
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(BAR(p_ready));
        // ---- dS^T = P^T (dP^T - Delta) -> shared (bf16, swizzled)
        ok = __all_sync(0xffffffffu, mbar_wait(BAR(dp_full), ph, wc, kWhereBwdCompute));
        if (ok && n > 0) ok = __all_sync(0xffffffffu, mbar_wait(BAR(ds_free), ph1, wc, kWhereBwdCompute));
        if (!ok) break;
        tc_fence_after();
        const uint32_t ds_row = sbase + kDSOff;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c32 = 2 * ch + cc;             // 32-column chunk
          uint32_t dp[32];
          tmem_ld32(t_r1 + 32 * c32, dp);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 dl = dl4[(32 * cc + i) >> 2];
            const uint64_t dv2[2] = {f2_pack(dl.x, dl.y), f2_pack(dl.z, dl.w)};
            float d[4];
#pragma unroll
            for (int j = 0; j < 4; j += 2) {        // two columns per packed FP32 pair
              const uint32_t pw = pk[16 * cc + ((i + j) >> 1)];
              const uint64_t p2 = f2_pack(__uint_as_float(pw << 16), __uint_as_float(pw & 0xFFFF0000u));
              const uint64_t x2 = f2_sub(
                  f2_pack(__uint_as_float(dp[i + j]), __uint_as_float(dp[i + j + 1])), dv2[j >> 1]);
              f2_unpack(f2_mul(p2, x2), d[j], d[j + 1]);
            }
            w[i >> 1] = pack_bf16(d[0], d[1]);
            w[(i >> 1) + 1] = pack_bf16(d[2], d[3]);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
            st_shared_v4(ds_row + tile128_chunk_off(r, 4 * c32 + k), w[4 * k], w[4 * k + 1],
                         w[4 * k + 2], w[4 * k + 3]);
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(BAR(ds_ready));
      }
    }
    // ---- epilogue: dK (x scale), dV rows of this key tile into the paged bf16 gradients
    if (ok && !drain_warp)
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(acc_done), 0, wc, kWhereBwdEpilogue));
    if (ok && !drain_warp) {
      tc_fence_after();
      const int u = r / p.page_size;
      bool valid;
      const int lp = tile_page(u, &valid);
      bool write = key_valid && valid;
      if (write && is_sel) {
        // the selection must be in range and strictly ascending (one owner per slot)
        const int pi = kt * ppt + u;
        if (lp < 0 || lp >= own_page0 || (pi > 0 && sel_g[pi - 1] >= lp)) {
          raise_status(p.status, kStatusBounds, kWhereBwdEpilogue);
          write = false;
        }
      }
      int slot = write ? p.pt[lp] : 0;
      if (write && (slot < 0 || slot >= p.num_slots)) {
        raise_status(p.status, kStatusBounds, kWhereBwdEpilogue);
        write = false;
      }
      const long row = ((static_cast<long>(slot) * p.hkv + g) * p.page_size + r % p.page_size) * 128
                       + 64 * ch;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* pool = which == 0 ? p.dk : p.dv;
        const uint32_t tcol = (which == 0 ? 384 : 256) + 64 * ch;
        const float mul = which == 0 ? p.scale : 1.f;
        uint4* dst = reinterpret_cast<uint4*>(pool + row);
        uint32_t rr[64];
        tmem_ld64(tmem + lane_base + tcol, rr);
        if (write) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint4 o = dst[i];
            const float* a = reinterpret_cast<const float*>(rr) + 8 * i;
            o.x = bf16x2_add(o.x, a[0] * mul, a[1] * mul);
            o.y = bf16x2_add(o.y, a[2] * mul, a[3] * mul);
            o.z = bf16x2_add(o.z, a[4] * mul, a[5] * mul);
            o.w = bf16x2_add(o.w, a[6] * mul, a[7] * mul);
            dst[i] = o;
          }
        }
      }
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

// Delta[h][t] = dout[t][h] . o[t][h], lse2[h][t] = lse[h][t] * log2(e); on the
// padding rows of the last query tile Delta = 0 and lse2 = +inf (so P = 0
// there).  With the forward's residual o_lo, o is taken as o + o_lo (exact in
// fp32): Delta is subtracted from dP = dout . v, which it nearly equals in a
// row whose attention sits on one key, so the bf16 rounding of o would
// otherwise reach dS.  Also zeroes the fp32 dq accumulator.  Half a warp per
// (t, h) row.
__global__ void bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                const __nv_bfloat16* __restrict__ o_lo,
                                const __nv_bfloat16* __restrict__ dout,
                                const float* __restrict__ lse, int hq, int chunk_len,
                                int padded_len, float* __restrict__ delta,
                                float* __restrict__ lse2, float* __restrict__ dq_acc) {
  const long row = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const int l16 = threadIdx.x & 15;
  const long n_rows = static_cast<long>(padded_len) * hq;
  if (row >= n_rows) return;
  const int t = static_cast<int>(row / hq), h = static_cast<int>(row % hq);
  float s = 0.f;
  if (t < chunk_len) {
    const uint4 a = reinterpret_cast<const uint4*>(o + row * 128)[l16];
    const uint4 b = reinterpret_cast<const uint4*>(dout + row * 128)[l16];
    const uint4 c = o_lo ? reinterpret_cast<const uint4*>(o_lo + row * 128)[l16]
                         : make_uint4(0, 0, 0, 0);
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
    const uint32_t wc[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float o0 = __uint_as_float(wa[i] << 16) + __uint_as_float(wc[i] << 16);
      const float o1 = __uint_as_float(wa[i] & 0xFFFF0000u) + __uint_as_float(wc[i] & 0xFFFF0000u);
      s = fmaf(o0, __uint_as_float(wb[i] << 16), s);
      s = fmaf(o1, __uint_as_float(wb[i] & 0xFFFF0000u), s);
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + row * 128) + 2 * l16;
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (l16 == 0) {
    const long o2 = static_cast<long>(h) * padded_len + t;
    delta[o2] = s;
    lse2[o2] = t < chunk_len ? lse[static_cast<long>(h) * chunk_len + t] * 1.4426950408889634f
                             : INFINITY;
  }
}

__global__ void dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                  long n8, float scale) {
  const long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
  uint4 v;
  v.x = pack_bf16(a.x * scale, a.y * scale);
  v.y = pack_bf16(a.z * scale, a.w * scale);
  v.z = pack_bf16(b.x * scale, b.y * scale);
  v.w = pack_bf16(b.z * scale, b.w * scale);
  reinterpret_cast<uint4*>(dq)[i] = v;
}

}  // namespace

size_t bf16_bwd_ws_bytes(int hq, int chunk_len, int head_dim) {
  const size_t padded = static_cast<size_t>((chunk_len + 127) / 128) * 128;
  return kStatusBytes + 2 * align_up(static_cast<size_t>(hq) * padded * 4, 256) +
         align_up(static_cast<size_t>(chunk_len) * hq * head_dim * 4, 256);
}

cudaError_t launch_attn_bwd_bf16(const void* q, const void* o, const void* o_lo,
                                 const void* dout, const float* lse, const KvDesc& kv,
                                 const int32_t* sel, int n_sel, int hq, int chunk_len,
                                 int chunk_start, float scale, void* dq, void* ws,
                                 uint64_t wait_ns, cudaStream_t st) {
  const int n_qtiles = (chunk_len + 127) / 128;
  const int padded = n_qtiles * 128;
  char* w = static_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(w);
  const size_t vec_bytes = align_up(static_cast<size_t>(hq) * padded * 4, 256);
  float* delta = reinterpret_cast<float*>(w + kStatusBytes);
  float* lse2 = reinterpret_cast<float*>(w + kStatusBytes + vec_bytes);
  float* dq_acc = reinterpret_cast<float*>(w + kStatusBytes + 2 * vec_bytes);
  CUtensorMap tq, tdo, tk, tv;
  {
    const uint64_t dims[3] = {128, static_cast<uint64_t>(hq), static_cast<uint64_t>(chunk_len)};
    const uint64_t strides[2] = {128 * 2, static_cast<uint64_t>(hq) * 128 * 2};
    const uint32_t box[3] = {64, 1, 128};
    if (!make_tmap_bf16(&tq, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tdo, dout, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t rows = static_cast<uint64_t>(kv.num_slots) * kv.hkv * kv.page_size;
    const uint64_t dims[2] = {128, rows};
    const uint64_t strides[1] = {128 * 2};
    const uint32_t box[2] = {64, static_cast<uint32_t>(kv.page_size)};
    if (!make_tmap_bf16(&tk, kv.k, 2, dims, strides, box)) return cudaErrorInvalidValue;
    if (!make_tmap_bf16(&tv, kv.v, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const long rows16 = static_cast<long>(padded) * hq * 16;
    bwd_prep_kernel<<<static_cast<unsigned>((rows16 + 255) / 256), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(o_lo),
        static_cast<const __nv_bfloat16*>(dout), lse, hq, chunk_len, padded, delta, lse2, dq_acc);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  BwdParams p;
  p.sel = sel;
  p.pt = kv.page_table;
  p.lse2 = lse2;
  p.delta = delta;
  p.dq_acc = dq_acc;
  p.dk = static_cast<__nv_bfloat16*>(kv.dk);
  p.dv = static_cast<__nv_bfloat16*>(kv.dv);
  p.status = status;
  p.n_sel = n_sel;
  p.hq = hq;
  p.hkv = kv.hkv;
  p.page_size = kv.page_size;
  p.chunk_len = chunk_len;
  p.chunk_start = chunk_start;
  p.num_slots = kv.num_slots;
  p.n_qtiles = n_qtiles;
  p.t_sel = (n_sel * kv.page_size + 127) / 128;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_ns = wait_ns;
  static PerDeviceOnce attr;
  {
    cudaError_t e = once_per_device(attr, [] {
      return cudaFuncSetAttribute(sparse_attn_bwd_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    });
    if (e != cudaSuccess) return e;
  }
  const int n_key_tiles = p.t_sel + n_qtiles;
  sparse_attn_bwd_kernel<<<n_key_tiles * kv.hkv, kThreads, kSmemBytes, st>>>(tq, tdo, tk, tv, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long n8 = static_cast<long>(chunk_len) * hq * 128 / 8;
  dq_convert_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, st>>>(
      dq_acc, static_cast<__nv_bfloat16*>(dq), n8, scale);
  return cudaGetLastError();
}

}  // namespace oomb
