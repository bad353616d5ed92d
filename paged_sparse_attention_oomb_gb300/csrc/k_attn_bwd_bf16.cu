// Step 4 of the path: backward of page-level sparse causal attention on the
// tcgen05 tensor cores, with the dK/dV accumulation into the paged gradient
// buffers fused into the tile loop.
// Method: "Out of the Memory Barrier" technical summary, section 2: "Paged
// Memory Management" (KV gradients live in pages and are accumulated in place
// outside autograd) and "Page-level Sparse Attention" (the backward reuses the
// forward's page choice).
//
// One CTA owns one 128-key tile of one KV head: a tile of selected pages
// (attended by every query tile of the chunk) or of the chunk's own pages
// (attended by the query tiles at or after it).  It loops over the G query
// heads of the group x the query tiles that see it; per iteration:
//   dP^T = V dO^T, S^T = K Q^T          (TMEM, keys on lanes, queries on columns)
//   P^T = exp(scale S^T - lse),  dS^T = P^T (dP^T - Delta)    (compute warps)
//   dV += P^T dO,  dK += dS^T Q          (TMEM accumulators, whole CTA life)
//   dQ_tile = dS K                       (TMEM, drained with fp32 reductions)
// At the end dK (x scale) and dV are added to the bf16 gradient pages of the
// tile's slots: one read-add-write and one rounding per slot per call.  Each
// (slot, KV head) has exactly one owner CTA, so no atomics touch dK/dV.
// Roles (192 threads): warp 0 TMA producer + TMEM allocator, warp 1 MMA
// issuer, warps 2..5 compute (TMEM lane quarter = warp % 4).
// TMEM: [0,128) S^T then dQ, [128,256) dP^T, [256,384) dV, [384,512) dK.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "oomb_internal.h"
#include "sm100.cuh"
#include "tmap.h"

namespace oomb {
namespace {

constexpr int kThreads = 192;
constexpr uint32_t kKOff = 0;
constexpr uint32_t kVOff = kTileBytes;
constexpr uint32_t kQOff = 2 * kTileBytes;
constexpr uint32_t kDOOff = 3 * kTileBytes;
constexpr uint32_t kPTOff = 4 * kTileBytes;
constexpr uint32_t kDSOff = 5 * kTileBytes;
constexpr uint32_t kVecOff = 6 * kTileBytes;      // lse[2][128], delta[2][128] floats
constexpr uint32_t kBarOff = kVecOff + 2048;
constexpr uint32_t kSmemBytes = kBarOff + 256 + 1024;

struct Bars {
  uint64_t kv_full;
  uint64_t q_full, q_empty;
  uint64_t do_full, do_empty;
  uint64_t s_full, dp_full, dq_full;
  uint64_t r0_free, r1_free;
  uint64_t pt_ready, ds_ready, pds_free;
  uint64_t acc_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdParams {
  const int32_t* sel;
  const int32_t* pt;
  const float* lse;        // [hq][chunk_len]
  const float* delta;      // [hq][n_qtiles*128]
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
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  const uint32_t bbase = sbase + kBarOff;
  float* vec = reinterpret_cast<float*>(smem + kVecOff);   // lse: [0,256), delta: [256,512)
#define BAR(f) bar_addr(bbase, &bars->f, bars)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
  const int n_own_pages = p.chunk_len / p.page_size;
  const int32_t* sel_g = p.sel + static_cast<long>(g) * p.n_sel;

  if (threadIdx.x == 0) {
    mbar_init(BAR(kv_full), 1);
    mbar_init(BAR(q_full), 1);
    mbar_init(BAR(q_empty), 1);
    mbar_init(BAR(do_full), 1);
    mbar_init(BAR(do_empty), 1);
    mbar_init(BAR(s_full), 1);
    mbar_init(BAR(dp_full), 1);
    mbar_init(BAR(dq_full), 1);
    mbar_init(BAR(r0_free), 128);
    mbar_init(BAR(r1_free), 128);
    mbar_init(BAR(pt_ready), 128);
    mbar_init(BAR(ds_ready), 128);
    mbar_init(BAR(pds_free), 1);
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

  // Logical page of slot-row u of this key tile, and whether its keys are real.
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(BAR(kv_full), 2 * kTileBytes);
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
        for (int hf = 0; hf < 2; ++hf) {
          const uint32_t off = hf * kHalfBytes + u * p.page_size * 128;
          tma_load_2d(sbase + kKOff + off, &tm_k, BAR(kv_full), hf * 64, row);
          tma_load_2d(sbase + kVOff + off, &tm_v, BAR(kv_full), hf * 64, row);
        }
      }
      int nq_issued = 0, ndo_issued = 0;
      for (int n = 0; n < n_iter; ++n) {
        const int h = g * grp + n / nq;
        const int qi = i0 + n % nq;
        const uint32_t ph1 = (n & 1) ^ 1;
        if (!mbar_wait(BAR(q_empty), ph1, wc, kWhereBwdProducer)) break;
        mbar_arrive_expect_tx(BAR(q_full), kTileBytes);
        tma_load_3d(sbase + kQOff, &tm_q, BAR(q_full), 0, h, qi * 128);
        tma_load_3d(sbase + kQOff + kHalfBytes, &tm_q, BAR(q_full), 64, h, qi * 128);
        ++nq_issued;
        if (!mbar_wait(BAR(do_empty), ph1, wc, kWhereBwdProducer)) break;
        const int rows = min(128, p.chunk_len - qi * 128);
        const uint32_t vb = sbase + kVecOff + (n & 1) * 512;
        mbar_arrive_expect_tx(BAR(do_full), kTileBytes + rows * 4 + 512);
        tma_load_3d(sbase + kDOOff, &tm_do, BAR(do_full), 0, h, qi * 128);
        tma_load_3d(sbase + kDOOff + kHalfBytes, &tm_do, BAR(do_full), 64, h, qi * 128);
        bulk_load(vb, p.lse + static_cast<long>(h) * p.chunk_len + qi * 128, rows * 4,
                  BAR(do_full));
        bulk_load(vb + 1024, p.delta + static_cast<long>(h) * p.n_qtiles * 128 + qi * 128, 512,
                  BAR(do_full));
        ++ndo_issued;
      }
      if (bars->abort_flag) {
        mbar_drain_wait(BAR(kv_full), 0);
        if (nq_issued > 0) mbar_drain_wait(BAR(q_full), (nq_issued - 1) & 1);
        if (ndo_issued > 0) mbar_drain_wait(BAR(do_full), (ndo_issued - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdKQ = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, 128, false, true);  // dV, dK
      constexpr uint32_t kIdDQ = idesc_bf16_f32(128, 128, true, true);    // dQ
      const uint32_t t_r0 = tmem, t_r1 = tmem + 128, t_dv = tmem + 256, t_dk = tmem + 384;
      bool ok = mbar_wait(BAR(kv_full), 0, wc, kWhereBwdMma);
      for (int n = 0; ok && n < n_iter; ++n) {
        const uint32_t ph = n & 1, ph1 = ph ^ 1;
        // dP^T = V dO^T
        if (!(ok = mbar_wait(BAR(do_full), ph, wc, kWhereBwdMma))) break;
        if (!(ok = mbar_wait(BAR(r1_free), ph1, wc, kWhereBwdMma))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(t_r1, desc_kmajor(sbase + kVOff, kk), desc_kmajor(sbase + kDOOff, kk), kIdKQ,
                  kk > 0);
        umma_commit(BAR(dp_full));
        // S^T = K Q^T
        if (!(ok = mbar_wait(BAR(q_full), ph, wc, kWhereBwdMma))) break;
        if (!(ok = mbar_wait(BAR(r0_free), ph1, wc, kWhereBwdMma))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(t_r0, desc_kmajor(sbase + kKOff, kk), desc_kmajor(sbase + kQOff, kk), kIdKQ,
                  kk > 0);
        umma_commit(BAR(s_full));
        // dV += P^T dO
        if (!(ok = mbar_wait(BAR(pt_ready), ph, wc, kWhereBwdMma))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(t_dv, desc_kmajor(sbase + kPTOff, kk), desc_mnmajor(sbase + kDOOff, kk), kIdAcc,
                  (n > 0 || kk > 0));
        umma_commit(BAR(do_empty));
        // dK += dS^T Q ; dQ = dS K
        if (!(ok = mbar_wait(BAR(ds_ready), ph, wc, kWhereBwdMma))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(t_dk, desc_kmajor(sbase + kDSOff, kk), desc_mnmajor(sbase + kQOff, kk), kIdAcc,
                  (n > 0 || kk > 0));
        umma_commit(BAR(q_empty));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(t_r0, desc_mnmajor(sbase + kDSOff, kk), desc_mnmajor(sbase + kKOff, kk), kIdDQ,
                  kk > 0);
        umma_commit(BAR(dq_full));
        umma_commit(BAR(pds_free));
      }
      if (ok) {
        umma_commit(BAR(acc_done));
      } else {
        umma_commit(BAR(drain));
        mbar_drain_wait(BAR(drain), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ compute
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;                  // key row (S/dP/dK/dV) or query row (dQ)
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const float LOG2E = 1.4426950408889634f;
    // key row validity and, for own tiles, its position within the chunk
    bool key_valid;
    tile_page(r / p.page_size, &key_valid);
    const int key_u = is_sel ? -1 : own_t * 128 + r;
    if (!is_sel) key_valid = key_valid && key_u < p.chunk_len;
    bool ok = true;
    for (int n = 0; n < n_iter; ++n) {
      const int h = g * grp + n / nq;
      const int qi = i0 + n % nq;
      const uint32_t ph = n & 1, ph1 = ph ^ 1;
      const float* lse_s = vec + (n & 1) * 128;
      const float* dl_s = vec + 256 + (n & 1) * 128;
      // columns c valid iff c < lim (query rows of the chunk, causal)
      int lo = 0;
      if (!is_sel && qi == own_t) lo = r;          // key r sees query columns c >= r
      const int lim = min(128, p.chunk_len - qi * 128);
      // ---- P^T from S^T
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(s_full), ph, wc, kWhereBwdCompute));
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(do_full), ph, wc, kWhereBwdCompute));
      if (!ok) break;
      tc_fence_after();
      float pr[128];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + c4 * 32, rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = c4 * 32 + i;
          const float x = fmaf(__uint_as_float(rr[i]), p.scale_log2, -lse_s[c] * LOG2E);
          pr[c] = (key_valid && c >= lo && c < lim) ? ex2(x) : 0.f;
        }
      }
      if (n > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(BAR(pds_free), ph1, wc, kWhereBwdCompute));
        if (!ok) break;
      }
      const uint32_t pt_row = sbase + kPTOff;
#pragma unroll
      for (int c = 0; c < 16; ++c)
        st_shared_v4(pt_row + tile128_chunk_off(r, c), pack_bf16(pr[8 * c], pr[8 * c + 1]),
                     pack_bf16(pr[8 * c + 2], pr[8 * c + 3]), pack_bf16(pr[8 * c + 4], pr[8 * c + 5]),
                     pack_bf16(pr[8 * c + 6], pr[8 * c + 7]));
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(BAR(pt_ready));
      // ---- dS^T = P^T (dP^T - Delta)
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(dp_full), ph, wc, kWhereBwdCompute));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + 128 + c4 * 32, rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = c4 * 32 + i;
          pr[c] = pr[c] * (__uint_as_float(rr[i]) - dl_s[c]);
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(r1_free));
      const uint32_t ds_row = sbase + kDSOff;
#pragma unroll
      for (int c = 0; c < 16; ++c)
        st_shared_v4(ds_row + tile128_chunk_off(r, c), pack_bf16(pr[8 * c], pr[8 * c + 1]),
                     pack_bf16(pr[8 * c + 2], pr[8 * c + 3]), pack_bf16(pr[8 * c + 4], pr[8 * c + 5]),
                     pack_bf16(pr[8 * c + 6], pr[8 * c + 7]));
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(BAR(ds_ready));
      // ---- drain dQ (TMEM lane = query row)
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(dq_full), ph, wc, kWhereBwdCompute));
      if (!ok) break;
      tc_fence_after();
      const int t = qi * 128 + r;
      float* dst = p.dq_acc + (static_cast<long>(t) * p.hq + h) * 128;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + c4 * 32, rr);
        if (t < p.chunk_len) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            red_add_v4(dst + c4 * 32 + 4 * i, __uint_as_float(rr[4 * i]) * p.scale,
                       __uint_as_float(rr[4 * i + 1]) * p.scale,
                       __uint_as_float(rr[4 * i + 2]) * p.scale,
                       __uint_as_float(rr[4 * i + 3]) * p.scale);
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(r0_free));
    }
    // ---- epilogue: dK, dV rows of this key tile into the paged bf16 gradients
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(BAR(acc_done), 0, wc, kWhereBwdEpilogue));
    if (ok) {
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
      const long row = ((static_cast<long>(slot) * p.hkv + g) * p.page_size + r % p.page_size) * 128;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* pool = which == 0 ? p.dk : p.dv;
        const float mul = which == 0 ? p.scale : 1.f;
        const uint32_t tcol = which == 0 ? 384 : 256;
        uint4* dst = reinterpret_cast<uint4*>(pool + row);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_base + tcol + c4 * 32, rr);
          if (write) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 o = dst[c4 * 4 + i];
              const float* a = reinterpret_cast<const float*>(rr) + 8 * i;
              o.x = bf16x2_add(o.x, a[0] * mul, a[1] * mul);
              o.y = bf16x2_add(o.y, a[2] * mul, a[3] * mul);
              o.z = bf16x2_add(o.z, a[4] * mul, a[5] * mul);
              o.w = bf16x2_add(o.w, a[6] * mul, a[7] * mul);
              dst[c4 * 4 + i] = o;
            }
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

// Delta[h][t] = dout[t][h] . o[t][h] (0 for the padding rows of the last
// query tile) and a zeroed fp32 dq accumulator.  Half a warp per (t, h) row.
__global__ void bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                const __nv_bfloat16* __restrict__ dout, int hq, int chunk_len,
                                int padded_len, float* __restrict__ delta,
                                float* __restrict__ dq_acc) {
  const long row = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  const int l16 = threadIdx.x & 15;
  const long n_rows = static_cast<long>(padded_len) * hq;
  if (row >= n_rows) return;
  const int t = static_cast<int>(row / hq), h = static_cast<int>(row % hq);
  float s = 0.f;
  if (t < chunk_len) {
    const uint4 a = reinterpret_cast<const uint4*>(o + row * 128)[l16];
    const uint4 b = reinterpret_cast<const uint4*>(dout + row * 128)[l16];
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s = fmaf(__uint_as_float(wa[i] << 16), __uint_as_float(wb[i] << 16), s);
      s = fmaf(__uint_as_float(wa[i] & 0xFFFF0000u), __uint_as_float(wb[i] & 0xFFFF0000u), s);
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + row * 128) + 2 * l16;
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (l16 == 0) delta[static_cast<long>(h) * padded_len + t] = s;
}

__global__ void dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                  long n8) {
  const long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
  uint4 v;
  v.x = pack_bf16(a.x, a.y);
  v.y = pack_bf16(a.z, a.w);
  v.z = pack_bf16(b.x, b.y);
  v.w = pack_bf16(b.z, b.w);
  reinterpret_cast<uint4*>(dq)[i] = v;
}

}  // namespace

size_t bf16_bwd_ws_bytes(int hq, int chunk_len, int head_dim) {
  const size_t padded = static_cast<size_t>((chunk_len + 127) / 128) * 128;
  return kStatusBytes + align_up(static_cast<size_t>(hq) * padded * 4, 256) +
         align_up(static_cast<size_t>(chunk_len) * hq * head_dim * 4, 256);
}

cudaError_t launch_attn_bwd_bf16(const void* q, const void* o, const void* dout,
                                 const float* lse, const KvDesc& kv, const int32_t* sel,
                                 int n_sel, int hq, int chunk_len, int chunk_start, float scale,
                                 void* dq, void* ws, uint64_t wait_ns, cudaStream_t st) {
  const int n_qtiles = (chunk_len + 127) / 128;
  const int padded = n_qtiles * 128;
  char* w = static_cast<char*>(ws);
  int* status = reinterpret_cast<int*>(w);
  float* delta = reinterpret_cast<float*>(w + kStatusBytes);
  float* dq_acc = reinterpret_cast<float*>(w + kStatusBytes +
                                           align_up(static_cast<size_t>(hq) * padded * 4, 256));
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
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), hq,
        chunk_len, padded, delta, dq_acc);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  BwdParams p;
  p.sel = sel;
  p.pt = kv.page_table;
  p.lse = lse;
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
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(sparse_attn_bwd_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int n_key_tiles = p.t_sel + n_qtiles;
  sparse_attn_bwd_kernel<<<n_key_tiles * kv.hkv, kThreads, kSmemBytes, st>>>(tq, tdo, tk, tv, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long n8 = static_cast<long>(chunk_len) * hq * 128 / 8;
  dq_convert_kernel<<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, st>>>(
      dq_acc, static_cast<__nv_bfloat16*>(dq), n8);
  return cudaGetLastError();
}

}  // namespace oomb
