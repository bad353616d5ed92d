// Step 3 of the path: forward of page-level sparse causal attention, bf16 in,
// fp32 accumulate, on the 5th-generation tensor cores (tcgen05 + TMEM).
// Method: "Out of the Memory Barrier" technical summary, section 2, item
// "Page-level Sparse Attention": the chunk attends the pages chosen by their
// representative vectors plus its own pages.
//
// One CTA computes one 128-row query tile of one query head against its key
// tiles: first the selected pages (ceil(n_sel * P / 128) tiles, no mask except
// a ragged last tile), then the chunk's own pages up to the diagonal tile.
// Roles (192 threads):
//   warp 0      TMA producer: Q once, then K/V tiles gathered page by page
//               through the page table (one 2-D box per page and 64-column half)
//               into a 2-stage ring; also allocates TMEM.
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM S
//               buffers, then O += P_{j-1} V_{j-1}; completion via tcgen05.commit.
//   warps 2..5  softmax, one thread per query row: reads S_j from TMEM, masks,
//               online softmax in base 2, writes P_j (bf16) to a 2-deep shared
//               ring in the 128-byte swizzled K-major layout.  O is rescaled in
//               TMEM only when a row maximum grows by more than 2^8 (the final
//               normalisation uses the same running maximum, so this is exact).
// TMEM: S0 [0,128), S1 [128,256), O [256,384) of a 512-column allocation.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "oomb_internal.h"
#include "sm100.cuh"
#include "tmap.h"

namespace oomb {
namespace {

constexpr int kThreads = 192;
constexpr uint32_t kQOff = 0;
constexpr uint32_t kKOff = kTileBytes;            // 2 stages
constexpr uint32_t kVOff = 3 * kTileBytes;        // 2 stages
constexpr uint32_t kPOff = 5 * kTileBytes;        // 2 buffers
constexpr uint32_t kBarOff = 7 * kTileBytes;
constexpr uint32_t kSmemBytes = kBarOff + 256 + 1024;   // + alignment slack
constexpr float kRescaleThreshold = 8.0f;         // log2 units

struct Bars {
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdParams {
  const int32_t* sel;
  const int32_t* pt;
  __nv_bfloat16* o;
  float* lse;
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
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  const uint32_t bbase = sbase + kBarOff;
#define BAR(f) bar_addr(bbase, &bars->f, bars)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heaviest query tiles (most own key tiles) first
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x) / p.hq;
  const int h = static_cast<int>(blockIdx.x) % p.hq;
  const int g = h / (p.hq / p.hkv);
  const int n_tiles = p.t_sel + qt + 1;
  const int ppt = 128 / p.page_size;               // pages per key tile
  const int own_page0 = p.chunk_start / p.page_size;
  const int n_own_pages = p.chunk_len / p.page_size;

  if (threadIdx.x == 0) {
    mbar_init(BAR(q_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(k_full[i]), 1);
      mbar_init(BAR(k_empty[i]), 1);
      mbar_init(BAR(v_full[i]), 1);
      mbar_init(BAR(v_empty[i]), 1);
      mbar_init(BAR(s_full[i]), 1);
      mbar_init(BAR(s_empty[i]), 128);
      mbar_init(BAR(p_full[i]), 128);
      mbar_init(BAR(o_done[i]), 1);
    }
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int issued = 0;                              // K/V tiles issued
      mbar_arrive_expect_tx(BAR(q_full), kTileBytes);
      tma_load_3d(sbase + kQOff, &tm_q, BAR(q_full), 0, h, qt * 128);
      tma_load_3d(sbase + kQOff + kHalfBytes, &tm_q, BAR(q_full), 64, h, qt * 128);
      const int32_t* sel_g = p.sel + static_cast<long>(g) * p.n_sel;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        int rows[8];
        for (int u = 0; u < ppt; ++u) {
          int lp;
          if (j < p.t_sel) {
            const int pi = j * ppt + u;
            lp = sel_g[pi < p.n_sel ? pi : 0];
            if (lp < 0 || lp >= own_page0) {
              raise_status(p.status, kStatusBounds, kWhereFwdProducer);
              lp = own_page0;
            }
          } else {
            lp = own_page0 + (j - p.t_sel) * ppt + u;
            if (lp >= own_page0 + n_own_pages) lp = own_page0;
          }
          int slot = p.pt[lp];
          if (slot < 0 || slot >= p.num_slots) {
            raise_status(p.status, kStatusBounds, kWhereFwdProducer);
            slot = 0;
          }
          rows[u] = (slot * p.hkv + g) * p.page_size;
        }
        if (!mbar_wait(BAR(k_empty[s]), ph ^ 1, wc, kWhereFwdProducer)) break;
        mbar_arrive_expect_tx(BAR(k_full[s]), kTileBytes);
        for (int u = 0; u < ppt; ++u)
          for (int hf = 0; hf < 2; ++hf)
            tma_load_2d(sbase + kKOff + s * kTileBytes + hf * kHalfBytes + u * p.page_size * 128,
                        &tm_k, BAR(k_full[s]), hf * 64, rows[u]);
        if (!mbar_wait(BAR(v_empty[s]), ph ^ 1, wc, kWhereFwdProducer)) {
          issued = 2 * j + 1;
          break;
        }
        mbar_arrive_expect_tx(BAR(v_full[s]), kTileBytes);
        for (int u = 0; u < ppt; ++u)
          for (int hf = 0; hf < 2; ++hf)
            tma_load_2d(sbase + kVOff + s * kTileBytes + hf * kHalfBytes + u * p.page_size * 128,
                        &tm_v, BAR(v_full[s]), hf * 64, rows[u]);
        issued = 2 * j + 2;
      }
      if (bars->abort_flag) {
        // unwinding: let every copy this thread issued land before the CTA exits
        mbar_drain_wait(BAR(q_full), 0);
        const int nk = (issued + 1) / 2, nv = issued / 2;   // K/V tiles issued
        for (int s = 0; s < 2; ++s) {
          const int lastk = (nk - 1 - s) >= 0 ? ((nk - 1 - s) / 2) * 2 + s : -1;
          if (lastk >= 0) mbar_drain_wait(BAR(k_full[s]), (lastk >> 1) & 1);
          const int lastv = (nv - 1 - s) >= 0 ? ((nv - 1 - s) / 2) * 2 + s : -1;
          if (lastv >= 0) mbar_drain_wait(BAR(v_full[s]), (lastv >> 1) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, 128, false, true);
      const uint32_t t_o = tmem + 256;
      bool ok = mbar_wait(BAR(q_full), 0, wc, kWhereFwdMma);
      auto issue_pv = [&](int jj) -> bool {
        const int s = jj & 1;
        const uint32_t ph = (jj >> 1) & 1;
        if (!mbar_wait(BAR(p_full[s]), ph, wc, kWhereFwdMma)) return false;
        if (!mbar_wait(BAR(v_full[s]), ph, wc, kWhereFwdMma)) return false;
        tc_fence_after();
        const uint32_t pa = sbase + kPOff + s * kTileBytes;
        const uint32_t va = sbase + kVOff + s * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(t_o, desc_kmajor(pa, kk), desc_mnmajor(va, kk), kIdPV, (jj > 0 || kk > 0));
        umma_commit(BAR(o_done[s]));
        umma_commit(BAR(v_empty[s]));
        return true;
      };
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int s = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(BAR(k_full[s]), ph, wc, kWhereFwdMma)) { ok = false; break; }
        if (!mbar_wait(BAR(s_empty[s]), ph ^ 1, wc, kWhereFwdMma)) { ok = false; break; }
        tc_fence_after();
        const uint32_t ka = sbase + kKOff + s * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + s * 128, desc_kmajor(sbase + kQOff, kk), desc_kmajor(ka, kk), kIdQK,
                  kk > 0);
        umma_commit(BAR(s_full[s]));
        umma_commit(BAR(k_empty[s]));
        if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_pv(n_tiles - 1);
      if (!ok) {
        umma_commit(BAR(drain));
        mbar_drain_wait(BAR(drain), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;                  // row of the query tile
    const int t = qt * 128 + r;                    // chunk row
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t t_o = tmem + lane_base + 256;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(s_full[b]), ph, wc, kWhereFwdSoftmax));
      if (!ok) break;
      tc_fence_after();
      float x[128];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + b * 128 + c4 * 32, rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c4 * 32 + i] = __uint_as_float(rr[i]);
      }
      tc_fence_before();
      mbar_arrive(BAR(s_empty[b]));
      // valid columns are [0, lim)
      int lim = 128;
      if (j < p.t_sel) {
        const int rem = (p.n_sel - j * ppt) * p.page_size;
        lim = rem < 128 ? rem : 128;
      } else if (j - p.t_sel == qt) {
        lim = r + 1;
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        x[c] = (c < lim) ? x[c] * p.scale_log2 : -INFINITY;
        mt = fmaxf(mt, x[c]);
      }
      if (j == 0) {
        m = mt;
      } else {
        const float m_new = fmaxf(m, mt);
        const bool need = m_new > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const int pb = (j - 1) & 1;
          ok = __all_sync(0xffffffffu,
                          mbar_wait(BAR(o_done[pb]), ((j - 1) >> 1) & 1, wc, kWhereFwdSoftmax));
          if (!ok) break;
          tc_fence_after();
          const float alpha = need ? ex2(m - m_new) : 1.f;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t rr[32];
            tmem_ld32(t_o + c4 * 32, rr);
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
            tmem_st32(t_o + c4 * 32, rr);
          }
          tmem_st_wait();
          if (need) {
            l *= alpha;
            m = m_new;
          }
        }
      }
      if (j >= 2) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(BAR(o_done[b]), ((j - 2) >> 1) & 1, wc, kWhereFwdSoftmax));
        if (!ok) break;
      }
      // P_j row r -> shared, bf16, swizzled K-major (keys are the K dimension)
      const uint32_t prow = sbase + kPOff + b * kTileBytes;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        float e[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          e[i] = ex2(x[c * 8 + i] - m);
          rs += e[i];
        }
        st_shared_v4(prow + tile128_chunk_off(r, c), pack_bf16(e[0], e[1]), pack_bf16(e[2], e[3]),
                     pack_bf16(e[4], e[5]), pack_bf16(e[6], e[7]));
      }
      l += rs;
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(BAR(p_full[b]));
    }
    if (ok) {
      const int jl = n_tiles - 1;
      ok = __all_sync(0xffffffffu,
                      mbar_wait(BAR(o_done[jl & 1]), (jl >> 1) & 1, wc, kWhereFwdSoftmax));
    }
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l;
      const bool row_ok = t < p.chunk_len;
      uint4* orow = reinterpret_cast<uint4*>(p.o + (static_cast<long>(t) * p.hq + h) * 128);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t rr[32];
        tmem_ld32(t_o + c4 * 32, rr);
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(rr[8 * i]) * inv, __uint_as_float(rr[8 * i + 1]) * inv);
            v.y = pack_bf16(__uint_as_float(rr[8 * i + 2]) * inv, __uint_as_float(rr[8 * i + 3]) * inv);
            v.z = pack_bf16(__uint_as_float(rr[8 * i + 4]) * inv, __uint_as_float(rr[8 * i + 5]) * inv);
            v.w = pack_bf16(__uint_as_float(rr[8 * i + 6]) * inv, __uint_as_float(rr[8 * i + 7]) * inv);
            orow[c4 * 4 + i] = v;
          }
        }
      }
      if (row_ok)
        p.lse[static_cast<long>(h) * p.chunk_len + t] = (m + __log2f(l)) * 0.69314718055994530942f;
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
                                 float* lse, int* status, uint64_t wait_ns, cudaStream_t st) {
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
  p.lse = lse;
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
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(sparse_attn_fwd_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  sparse_attn_fwd_kernel<<<p.n_qtiles * hq, kThreads, kSmemBytes, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace oomb
