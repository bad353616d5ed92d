// fp32 forward and backward of the page-level sparse attention on CUDA cores
// (FFMA), head_dim 64.  This path serves fp32 workloads, whose 1e-4 accuracy
// TF32 tensor cores cannot reach.  Same key set as the bf16 path: every token
// of the selected pages, then the chunk's own tokens up to the query position.
#include <cuda_runtime.h>

#include <cstdint>

#include "oomb_internal.h"
#include "sm100.cuh"

namespace oomb {
namespace {

constexpr int D = 64;
constexpr int KC = 32;   // keys per shared-memory chunk

struct KeyMap {
  const int32_t* pt;
  const int32_t* sel_g;  // sel row of this KV head
  int n_sel, page_size, num_slots, hkv, g, own_page0, n_cand, n_own_pages;
  // Global row (in units of D floats) of key kk of the key list, or -1 if the
  // index is invalid (recorded as a bounds error).
  __device__ long row(int kk, int* status) const {
    const int sel_keys = n_sel * page_size;
    int lp, off;
    if (kk < sel_keys) {
      lp = sel_g[kk / page_size];
      off = kk % page_size;
      if (lp < 0 || lp >= n_cand) {
        raise_status(status, kStatusBounds, kWhereFp32);
        return -1;
      }
    } else {
      const int u = kk - sel_keys;
      if (u / page_size >= n_own_pages) return -1;
      lp = own_page0 + u / page_size;
      off = u % page_size;
    }
    const int slot = pt[lp];
    if (slot < 0 || slot >= num_slots) {
      raise_status(status, kStatusBounds, kWhereFp32);
      return -1;
    }
    return (static_cast<long>(slot) * hkv + g) * page_size + off;
  }
};

// One CTA = 128 query rows of one head; thread = query row.
__global__ void __launch_bounds__(128) fwd_fp32_kernel(const float* __restrict__ q,
                                                       const float* __restrict__ kp,
                                                       const float* __restrict__ vp, KeyMap km0,
                                                       int hq, int chunk_len, float scale_log2,
                                                       float* __restrict__ o,
                                                       float* __restrict__ lse, int* status) {
  __shared__ float4 ks[KC][D / 4];
  __shared__ float4 vs[KC][D / 4];
  __shared__ int kvalid[KC];
  const int h = blockIdx.y, grp = hq / km0.hkv, g = h / grp;
  KeyMap km = km0;
  km.g = g;
  km.sel_g = km0.sel_g + static_cast<long>(g) * km0.n_sel;
  const int t = blockIdx.x * 128 + threadIdx.x;
  const int t_last = min(chunk_len, (blockIdx.x + 1) * 128) - 1;
  const int sel_keys = km.n_sel * km.page_size;
  const int nk = sel_keys + t_last + 1;
  float qr[D], acc[D];
  const bool row_ok = t < chunk_len;
#pragma unroll
  for (int d = 0; d < D; ++d) {
    qr[d] = row_ok ? q[(static_cast<long>(t) * hq + h) * D + d] : 0.f;
    acc[d] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int k0 = 0; k0 < nk; k0 += KC) {
    {
      const int j = threadIdx.x >> 2, part = threadIdx.x & 3;
      const int kk = k0 + j;
      long r = -1;
      if (kk < nk) r = km.row(kk, status);
      if (part == 0) kvalid[j] = (r >= 0);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = part * 4 + i;
        ks[j][c] = r >= 0 ? reinterpret_cast<const float4*>(kp + r * D)[c] : make_float4(0, 0, 0, 0);
        vs[j][c] = r >= 0 ? reinterpret_cast<const float4*>(vp + r * D)[c] : make_float4(0, 0, 0, 0);
      }
    }
    __syncthreads();
    float s[KC];
    float cmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      const int kk = k0 + j;
      float dot = 0.f;
#pragma unroll
      for (int c = 0; c < D / 4; ++c) {
        const float4 kv = ks[j][c];
        dot = fmaf(qr[4 * c], kv.x, dot);
        dot = fmaf(qr[4 * c + 1], kv.y, dot);
        dot = fmaf(qr[4 * c + 2], kv.z, dot);
        dot = fmaf(qr[4 * c + 3], kv.w, dot);
      }
      const bool ok = kvalid[j] && kk < nk && (kk < sel_keys || kk - sel_keys <= t);
      s[j] = ok ? dot * scale_log2 : -INFINITY;
      cmax = fmaxf(cmax, s[j]);
    }
    const float m_new = fmaxf(m, cmax);
    if (m_new > -INFINITY) {
      const float alpha = exp2f(m - m_new);
      l *= alpha;
#pragma unroll
      for (int d = 0; d < D; ++d) acc[d] *= alpha;
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        const float p = exp2f(s[j] - m_new);
        l += p;
#pragma unroll
        for (int c = 0; c < D / 4; ++c) {
          const float4 vv = vs[j][c];
          acc[4 * c] = fmaf(p, vv.x, acc[4 * c]);
          acc[4 * c + 1] = fmaf(p, vv.y, acc[4 * c + 1]);
          acc[4 * c + 2] = fmaf(p, vv.z, acc[4 * c + 2]);
          acc[4 * c + 3] = fmaf(p, vv.w, acc[4 * c + 3]);
        }
      }
      m = m_new;
    }
    __syncthreads();
  }
  if (row_ok) {
    const float inv = 1.f / l;
#pragma unroll
    for (int d = 0; d < D; ++d) o[(static_cast<long>(t) * hq + h) * D + d] = acc[d] * inv;
    lse[static_cast<long>(h) * chunk_len + t] = (m + log2f(l)) * 0.69314718055994530942f;
  }
}

__global__ void delta_fp32_kernel(const float* __restrict__ o, const float* __restrict__ dout,
                                  int hq, int chunk_len, float* __restrict__ delta) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;   // i = t * hq + h
  if (i >= chunk_len * hq) return;
  const float4* a = reinterpret_cast<const float4*>(o + static_cast<long>(i) * D);
  const float4* b = reinterpret_cast<const float4*>(dout + static_cast<long>(i) * D);
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < D / 4; ++c) {
    const float4 x = a[c], y = b[c];
    s = fmaf(x.x, y.x, s); s = fmaf(x.y, y.y, s); s = fmaf(x.z, y.z, s); s = fmaf(x.w, y.w, s);
  }
  const int t = i / hq, h = i % hq;
  delta[static_cast<long>(h) * chunk_len + t] = s;
}

// dq: thread = query row, same key walk as the forward.
__global__ void __launch_bounds__(128) dq_fp32_kernel(
    const float* __restrict__ q, const float* __restrict__ dout, const float* __restrict__ lse,
    const float* __restrict__ delta, const float* __restrict__ kp, const float* __restrict__ vp,
    KeyMap km0, int hq, int chunk_len, float scale, float* __restrict__ dq, int* status) {
  __shared__ float4 ks[KC][D / 4];
  __shared__ float4 vs[KC][D / 4];
  __shared__ int kvalid[KC];
  const int h = blockIdx.y, grp = hq / km0.hkv, g = h / grp;
  KeyMap km = km0;
  km.g = g;
  km.sel_g = km0.sel_g + static_cast<long>(g) * km0.n_sel;
  const int t = blockIdx.x * 128 + threadIdx.x;
  const int t_last = min(chunk_len, (blockIdx.x + 1) * 128) - 1;
  const int sel_keys = km.n_sel * km.page_size;
  const int nk = sel_keys + t_last + 1;
  const bool row_ok = t < chunk_len;
  const float LOG2E = 1.4426950408889634f;
  const float sl2 = scale * LOG2E;
  float qr[D], dor[D], acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) {
    qr[d] = row_ok ? q[(static_cast<long>(t) * hq + h) * D + d] : 0.f;
    dor[d] = row_ok ? dout[(static_cast<long>(t) * hq + h) * D + d] : 0.f;
    acc[d] = 0.f;
  }
  const float lse2 = row_ok ? lse[static_cast<long>(h) * chunk_len + t] * LOG2E : 0.f;
  const float dl = row_ok ? delta[static_cast<long>(h) * chunk_len + t] : 0.f;
  for (int k0 = 0; k0 < nk; k0 += KC) {
    {
      const int j = threadIdx.x >> 2, part = threadIdx.x & 3;
      const int kk = k0 + j;
      long r = -1;
      if (kk < nk) r = km.row(kk, status);
      if (part == 0) kvalid[j] = (r >= 0);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = part * 4 + i;
        ks[j][c] = r >= 0 ? reinterpret_cast<const float4*>(kp + r * D)[c] : make_float4(0, 0, 0, 0);
        vs[j][c] = r >= 0 ? reinterpret_cast<const float4*>(vp + r * D)[c] : make_float4(0, 0, 0, 0);
      }
    }
    __syncthreads();
    for (int j = 0; j < KC; ++j) {
      const int kk = k0 + j;
      const bool ok = row_ok && kvalid[j] && kk < nk && (kk < sel_keys || kk - sel_keys <= t);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int c = 0; c < D / 4; ++c) {
        const float4 kv = ks[j][c], vv = vs[j][c];
        s = fmaf(qr[4 * c], kv.x, s); s = fmaf(qr[4 * c + 1], kv.y, s);
        s = fmaf(qr[4 * c + 2], kv.z, s); s = fmaf(qr[4 * c + 3], kv.w, s);
        dp = fmaf(dor[4 * c], vv.x, dp); dp = fmaf(dor[4 * c + 1], vv.y, dp);
        dp = fmaf(dor[4 * c + 2], vv.z, dp); dp = fmaf(dor[4 * c + 3], vv.w, dp);
      }
      const float p = ok ? exp2f(s * sl2 - lse2) : 0.f;
      const float ds = p * (dp - dl);
#pragma unroll
      for (int c = 0; c < D / 4; ++c) {
        const float4 kv = ks[j][c];
        acc[4 * c] = fmaf(ds, kv.x, acc[4 * c]);
        acc[4 * c + 1] = fmaf(ds, kv.y, acc[4 * c + 1]);
        acc[4 * c + 2] = fmaf(ds, kv.z, acc[4 * c + 2]);
        acc[4 * c + 3] = fmaf(ds, kv.w, acc[4 * c + 3]);
      }
    }
    __syncthreads();
  }
  if (row_ok) {
#pragma unroll
    for (int d = 0; d < D; ++d) dq[(static_cast<long>(t) * hq + h) * D + d] = acc[d] * scale;
  }
}

// dK/dV: two threads per key (32 dims each); CTA = 64 keys of one KV head;
// loops over the G heads of the group and the query rows that see the key,
// then adds its sums into the paged fp32 gradient buffers (one owner per key).
constexpr int QC = 32;
__global__ void __launch_bounds__(128) dkdv_fp32_kernel(
    const float* __restrict__ q, const float* __restrict__ dout, const float* __restrict__ lse,
    const float* __restrict__ delta, const float* __restrict__ kp, const float* __restrict__ vp,
    float* __restrict__ dkp, float* __restrict__ dvp, KeyMap km0, int hq, int chunk_len,
    float scale, int* status) {
  __shared__ float qs[QC][D];
  __shared__ float dos[QC][D];
  __shared__ float lse2s[QC], dls[QC];
  const int g = blockIdx.y, grp = hq / km0.hkv;
  KeyMap km = km0;
  km.g = g;
  km.sel_g = km0.sel_g + static_cast<long>(g) * km0.n_sel;
  const int sel_keys = km.n_sel * km.page_size;
  const int nk = sel_keys + chunk_len;
  const int kk = blockIdx.x * 64 + (threadIdx.x >> 1);
  const int half = threadIdx.x & 1;
  const float LOG2E = 1.4426950408889634f;
  const float sl2 = scale * LOG2E;
  long r = -1;
  if (kk < nk) r = km.row(kk, status);
  const bool key_ok = r >= 0;
  float kr[32], vr[32], dk[32], dv[32];
#pragma unroll
  for (int d = 0; d < 32; ++d) {
    kr[d] = key_ok ? kp[r * D + half * 32 + d] : 0.f;
    vr[d] = key_ok ? vp[r * D + half * 32 + d] : 0.f;
    dk[d] = 0.f;
    dv[d] = 0.f;
  }
  // first query row that may see any key of this CTA
  const int kk0 = blockIdx.x * 64;
  const int t_begin = kk0 < sel_keys ? 0 : ((kk0 - sel_keys) / QC) * QC;
  for (int h = g * grp; h < (g + 1) * grp; ++h) {
    for (int tc = t_begin; tc < chunk_len; tc += QC) {
      __syncthreads();
      for (int i = threadIdx.x; i < QC * D; i += blockDim.x) {
        const int j = i / D, d = i % D, t = tc + j;
        qs[j][d] = t < chunk_len ? q[(static_cast<long>(t) * hq + h) * D + d] : 0.f;
        dos[j][d] = t < chunk_len ? dout[(static_cast<long>(t) * hq + h) * D + d] : 0.f;
      }
      if (threadIdx.x < QC) {
        const int t = tc + threadIdx.x;
        lse2s[threadIdx.x] = t < chunk_len ? lse[static_cast<long>(h) * chunk_len + t] * LOG2E : 0.f;
        dls[threadIdx.x] = t < chunk_len ? delta[static_cast<long>(h) * chunk_len + t] : 0.f;
      }
      __syncthreads();
      for (int j = 0; j < QC; ++j) {
        const int t = tc + j;
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int d = 0; d < 32; ++d) {
          s = fmaf(qs[j][half * 32 + d], kr[d], s);
          dp = fmaf(dos[j][half * 32 + d], vr[d], dp);
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        dp += __shfl_xor_sync(0xffffffffu, dp, 1);
        const bool ok = key_ok && t < chunk_len && (kk < sel_keys || kk - sel_keys <= t);
        const float p = ok ? exp2f(s * sl2 - lse2s[j]) : 0.f;
        const float ds = p * (dp - dls[j]);
#pragma unroll
        for (int d = 0; d < 32; ++d) {
          dk[d] = fmaf(ds, qs[j][half * 32 + d], dk[d]);
          dv[d] = fmaf(p, dos[j][half * 32 + d], dv[d]);
        }
      }
    }
  }
  if (key_ok) {
#pragma unroll
    for (int d = 0; d < 32; ++d) {
      dkp[r * D + half * 32 + d] += scale * dk[d];
      dvp[r * D + half * 32 + d] += dv[d];
    }
  }
}

KeyMap make_keymap(const KvDesc& kv, const int32_t* sel, int n_sel, int chunk_len,
                   int chunk_start) {
  KeyMap km;
  km.pt = kv.page_table;
  km.sel_g = sel;
  km.n_sel = n_sel;
  km.page_size = kv.page_size;
  km.num_slots = kv.num_slots;
  km.hkv = kv.hkv;
  km.g = 0;
  km.own_page0 = chunk_start / kv.page_size;
  km.n_cand = chunk_start / kv.page_size;
  km.n_own_pages = (chunk_len + kv.page_size - 1) / kv.page_size;   // the last may be partial
  return km;
}

}  // namespace

size_t fp32_bwd_ws_bytes(int hq, int chunk_len) {
  return kStatusBytes + align_up(static_cast<size_t>(hq) * chunk_len * 4, 256);
}

cudaError_t launch_attn_fwd_fp32(const float* q, const KvDesc& kv, const int32_t* sel, int n_sel,
                                 int hq, int chunk_len, int chunk_start, float scale, float* o,
                                 float* lse, int* status, cudaStream_t st) {
  const KeyMap km = make_keymap(kv, sel, n_sel, chunk_len, chunk_start);
  const dim3 grid((chunk_len + 127) / 128, hq);
  fwd_fp32_kernel<<<grid, 128, 0, st>>>(q, static_cast<const float*>(kv.k),
                                        static_cast<const float*>(kv.v), km, hq, chunk_len,
                                        scale * 1.4426950408889634f, o, lse, status);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_fp32(const float* q, const float* o, const float* dout,
                                 const float* lse, const KvDesc& kv, const int32_t* sel,
                                 int n_sel, int hq, int chunk_len, int chunk_start, float scale,
                                 float* dq, void* ws, cudaStream_t st) {
  int* status = static_cast<int*>(ws);
  float* delta = reinterpret_cast<float*>(static_cast<char*>(ws) + kStatusBytes);
  const KeyMap km = make_keymap(kv, sel, n_sel, chunk_len, chunk_start);
  const int n = chunk_len * hq;
  delta_fp32_kernel<<<(n + 255) / 256, 256, 0, st>>>(o, dout, hq, chunk_len, delta);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dq_fp32_kernel<<<dim3((chunk_len + 127) / 128, hq), 128, 0, st>>>(
      q, dout, lse, delta, static_cast<const float*>(kv.k), static_cast<const float*>(kv.v), km,
      hq, chunk_len, scale, dq, status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int nk = n_sel * kv.page_size + chunk_len;
  dkdv_fp32_kernel<<<dim3((nk + 63) / 64, kv.hkv), 128, 0, st>>>(
      q, dout, lse, delta, static_cast<const float*>(kv.k), static_cast<const float*>(kv.v),
      static_cast<float*>(kv.dk), static_cast<float*>(kv.dv), km, hq, chunk_len, scale, status);
  return cudaGetLastError();
}

}  // namespace oomb
