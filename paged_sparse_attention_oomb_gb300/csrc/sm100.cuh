// Blackwell (sm_100 family, built for sm_103a) primitives as inline PTX:
// mbarriers with bounded waits, TMA tiled loads, tcgen05 MMA / TMEM access and
// the shared-memory matrix descriptors those MMAs read.
//
// Shared-memory tile format used by every tensor-core operand here ("tile128"):
// a 128 x 128 bf16 matrix stored as two 64-column halves, each half 128 rows
// of 128 bytes in the 128-byte swizzle pattern (16-byte chunk c of row r is
// stored at chunk c ^ (r % 8)), half 1 at +16 KiB.  A TMA box of 64 x 128
// elements with CU_TENSOR_MAP_SWIZZLE_128B writes exactly one half.  The same
// bytes serve as a K-major operand (rows = M or N, columns = K) or as an
// MN-major operand (rows = K, columns = M or N) by choosing the descriptor.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace oomb {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread is suspended (issues nothing) until the
// phase completes or `hint_ns` nanoseconds pass, so waiting warps leave the
// issue slots to the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every wait in these kernels is bounded: after `limit_ns` nanoseconds it
// records a timeout (status word in global memory + CTA abort flag) and
// returns false; it also returns false early once another role of the CTA
// has raised the abort flag.  Callers then unwind without touching more data.
struct WaitCtl {
  int* status;                 // global: [0] status code, [1] where, [2] block
  volatile int* abort_flag;    // shared
  uint64_t limit_ns;
};

constexpr int kStatusTimeout = 4;
constexpr int kStatusBounds = 5;
constexpr int kStatusNonFinite = 6;

__device__ __forceinline__ void raise_status(int* status, int code, int where) {
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = where;
    status[2] = static_cast<int>(blockIdx.x);
  }
}

constexpr uint32_t kSleepHintNs = 200000;   // re-check abort flag and limit every 0.2 ms

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                          int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*c.abort_flag) return false;
    if (global_timer_ns() - t0 > c.limit_ns) {
      raise_status(c.status, kStatusTimeout, where);
      *c.abort_flag = 1;
      return false;
    }
  }
}

// Non-blocking probe of a phase: true once the phase with this parity is complete.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Same contract as mbar_wait, without the long suspend hint: for the warp that
// issues the MMAs, whose wake-up latency is on the critical path.
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                               int where) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (true) {
    // try_wait parks the warp in hardware until the phase completes (or a
    // short system time limit passes): no issue slots taken from the warps
    // sharing this SM sub-partition
    if (mbar_try_wait(bar, parity)) return true;
    if ((++n & 15u) == 0) {
      if (*c.abort_flag) return false;
      if (global_timer_ns() - t0 > c.limit_ns) {
        raise_status(c.status, kStatusTimeout, where);
        *c.abort_flag = 1;
        return false;
      }
    }
  }
}

// Wait used only while unwinding after an abort: a fixed, generous bound,
// independent of the (possibly tiny, test-set) limit of the normal waits.
__device__ __forceinline__ bool mbar_drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_sleep(bar, parity, kSleepHintNs)) {
    if (global_timer_ns() - t0 > 2000000000ull) return false;
  }
  return true;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Plain (untiled) bulk copy global -> shared; both addresses 16-byte aligned,
// size a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  __syncwarp();
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  __syncwarp();
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  __syncwarp();
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make generic-proxy shared-memory writes visible to the async proxy (MMA/TMA).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 in, fp32 accumulate.
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every MMA issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// One lane of a converged warp (the same lane every time): lets a whole warp
// run an issue loop in lockstep while a single thread issues the MMAs.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulator.
// a_mn / b_mn: operand stored MN-major (transposed) instead of K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n, bool a_mn, bool b_mn) {
  return (1u << 4)                                    // accumulator f32
         | (1u << 7)                                  // A bf16
         | (1u << 10)                                 // B bf16
         | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;   // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;   // 128-byte swizzle
  return d;
}

constexpr uint32_t kHalfBytes = 128 * 128;   // one 64-column half of a tile128
constexpr uint32_t kTileBytes = 2 * kHalfBytes;

// tile128 operand descriptors, split into a per-tile base (computed once) and a
// per-k-step constant added to the start-address field.  K-major (rows are M or
// N, columns are K): k-step kk covers columns [16 kk, 16 kk + 16) at byte
// offset (kk / 4) * 16 KiB + (kk % 4) * 32; leading byte offset 16, stride 1024.
// MN-major (rows are K, columns are M or N): k-step kk covers rows
// [16 kk, 16 kk + 16) at byte offset kk * 2048; leading byte offset one
// 64-column half, stride 1024.  The split is exact because shared addresses are
// below 256 KiB, so the 14-bit field never carries.  Keeps the MMA-issuing
// thread to a handful of instructions per MMA: it shares its SM sub-partition
// with busy compute warps.
__device__ __forceinline__ uint64_t desc_kmajor0(uint32_t tile) {
  return sdesc_sw128(tile, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mnmajor0(uint32_t tile) {
  return sdesc_sw128(tile, kHalfBytes, 1024);
}
__host__ __device__ constexpr uint64_t kstep_kmajor(int kk) {
  return static_cast<uint64_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
}
__host__ __device__ constexpr uint64_t kstep_mnmajor(int kk) {
  return static_cast<uint64_t>((kk * 2048) >> 4);
}
// Descriptor offset of a whole tile128 (stage s of a ring starts s tiles on).
constexpr uint64_t kTileDesc = kTileBytes >> 4;
// desc_mnmajor0(t) == desc_kmajor0(t) + kDescMn: only the leading-byte-offset
// field differs (16 bytes -> one 64-column half).
constexpr uint64_t kDescMn = static_cast<uint64_t>((kHalfBytes >> 4) - 1) << 16;
// Opaque copy: keeps the compiler from hoisting per-k-step descriptor sums out
// of a loop (which would pin dozens of 64-bit registers in the issuing thread).
__device__ __forceinline__ uint64_t opaque(uint64_t x) {
  uint64_t y;
  asm volatile("mov.b64 %0, %1;" : "=l"(y) : "l"(x));
  return y;
}
// Descriptor offset of a byte offset within shared memory.
__host__ __device__ constexpr uint64_t desc_off(uint32_t bytes) { return bytes >> 4; }

// Byte offset of the 16-byte chunk `c` (0..15, 8 bf16 each) of row `r` in a tile128.
__device__ __forceinline__ uint32_t tile128_chunk_off(int r, int c) {
  return (c >> 3) * kHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

#define OOMB_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                   "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
// 32 consecutive TMEM columns of this thread's lane -> 32 registers; waits for
// completion inside the same asm so no use of the registers can move above it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  __syncwarp();   // .sync.aligned: the whole warp must be converged here
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : OOMB_R8(0), OOMB_R8(8), OOMB_R8(16), OOMB_R8(24)
      : "r"(taddr)
      : "memory");
}
#undef OOMB_R8

#define OOMB_O8(a, i) "=r"(a[i]), "=r"(a[i + 1]), "=r"(a[i + 2]), "=r"(a[i + 3]), \
                      "=r"(a[i + 4]), "=r"(a[i + 5]), "=r"(a[i + 6]), "=r"(a[i + 7])
// 64 consecutive TMEM columns of this thread's lane, one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  __syncwarp();
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : OOMB_O8(r, 0), OOMB_O8(r, 8), OOMB_O8(r, 16), OOMB_O8(r, 24), OOMB_O8(r, 32),
        OOMB_O8(r, 40), OOMB_O8(r, 48), OOMB_O8(r, 56)
      : "r"(taddr)
      : "memory");
}
// 128 consecutive TMEM columns of this thread's lane (two x64 loads in flight
// together), one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  __syncwarp();
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,"
      "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
      "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%129];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : OOMB_O8(r, 0), OOMB_O8(r, 8), OOMB_O8(r, 16), OOMB_O8(r, 24), OOMB_O8(r, 32),
        OOMB_O8(r, 40), OOMB_O8(r, 48), OOMB_O8(r, 56), OOMB_O8(r, 64), OOMB_O8(r, 72),
        OOMB_O8(r, 80), OOMB_O8(r, 88), OOMB_O8(r, 96), OOMB_O8(r, 104), OOMB_O8(r, 112),
        OOMB_O8(r, 120)
      : "r"(taddr), "r"(taddr + 64)
      : "memory");
}
#undef OOMB_O8
// Warpgroup register reallocation (all four warps of the warpgroup execute it).
template <uint32_t N>
__device__ __forceinline__ void regs_increase() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_decrease() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
#define OOMB_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                   "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  __syncwarp();
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      OOMB_W8(0), OOMB_W8(8), OOMB_W8(16), OOMB_W8(24)
      : "memory");
}
#undef OOMB_W8
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Two floats -> packed bf16x2, `lo` in the low half (element with the lower index).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Packed FP32 pairs (sm_100 family): one instruction applies the scalar
// operation to both halves, each rounded exactly as the scalar instruction
// would be; `lo` is the low 32 bits.  Halves the instruction count of the
// element-wise softmax arithmetic, which is issue-bound.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// Maximum of three floats in one instruction (sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void red_add_f32(float* addr, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(a) : "memory");
}

}  // namespace oomb
