// Device-side building blocks shared by the sm_103a kernels: shared-memory
// barriers (mbarrier) with bounded waits, TMA tile loads, and the tcgen05
// tensor-core / tensor-memory (TMEM) instructions, all as inline PTX.
//
// Every spin-wait here gives up after a time limit read from %globaltimer;
// the caller then records SPARGE_ERR_TIMEOUT in the status word and returns,
// so a logic error can never hang the GPU.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sparge.h"

#define SPARGE_DEV __device__ __forceinline__

namespace sparge {

// Default limit for one barrier wait (2 s); a wait that passes it aborts the CTA.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

SPARGE_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

SPARGE_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Records the first error code of a launch in the caller's status word.
SPARGE_DEV void report_error(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

// ----------------------------------------------------------------- mbarrier
SPARGE_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
SPARGE_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
SPARGE_DEV void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}
SPARGE_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}
// Adds `bytes` to the transaction count of the current phase (no arrival).
SPARGE_DEV void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
SPARGE_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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
// Non-blocking test: true when the phase with the given parity has completed.
SPARGE_DEV bool mbar_test_wait(uint32_t bar, uint32_t parity) {
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
// Waits for the phase with the given parity to complete; false after the limit.
SPARGE_DEV bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// Every lane of the warp waits; the result is the same in all lanes (a lane
// that timed out makes the whole warp report failure), so warp-wide tcgen05
// instructions after it stay convergent.
SPARGE_DEV bool warp_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns = kWaitTimeoutNs) {
  const bool ok = mbar_wait(bar, parity, timeout_ns);
  return __all_sync(0xffffffffu, ok);
}

// 16-byte read-only global load that does not allocate in L1 (for data each
// thread reads once while streaming).
SPARGE_DEV uint4 ldg_no_l1(const uint4* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

// ----------------------------------------------------------------- fences
SPARGE_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
SPARGE_DEV void named_barrier_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ----------------------------------------------------------------- TMA
SPARGE_DEV void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}
// 3-D tiled load (coordinates innermost first) completing on an mbarrier.
SPARGE_DEV void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// ----------------------------------------------------------------- tcgen05
SPARGE_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
SPARGE_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
SPARGE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
SPARGE_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SPARGE_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Arrives once on `bar` when every tcgen05 op issued so far by this thread completes.
SPARGE_DEV void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// D(tmem) (+)= A(smem) * B(smem)^T, bf16 inputs, fp32 accumulate.
SPARGE_DEV void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f16 with bf16 A/B and an fp32 accumulator.
// a_mn / b_mn select the MN-major ("transposed") smem layout of A / B.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                            // D format: f32
         | (1u << 7)                          // A format: bf16
         | (1u << 10)                         // B format: bf16
         | ((a_mn ? 1u : 0u) << 15)           // A major
         | ((b_mn ? 1u : 0u) << 16)           // B major
         | (static_cast<uint32_t>(N >> 3) << 17)
         | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor for the 128-byte swizzled canonical layout.
// K-major: rows of 128 B, 8-row atoms of 1024 B, `sbo` = stride between atoms
// along M/N (lbo unused).  MN-major: 64-element (128 B) rows along M/N, 8 rows
// along K per atom; `lbo` = stride between 64-element chunks along M/N, `sbo` =
// stride between 8-row groups along K.  Atoms must be 1024-byte aligned.
SPARGE_DEV uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Moves a shared-memory descriptor's start address by `bytes` (a multiple of
// 16).  Shared addresses stay below 2^18, so the 14-bit field cannot carry.
// Issue loops add constant offsets to a base descriptor built once per tile:
// rebuilding both descriptors per MMA costs about 63 cycles of issue per
// 128 x 64 x 16 MMA on sm_103a, more than the 48 the tensor pipe needs.
SPARGE_DEV uint64_t sdesc_add(uint64_t desc, uint32_t bytes) {
  return desc + static_cast<uint64_t>(bytes >> 4);
}

// Byte offset of element (row, col) of a bf16 tile stored as 128-byte rows with
// the 128-byte swizzle (16-byte chunk index XOR row % 8); tile base 1024-aligned.
SPARGE_DEV uint32_t sw128_offset(uint32_t row, uint32_t col_bytes) {
  return row * 128u + ((((col_bytes >> 4) ^ (row & 7u)) << 4) | (col_bytes & 15u));
}

// TMEM loads: 32 lanes x 32-bit, N consecutive columns per thread.
#define SPARGE_TMEM_LD_X16(taddr, r)                                                        \
  asm volatile(                                                                             \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
      "%14,%15}, [%16];"                                                                    \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),  \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),          \
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])                                               \
      : "r"(taddr))

// Waits for prior tcgen05.ld; the registers are tied in so no use can be
// scheduled before the wait.
#define SPARGE_TMEM_WAIT_LD16(r)                                                            \
  asm volatile("tcgen05.wait::ld.sync.aligned;"                                             \
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),    \
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),  \
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])::"memory")

// Loads 32 fp32 columns of one TMEM lane starting at `addr` (warp-wide;
// the warp's lane quarter is the one it may access).
SPARGE_DEV void tmem_ld32(uint32_t addr, float (&x)[32]) {
  uint32_t ra[16], rb[16];
  SPARGE_TMEM_LD_X16(addr + 0, ra);
  SPARGE_TMEM_LD_X16(addr + 16, rb);
  SPARGE_TMEM_WAIT_LD16(ra);
  SPARGE_TMEM_WAIT_LD16(rb);
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    x[c] = __uint_as_float(ra[c]);
    x[16 + c] = __uint_as_float(rb[c]);
  }
}

#define SPARGE_TMEM_ST_X16(taddr, r)                                                        \
  asm volatile(                                                                             \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12," \
      "%13,%14,%15,%16};" ::"r"(taddr),                                                     \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),     \
      "r"(r[15])                                                                            \
      : "memory")

#define SPARGE_TMEM_ST_X8(taddr, r)                                                         \
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), \
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),       \
               "r"(r[7])                                                                          \
               : "memory")

SPARGE_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// TMEM address of (lane, column) relative to an allocation base.
SPARGE_DEV uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

SPARGE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x by the hardware approximation (MUFU.EX2), subnormal results flushed.
// Packed fp32 pairs: fma / add / mul on two fp32 values in one instruction
// (sm_100 and later), each lane rounded to nearest like the scalar forms, so
// results are bit-identical to fmaf / + / *.  They halve the issue slots of the
// elementwise work between the MMAs.
SPARGE_DEV uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
SPARGE_DEV float f32x2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
SPARGE_DEV float f32x2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
SPARGE_DEV uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
SPARGE_DEV uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
SPARGE_DEV uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Three-input fp32 max / min (one instruction on sm_100 and later).
SPARGE_DEV float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
SPARGE_DEV float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

SPARGE_DEV float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

SPARGE_DEV uint32_t elect_lane0() { return (threadIdx.x & 31u) == 0u; }

// One lane of a converged warp, chosen by elect.sync (the lowest active lane:
// with the full warp converged, the same lane every time, so the MMAs and the
// commits that track them come from one thread).
//
// MMA issue from a converged warp: every lane runs the issue loop (waits,
// descriptor arithmetic) and each tcgen05.mma / tcgen05.commit sits in its own
// elect.sync branch.  Measured on sm_103a with a drained pipe: 27 cycles per
// 128 x 64 x 16 MMA issued this way against 61 when one lane runs the loop
// alone in a divergent branch -- and at 48 to 64 cycles per MMA the tensor
// pipe is otherwise starved by its own issuer.
SPARGE_DEV bool elect_sync() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}
SPARGE_DEV void warp_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                              uint32_t accumulate) {
  if (elect_sync()) tc_mma_bf16(d_tmem, adesc, bdesc, idesc, accumulate);
  __syncwarp();
}
// D(tmem) (+)= A(tmem) * B(smem): A is M x 16 bf16 in TMEM (lane = row, column c
// holds elements 2c, 2c + 1).
SPARGE_DEV void tc_mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
SPARGE_DEV void warp_mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                 uint32_t accumulate) {
  if (elect_sync()) tc_mma_bf16_ta(d_tmem, a_tmem, bdesc, idesc, accumulate);
  __syncwarp();
}
SPARGE_DEV void warp_commit(uint32_t bar) {
  if (elect_sync()) tc_commit(bar);
  __syncwarp();
}

}  // namespace sparge
