// moe_ptx.cuh -- thin inline-PTX wrappers used by the streaming kernels:
// mbarriers with bounded waits, TMA bulk copies, fp4 -> f16 converts and the
// f16 tensor-core MMA.  Internal header.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `parity` to complete.  Gives up after
// `limit_cycles` SM clock cycles and returns false (the caller records an
// error and winds down); never spins forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  long long limit_cycles,
                                                  const volatile int *global_err = nullptr) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    // the clock (and the grid-wide error word, set by any CTA that gave up)
    // is read every 64 polls only (try_wait itself suspends the thread for a
    // short while when the phase is not complete)
    if ((n & 63) == 0) {
      if (clock64() - t0 > limit_cycles) return false;
      if (global_err && *global_err) return false;
    }
  }
}

// Acquire load of a global counter (gpu scope).
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Waits until the global counter *p reaches `need` (written by other CTAs of
// the same grid that are already running), for at most `limit_cycles`;
// returns false on timeout or when the grid-wide error word is set.
__device__ __forceinline__ bool wait_count_bounded(const int *p, int need, long long limit_cycles,
                                                   const volatile int *global_err) {
  if (ld_acquire_gpu(p) >= need) return true;
  const long long t0 = clock64();
  while (ld_acquire_gpu(p) < need) {
    if (clock64() - t0 > limit_cycles) return false;
    if (global_err && *global_err) return false;
    __nanosleep(256);
  }
  return true;
}

// Programmatic dependent launch.  griddep_wait: the calling thread waits until
// the grid launched before this one in the stream has completed and its memory
// is visible (a no-op when this grid was not launched as a dependent).
// griddep_launch_dependents: this CTA allows the next grid in the stream, if
// launched as a dependent, to start (it still waits for completion itself).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Orders this thread's earlier generic-proxy view of global memory before its
// later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// TMA bulk copy global -> shared (this CTA), completing `bytes` of
// transaction count on `bar`.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void tma_bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                             uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Bulk prefetch of global memory into L2 (a hint; no completion to wait for).
// src and bytes must be multiples of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Four bytes of packed e2m1 pairs -> four f16x2 registers (low nibble in the
// low half), one hardware convert per byte.  Exact: every e2m1 value is an
// f16 value.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

__device__ __forceinline__ void ldmatrix_x4_b16(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x2_b16(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1, const float (&c)[4]) {
  // register-only: not volatile, so the compiler may interleave it with the
  // surrounding conversions
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

}  // namespace moe

// ----------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core) and tensor TMA wrappers.
namespace moe {

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tiled TMA load (tensor map in param / const / global space).
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int x, int y,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// TMEM allocation (one full warp); the allocated base address is written to
// shared memory at `dst`.  ncols: power of two >= 32.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16/f16 operands,
// fp32 accumulate); issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand tile laid out by TMA
// (or by hand) with the 128-byte swizzle: rows of 128 bytes, groups of 8 rows
// 1024 bytes apart.  Advancing the start address by 32 bytes moves 16 bf16
// elements along K inside the swizzle atom.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);   // start address
  d |= (uint64_t)1 << 16;                     // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                     // descriptor version
  d |= (uint64_t)2 << 61;                     // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, f16 x f16 -> fp32, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int m, int n) {
  return (1u << 4)                       // D format fp32
         | ((uint32_t)(n >> 3) << 17)    // A, B format f16 (0)
         | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Instruction descriptor: kind::f16, bf16 x bf16 -> fp32, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int m, int n) {
  return (1u << 4)                       // D format fp32
         | (1u << 7)                     // A format bf16
         | (1u << 10)                    // B format bf16
         | ((uint32_t)(n >> 3) << 17)    // N
         | ((uint32_t)(m >> 4) << 24);   // M
}

}  // namespace moe

namespace moe {

// D[tmem] (+)= A * B^T, kind::f8f6f4 (e4m3 x e4m3 here), fp32 accumulate.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor: kind::f8f6f4, e4m3 x e4m3 -> fp32, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_e4m3(int m, int n) {
  return (1u << 4)                       // D format fp32
         | (0u << 7)                     // A format e4m3
         | (0u << 10)                    // B format e4m3
         | ((uint32_t)(n >> 3) << 17)
         | ((uint32_t)(m >> 4) << 24);
}

// d0 += a0 * s, d1 += a1 * s in one packed fp32x2 FMA (round to nearest).
__device__ __forceinline__ void fma_f32x2(float &d0, float &d1, float a0, float a1, float s) {
  asm("{\n\t.reg .b64 pa, pd, ps;\n\t"
      "mov.b64 pa, {%2, %3};\n\t"
      "mov.b64 pd, {%0, %1};\n\t"
      "mov.b64 ps, {%4, %4};\n\t"
      "fma.rn.f32x2 pd, pa, ps, pd;\n\t"
      "mov.b64 {%0, %1}, pd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(s));
}

}  // namespace moe

// ----------------------------------------------------------------------------
// Block-scaled tcgen05 MMA (PTX ISA, "tcgen05.mma" with .block_scale, and
// "tcgen05.cp"; the forms below are the ones the ISA lists for sm_100a /
// sm_103a: kind::mxf4nvf4 with .scale_vec::4X, 32x128b.warpx4 copies).
namespace moe {

// D[tmem] (+)= (A .* SFA) * (B .* SFB)^T, kind::mxf4nvf4, scale_vec::4X: A and
// B are packed e2m1 (two per byte, K-major, 64 elements = 32 bytes per
// instruction), each 16-element block of a row carries one ue4m3 scale
// factor; fp32 accumulate.  sfa / sfb: Tensor Memory addresses of the scale
// factors of this instruction's 64-element K step (layout: tc_sf_layout).
__device__ __forceinline__ void umma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::mxf4nvf4 (the ISA's descriptor table for
// .kind::mxf8f6f4 / .kind::mxf4 / .kind::mxf4nvf4), both operands K-major:
//   bits  0-1  sparsity selector (0), bit 2 dense (0), bit 3 reserved
//   bits  4-5  scale-factor id of B (0: the whole 32-bit word, 4X)
//   bits  7-9  A type: E2M1 = 1 (the mxf4 kinds' encoding)
//   bits 10-12 B type: E2M1 = 1
//   bits 13-14 negate A / B (0); bits 15-16 transpose A / B (0: K-major)
//   bits 17-22 N >> 3
//   bit  23    scale-factor type: UE4M3 = 0, UE8M0 = 1
//   bits 24-28 M >> 4
//   bits 29-30 scale-factor id of A (0)
//   bit  31    K of the instruction: 0 = 64 (dense)
// The accumulator is fp32 for these kinds (no D-type field).
__host__ __device__ constexpr uint32_t umma_idesc_nvf4(int m, int n) {
  return (1u << 7)                       // A: E2M1
         | (1u << 10)                    // B: E2M1
         | ((uint32_t)(n >> 3) << 17)    // N
         | (0u << 23)                    // scale factors UE4M3
         | ((uint32_t)(m >> 4) << 24);   // M
}

// Shared-memory descriptor of one scale-factor chunk for tcgen05.cp
// .32x128b: 32 rows of 16 bytes, no swizzle; core matrices (8 rows x 16 B)
// 128 bytes apart along the rows (stride byte offset); one core matrix wide,
// so the leading byte offset is not used.
__device__ __forceinline__ uint64_t sf_smem_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);   // start address
  d |= (uint64_t)(128 >> 4) << 32;           // stride byte offset
  d |= (uint64_t)1 << 46;                     // descriptor version
  return d;                                   // layout 0: no swizzle
}

// Shared-memory descriptor of a 128-row x 32-byte source for tcgen05.cp
// .128x256b: no swizzle, 8-row x 16-byte core matrices; the two core
// matrices of a row group 128 bytes apart (leading byte offset, along the
// row), row groups 256 bytes apart (stride byte offset).
__device__ __forceinline__ uint64_t sf256_smem_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);   // start address
  d |= (uint64_t)(128 >> 4) << 16;           // leading byte offset
  d |= (uint64_t)(256 >> 4) << 32;           // stride byte offset
  d |= (uint64_t)1 << 46;                     // descriptor version
  return d;                                   // layout 0: no swizzle
}

// Copy 128 rows x 256 bits from shared memory (descriptor) to Tensor Memory
// columns [taddr, taddr + 8): lane L, column c + w receives bytes
// [4 w, 4 w + 4) of row L.  Issued by one thread; ordered before the MMAs it
// issues later.
__device__ __forceinline__ void tc_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Copy 32 rows x 128 bits from shared memory (descriptor) to Tensor Memory
// columns [taddr, taddr + 4), replicated into all four 32-lane quarters
// (.warpx4): lane 32q + i, column c + w holds bytes [16 i + 4 w, 16 i + 4 w + 4)
// of the chunk.  Issued by one thread; ordered before the MMAs it issues later.
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

}  // namespace moe
