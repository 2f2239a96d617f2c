// tq_umma.cuh -- fifth-generation tensor-core (tcgen05) primitives for
// sm_103a: tensor-memory allocation, shared-memory matrix descriptors, the
// single-thread MMA issue, its completion through an mbarrier, and the
// tensor-memory loads of the accumulator.  Inline PTX only.
#pragma once

#include <stdint.h>

namespace tq {
namespace umma {

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(count) : "memory");
}
// Makes the initialisation visible to the asynchronous proxy (the MMA unit
// arrives on the barrier) before the CTA barrier that follows it.
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ bool mbar_try_wait(uint32_t mbar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(mbar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same with a suspend-time hint: the thread may sleep up to hint_ns
// (waking when the phase completes) instead of returning at once.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t mbar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(mbar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete, for at most
// limit_ns of wall-clock time; false when the time ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t mbar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(mbar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait_sleep(mbar, parity, 20000u)) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------- tensor memory
// Allocation and release are warp-wide; the allocated base address (lane 0,
// first column) is written to the shared-memory word at dst.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Ordering of tcgen05 operations around thread synchronisation.
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes made visible to the tensor core's
// (asynchronous-proxy) operand reads; each writing thread issues it before
// the CTA barrier that precedes the MMA.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout: rows of 128 bytes (64 fp16 values along K), 8-row groups
// of 1024 bytes one after the other (stride-dimension offset 1024 bytes),
// the 16-byte chunk c of row r stored at chunk position c ^ (r mod 8).  The
// group base must be 1024-byte aligned; a K step inside the 128-byte row
// advances the start address by its byte offset.  Fields: start address >> 4
// (bits 0-13), leading-dimension offset >> 4 (bits 16-29; not used by a
// swizzled K-major operand, set to 1), stride-dimension offset >> 4 (bits
// 32-45), descriptor version 1 (bits 46-47), base offset 0 (bits 49-51),
// swizzle mode 2 = 128-byte (bits 61-63).
__host__ __device__ constexpr uint64_t desc_sw128_kmajor(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16 with fp16 A and B, fp32 accumulator,
// both operands K-major, no negation, dense: D format (bits 4-5) 1 = f32,
// A format (bits 7-9) and B format (bits 10-12) 0 = f16, N >> 3 (bits
// 17-22), M >> 4 (bits 24-28).
template <int M, int N>
__host__ __device__ constexpr uint32_t idesc_f16_f32() {
  static_assert(M == 64 || M == 128, "M of a one-CTA MMA");
  static_assert(N % 16 == 0 && N >= 16 && N <= 256, "N of an M=128 MMA");
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The two encodings worked out by hand for the operands used here.
static_assert(idesc_f16_f32<128, 128>() == 0x08200010u, "D f32 = 1 << 4, N / 8 = 16 << 17, M / 16 = 8 << 24");
static_assert(desc_sw128_kmajor(0x400u) == 0x4000404000010040ull,
              "start 0x400 >> 4, LBO 1 << 16, SBO 64 << 32, version 1 << 46, 128-byte swizzle 2 << 61");

// --------------------------------------------------------------- the MMA
// D[M x N] (tensor memory, fp32) = A[M x K] B[N x K]^T (+ D when accumulate),
// K = 16, both operands in shared memory.  Issued by one thread.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the mbarrier when every MMA this thread issued before it
// has completed (their operand reads included).
__device__ __forceinline__ void commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar) : "memory");
}

// Thread t of the warp reads tensor-memory lane (lane field of taddr) + t,
// 32 consecutive 32-bit columns from the column field of taddr; waits for
// the load in the same statement so that no use of v can move above it.
// A warp may only address the 32 lanes of its own sub-partition
// (32 * (warp id mod 4) ...).
__device__ __forceinline__ void ld_32x32b_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

}  // namespace umma
}  // namespace tq
