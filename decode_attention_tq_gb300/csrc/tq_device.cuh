// tq_device.cuh -- device helpers shared by the libtq kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "tq.h"

namespace tq {

constexpr int kD = 128;       // head_dim supported by the kernels
constexpr int kM = 128;       // QJL sketch length supported by the kernels
constexpr int kTile = 16;     // tokens per attention tile (one mma M / K tile)
constexpr float kLog2e = 1.4426950408889634f;

// Power-of-two scales that keep fp16 MMA operands away from overflow and
// subnormals: centroids are stored x256, attention weights x64.
constexpr float kCentScale = 256.0f;
constexpr float kWeightScale = 64.0f;
// Lazy softmax bounds of the attention kernel: weights p * n / nu stay below
// 2^kLazyLog2 * kLazyNu = 512, so 512 * kWeightScale = 32768 fits in fp16.
constexpr float kLazyLog2 = 8.0f;
constexpr float kLazyNu = 2.0f;

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_half2_raw(__half lo, __half hi) {
  return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// Split x into fp16 hi + fp16 lo with hi + lo == x to ~2^-22 relative.
__device__ __forceinline__ void split_half(float x, __half &hi, __half &lo) {
  hi = __float2half_rn(x);
  lo = __float2half_rn(x - __half2float(hi));
}

// D[16x8] += A[16x16] * B[16x8], fp16 inputs, fp32 accumulation (row.col).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Programmatic dependent launch: a kernel launched as a dependent may start
// while the previous kernel on the stream runs; griddep_wait() blocks until
// that kernel has completed and its writes are visible (a no-op for a normal
// launch).  griddep_launch_dependents() lets the next dependent kernel start.
// Asynchronous global -> shared copies (no registers held while in flight);
// cp_async_wait_all() waits for all of this thread's copies.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((unsigned)__cvta_generic_to_shared(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async8(void *smem, const void *gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"((unsigned)__cvta_generic_to_shared(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void report(int32_t *err_word, int32_t bit) {
  if (err_word) atomicOr(err_word, bit);
}

__device__ __forceinline__ float warp_max_xor(float v, int lo_mask_bits) {
  // reduce over lanes differing in the lane-id bits set in lo_mask_bits
#pragma unroll
  for (int m = 1; m < 32; m <<= 1)
    if (lo_mask_bits & m) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

__device__ __forceinline__ float warp_sum_xor(float v, int lo_mask_bits) {
#pragma unroll
  for (int m = 1; m < 32; m <<= 1)
    if (lo_mask_bits & m) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// In-register butterflies of an unnormalized Walsh-Hadamard transform over
// the N values a thread holds (coordinates base..base+N-1, pairs (i, i+h)).
template <int N>
__device__ __forceinline__ void fwht_local(float (&x)[N]) {
#pragma unroll
  for (int h = 1; h < N; h <<= 1)
#pragma unroll
    for (int i = 0; i < N; i += 2 * h)
#pragma unroll
      for (int j = i; j < i + h; j++) {
        float a = x[j], b = x[j + h];
        x[j] = a + b;
        x[j + h] = a - b;
      }
}

// Cross-lane butterfly stage: partner lane = lane ^ lane_xor holds the
// coordinates (i XOR h); the lower lane keeps a + b, the upper one a - b.
template <int N>
__device__ __forceinline__ void fwht_xlane(float (&x)[N], int lane_xor, bool upper) {
#pragma unroll
  for (int i = 0; i < N; i++) {
    float other = __shfl_xor_sync(0xffffffffu, x[i], lane_xor);
    x[i] = upper ? (other - x[i]) : (x[i] + other);
  }
}

}  // namespace tq
