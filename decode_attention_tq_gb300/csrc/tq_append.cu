// tq_append.cu -- the per-step window roll of a decode step (sm_103a).
//
// A cache is compressed pages plus an fp16 recent window of W tokens kept as
// a ring per sequence ("TurboQuant Family Design Study for CPU and Browser
// WASM KV Caches", 'Packed format and complete bit accounting': the last W
// tokens stay fp16; 'Append cost and memory-bandwidth tradeoffs': the append
// runs once per generated token; 'Paging, lifecycle, and cache identity':
// fixed pages filled in order).  One block per sequence:
//
//   * W > 0, window not full: the new token goes to ring slot win_lens[b];
//   * W > 0, window full: the oldest token (ring slot win_head[b]) is copied
//     to the staging buffer with the page slot of compressed position
//     comp_lens[b], and the new token takes its ring slot;
//   * W == 0: the new token itself is staged.
//
// The staged tokens are then encoded into the pages by the encode kernel
// (slot -1: nothing staged).  A block updates only its own sequence's
// counters, after all of its threads have read them.
#include "tq_internal.cuh"

namespace tq {

namespace {

constexpr int kChunks = kD / 8;  // 16-byte chunks per head vector

__device__ __forceinline__ void copy16(__half *dst, const __half *src) {
  *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
}

__global__ void __launch_bounds__(256) window_roll_kernel(const RollArgs a) {
  const int b = blockIdx.x;
  const int W = a.W, H = a.H, P = a.P;
  const int len = W > 0 ? a.win_lens[b] : 0;
  const int head = W > 0 ? a.win_head[b] : 0;
  const int comp = a.comp_lens[b];
  __syncthreads();  // every thread has read the counters before thread 0 may write them

  const int n = H * kChunks;  // chunks per kind
  const int64_t vec0 = (int64_t)b * H;
  const int64_t win_h = (int64_t)W * kD;  // head stride inside a sequence's window
  // chunk i of the 2n (K then V): kind, head, element offset
  auto at = [&](int i, int &kind, int &h, int &e) {
    kind = i >= n;
    const int c = kind ? i - n : i;
    h = c / kChunks;
    e = (c % kChunks) * 8;
  };

  if (comp < 0 || (W > 0 && (len < 0 || len > W || head < 0 || head >= W))) {
    if (threadIdx.x == 0) {
      report(a.err_word, TQ_DEVERR_LENGTH);
      a.stage_slots[b] = -1;
    }
    return;
  }
  if (W > 0 && len < W) {  // fill the window
    for (int i = threadIdx.x; i < 2 * n; i += blockDim.x) {
      int kind, h, e;
      at(i, kind, h, e);
      const __half *src = (kind ? a.v_new : a.k_new) + (vec0 + h) * kD + e;
      __half *dst = (kind ? a.v_win : a.k_win) + vec0 * win_h + h * win_h + (int64_t)len * kD + e;
      copy16(dst, src);
    }
    if (threadIdx.x == 0) {
      a.stage_slots[b] = -1;
      a.win_lens[b] = len + 1;
    }
    return;
  }

  const int pi = comp / P;
  const int64_t page = pi < a.max_pages ? a.block_tables[(int64_t)b * a.max_pages + pi] : -1;
  if (page < 0 || page >= a.num_pages) {
    if (threadIdx.x == 0) {
      report(a.err_word, pi < a.max_pages ? TQ_DEVERR_PAGE_RANGE : TQ_DEVERR_LENGTH);
      a.stage_slots[b] = -1;
    }
    return;
  }
  // stage the token that leaves (or, without a window, the new one)
  for (int i = threadIdx.x; i < 2 * n; i += blockDim.x) {
    int kind, h, e;
    at(i, kind, h, e);
    const __half *src = W == 0 ? (kind ? a.v_new : a.k_new) + (vec0 + h) * kD + e
                               : (kind ? a.v_win : a.k_win) + vec0 * win_h + h * win_h + (int64_t)head * kD + e;
    copy16((kind ? a.stage_v : a.stage_k) + (vec0 + h) * kD + e, src);
  }
  if (W > 0) {
    __syncthreads();  // the ring slot has been read by every thread
    for (int i = threadIdx.x; i < 2 * n; i += blockDim.x) {
      int kind, h, e;
      at(i, kind, h, e);
      copy16((kind ? a.v_win : a.k_win) + vec0 * win_h + h * win_h + (int64_t)head * kD + e,
             (kind ? a.v_new : a.k_new) + (vec0 + h) * kD + e);
    }
  }
  if (threadIdx.x == 0) {
    a.stage_slots[b] = (int32_t)(page * P + comp % P);
    if (W > 0) a.win_head[b] = head + 1 == W ? 0 : head + 1;
    a.comp_lens[b] = comp + 1;
  }
}

}  // namespace

cudaError_t launch_window_roll(const RollArgs &a, cudaStream_t st) {
  if (a.B <= 0) return cudaSuccess;
  window_roll_kernel<<<a.B, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tq
