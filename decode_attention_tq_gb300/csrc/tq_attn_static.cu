// tq_attn_static.cu -- tq_decode_attn_static: decode attention whose scratch
// is a fixed device array in the library image instead of a caller
// workspace, for callers that have no allocator to draw a workspace from
// (a plug-in handed bare tensor pointers by its host framework, or a loop
// that must not enter any allocator).  Nothing here allocates: the array is
// part of the loaded module, its address is looked up on every call, and the
// call then runs the ordinary tq_decode_attn on it.
#include "tq.h"
#include "tq_internal.cuh"

namespace {

constexpr size_t kScratchBytes = TQ_STATIC_SCRATCH_BYTES;

// The scratch: every call on a device uses this one buffer (calls must not
// overlap in time).  No word of it needs to start at zero.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch in the current context.  Looked up on every
// call rather than cached per device: a context that is torn down and created
// again (cudaDeviceReset) loads the module anew, possibly at another address.
// Once the module is loaded in the context this is a host-side table lookup
// that allocates nothing; the first call in a context may load the module,
// which is why that first call must come before any stream capture.
tq_status scratch_address(void **ptr) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return TQ_ERR_CUDA;
  *ptr = p;
  return TQ_OK;
}

}  // namespace

extern "C" tq_status tq_decode_attn_static(const tq_format *fmt, int batch, int num_q_heads, const void *q_f16,
                                           const void *page_pool, int64_t num_pages, const int32_t *block_tables,
                                           int max_pages, const int32_t *comp_lens, const void *k_win_f16,
                                           const void *v_win_f16, const int32_t *win_lens, int window,
                                           const uint8_t *k_signs, const uint8_t *v_signs, const float *k_codebook,
                                           const float *v_codebook, const float *S, float *out, int32_t *err_word,
                                           void *stream) {
  size_t need = 0;
  tq_status s = tq_decode_attn_workspace_size(fmt, batch, num_q_heads, max_pages, window, &need);
  if (s != TQ_OK) return s;
  if (need > kScratchBytes) return TQ_ERR_SCRATCH_LIMIT;
  void *scratch = nullptr;
  s = scratch_address(&scratch);
  if (s != TQ_OK) return s;
  return tq_decode_attn(fmt, batch, num_q_heads, q_f16, page_pool, num_pages, block_tables, max_pages, comp_lens,
                        k_win_f16, v_win_f16, win_lens, window, k_signs, v_signs, k_codebook, v_codebook, S, out,
                        scratch, kScratchBytes, err_word, stream);
}
