// tq_attn_kmix.cu -- instantiations of the main decode-attention kernel for
// mixed-rate keys: 3.5 bits (4 + 3) and 2.5 bits (3 + 2) per channel.
#include "tq_attn_main.cuh"

namespace tq {

// Builds with the shared-memory staging ring (TQ_TMA_STAGING=1, a measured
// alternative) carry uniform key widths only: there the mixed kinds report
// an invalid configuration.
#if TQ_TMA_STAGING
cudaError_t attn_main_k34(const AttnArgs &, int, bool, int, bool, int *, int, cudaStream_t) {
  return cudaErrorInvalidValue;
}
cudaError_t attn_main_k23(const AttnArgs &, int, bool, int, bool, int *, int, cudaStream_t) {
  return cudaErrorInvalidValue;
}
#else
cudaError_t attn_main_k34(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                          int blocks, cudaStream_t st) {
  return attn_main_dispatch<34>(a, v_bits, qjl, nt, query_only, blocks_per_sm, blocks, st);
}

cudaError_t attn_main_k23(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                          int blocks, cudaStream_t st) {
  return attn_main_dispatch<23>(a, v_bits, qjl, nt, query_only, blocks_per_sm, blocks, st);
}
#endif

}  // namespace tq
