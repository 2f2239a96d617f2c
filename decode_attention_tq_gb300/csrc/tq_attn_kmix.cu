// tq_attn_kmix.cu -- instantiations of the main decode-attention kernel for
// mixed-rate keys: 3.5 bits (4 + 3) and 2.5 bits (3 + 2) per channel.
#include "tq_attn_main.cuh"

namespace tq {

cudaError_t attn_main_k34(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                          int blocks, cudaStream_t st) {
  return attn_main_dispatch<34, false>(a, v_bits, qjl, nt, query_only, blocks_per_sm, blocks, st);
}

cudaError_t attn_main_k23(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                          int blocks, cudaStream_t st) {
  return attn_main_dispatch<23, false>(a, v_bits, qjl, nt, query_only, blocks_per_sm, blocks, st);
}
}  // namespace tq
