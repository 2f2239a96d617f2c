// tq_attn_kmix_qop.cu -- instantiations of the main decode-attention kernel for
// mixed-rate keys (3.5 and 2.5 bits) that take the prep kernel's ready-made
// query operands (short tile ranges per warp).
#include "tq_attn_main.cuh"

namespace tq {

cudaError_t attn_main_k34_qop(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                              int blocks, cudaStream_t st) {
  return attn_main_dispatch<34, true>(a, v_bits, qjl, nt, query_only, blocks_per_sm, blocks, st);
}

cudaError_t attn_main_k23_qop(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                              int blocks, cudaStream_t st) {
  return attn_main_dispatch<23, true>(a, v_bits, qjl, nt, query_only, blocks_per_sm, blocks, st);
}

}  // namespace tq
