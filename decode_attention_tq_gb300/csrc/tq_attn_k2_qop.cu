// tq_attn_k2_qop.cu -- instantiations of the main decode-attention kernel for
// 2-bit keys that take the prep kernel's ready-made query operands (short
// tile ranges per warp); a translation unit of its own to compile in parallel.
#include "tq_attn_main.cuh"

namespace tq {

cudaError_t attn_main_k2_qop(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                             int blocks, cudaStream_t st) {
  return attn_main_dispatch<2, true>(a, v_bits, qjl, nt, query_only, blocks_per_sm, blocks, st);
}

}  // namespace tq
