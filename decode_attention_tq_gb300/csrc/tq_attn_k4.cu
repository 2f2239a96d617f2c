// tq_attn_k4.cu -- instantiations of the main decode-attention kernel for
// 4-bit keys (one translation unit per key width so they compile in parallel).
#include "tq_attn_main.cuh"

namespace tq {

cudaError_t attn_main_k4(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                         int blocks, cudaStream_t st) {
  return attn_main_dispatch<4, false>(a, v_bits, qjl, nt, query_only, blocks_per_sm, blocks, st);
}

}  // namespace tq
