// tq_internal.cuh -- argument blocks and launcher declarations shared by the
// libtq translation units.
#pragma once

#include <utility>

#include <cuda_runtime.h>

#include "tq_device.cuh"

namespace tq {

struct EncodeArgs {
  const __half *x;
  int64_t n_tokens;
  int H, P;
  const int32_t *slot_mapping;
  uint8_t *pool;
  int64_t num_pages, page_bytes, slab_bytes;
  int64_t norm_off, codes_off, gamma_off, signs_off;
  int code_bytes;
  bool grouped;  // value-code stream: 16-token groups, chunk-major (value_chunk_offset),
                 // offset pairs interleaved for 2- and 4-bit codes (value_pairs_interleaved)
  bool norm_correct;  // store n / ||y_hat|| (no QJL)
  const uint8_t *signs;
  const float *codebook;
  const float *S;
  int32_t *err_word;
};

// Per-step append (tq_append_window): see tq_append.cu.
struct RollArgs {
  const __half *k_new, *v_new;  // [B][H][d]
  __half *k_win, *v_win;        // [B][H][W][d] (W > 0)
  int B, H, W, P, max_pages;
  int64_t num_pages;
  int32_t *win_lens, *win_head, *comp_lens;  // [B], updated in place
  const int32_t *block_tables;               // [B][max_pages]
  int32_t *err_word;
};

struct DecodeArgs {
  const uint8_t *pool;
  int64_t n_tokens;
  int H, P;
  const int32_t *slot_mapping;
  int64_t num_pages, page_bytes, slab_bytes;
  int64_t norm_off, codes_off, gamma_off, signs_off;
  int code_bytes;
  bool grouped;
  const uint8_t *signs;
  const float *codebook;
  const float *S;
  float qjl_coef;  // factor of gamma * S^T (2z - 1) in y_hat
  float *out;
  int32_t *err_word;
};

// The value-code section keeps each token's LSB-first bitstream in chunks of
// 16 coordinates (2*bits bytes) and stores a group of 16 tokens chunk by
// chunk; inside a chunk row the tokens of the group sit in the order
// 0,1,8,9, 2,3,10,11, 4,5,12,13, 6,7,14,15, so that one thread of the
// attention kernel finds chunk r of the tokens it multiplies (2t, 2t+1,
// 2t+8, 2t+9) in one contiguous run.  Offset of chunk r of the token at page
// offset `off`, from the start of the section:
__host__ __device__ __forceinline__ int64_t value_chunk_offset(int64_t off, int r, int bits) {
  const int i = (int)(off & 15);
  const int slot = 4 * ((i & 7) >> 1) + 2 * (i >> 3) + (i & 1);
  return (off >> 4) * (2 * kD * bits) + (int64_t)r * (16 * 2 * bits) + slot * (2 * bits);  // group = 16 * kD * bits / 8 bytes
}

// 2- and 4-bit value codes interleave the tokens of each page-offset pair
// (2p, 2p+1) inside their two chunk slots: the pair's 4*bits bytes are two
// LSB-first streams of bits-wide fields, the even coordinates c of the chunk
// first, then the odd ones, field 2 (c div 2) + (offset mod 2) holding the
// code of coordinate c of one of the two tokens.  The attention kernel then
// reads, for a pair of tokens, one register of both tokens' codes per two
// coordinates as stored.
__host__ __device__ constexpr bool value_pairs_interleaved(int bits) { return bits == 2 || bits == 4; }

// Query operands of the split-KV main kernel, written by the prep kernel:
// per query row four parts of 64 fp16x2 words, the rotated query scaled by
// 2^q_exp[0] split into fp16 hi (part 0) and lo (part 1) and the QJL
// projection scaled by 2^q_exp[1] likewise (parts 2, 3).  Word 16t + w of a
// part holds coordinates of slice t (32t .. 32t + 31) as a main-kernel lane
// of that slice takes them as B-operand registers (w = 0 .. 15): the query
// words pair slice coordinates (2w, 2w + 1), the QJL words pair slice values
// (w, w + 16), i.e. fp16 index 2 (i mod 16) + (i div 16) of the slice holds
// QJL value i.
__host__ __device__ __forceinline__ int qop_qjl_half(int i) { return 2 * (i & 15) + (i >> 4); }

// Workspace header written by the prep kernel and read by the others.
struct AttnHeader {
  int64_t total_tiles;  // sum over (b, h) of ceil(comp_len / 16)
  int64_t active_warps; // warps that own a non-empty tile range
};

struct AttnArgs {
  // cache
  const uint8_t *pool;
  int64_t num_pages, page_bytes, slab_bytes;
  int64_t k_norm_o, k_gamma_o, k_codes_o, k_signs_o, v_norm_o, v_codes_o;  // section offsets in a slab
  int k_code_bytes, v_code_bytes;
  int B, Hq, H, G, P, max_pages, window;
  const int32_t *block_tables;
  const int32_t *comp_lens;
  const __half *q;
  const __half *k_win;
  const __half *v_win;
  const int32_t *win_lens;
  const uint8_t *k_signs, *v_signs;
  const float *k_cb, *v_cb;
  const float *S;
  float qjl_coef;  // factor of gamma * S^T (2z - 1) in y_hat
  float *out;
  int32_t *err_word;
  // workspace sections
  AttnHeader *hdr;
  int64_t *pre;      // [B + 1] prefix sums of tiles per sequence
  int32_t *clen;     // [B] clamped compressed lengths
  int32_t *wlen;     // [B] clamped window lengths
  float *q_rot;      // [B][Hq][d]
  int32_t *q_exp;    // [B][Hq][2] power-of-two exponents for the fp16 operands
  uint32_t *q_op;    // [B][Hq][4][64] the main kernel's fp16x2 query operands (qop_word)
  float2 *q_cst;     // [B][Hq] score constants (key part, QJL part) in the log2 domain
  float *seg_ml;     // [slots][G][2]  (max in log2 units, sum)
  float *seg_acc;    // [slots][G][d]  rotated-domain value accumulator
  float *win_ml;     // [B][Hq][window chunks][2]
  float *win_acc;    // [B][Hq][window chunks][d]  raw-domain window accumulators
  float *merge_part; // [B][Hq][merge_slices][kMergePartStride] slice results of the wide merge
                     // (accumulator [d], then max, sum; records 16-byte aligned)
  int32_t *merge_cnt;  // [B][Hq] slices of a row done (zeroed by the prep kernel)
  int nw_launch;     // warps launched for the main kernel
  int min_tiles;     // fewest tiles a warp is given
  int merge_slices;  // blocks per row of the wide merge (1: no slice results)
  bool pdl;          // host: launch main and merge as programmatic dependents
  bool raw;          // KIVI cache: no query rotation, the accumulators are raw-domain
  bool qop_keys;     // host: launch the main kernel that loads its key-score query operands from q_op
  bool win_apart;    // window partials by their own kernel after the main kernel (else in the prep kernel)
};

// KIVI-style control arm (tq_kivi.cu): encode of keys (per-channel groups of
// one page) or values (per token), and reconstruction for tests.  Section
// offsets are those of tq_kivi_layout for the kind.
struct KiviEncodeArgs {
  const __half *x;             // [N][H][d]
  int64_t n_tokens;
  int H, P;
  const int32_t *page_ids;     // keys: [ceil(N / P)]
  const int32_t *slot_mapping; // values: [N]
  uint8_t *pool;
  int64_t num_pages, page_bytes, slab_bytes;
  int64_t params_off, codes_off;
  int32_t *err_word;
};
struct KiviDecodeArgs {
  const uint8_t *pool;
  int64_t n_tokens;
  int H, P, kind;
  const int32_t *slot_mapping;
  int64_t num_pages, page_bytes, slab_bytes;
  int64_t params_off, codes_off;
  float *out;
  int32_t *err_word;
};
cudaError_t launch_kivi_encode(const KiviEncodeArgs &a, int kind, int bits, cudaStream_t st);
cudaError_t launch_kivi_decode(const KiviDecodeArgs &a, int bits, cudaStream_t st);
// KIVI main attention kernel (AttnArgs with raw = true; k_norm_o / v_norm_o
// hold the K and V (scale, zero) sections)
cudaError_t kivi_main(const AttnArgs &a, int k_bits, int v_bits, int nt, bool query_only, int *blocks_per_sm,
                      int blocks, cudaStream_t st);
__host__ __device__ constexpr int kivi_threads(int nt) { return nt == 1 ? 512 : 256; }

cudaError_t launch_encode(const EncodeArgs &a, int bits, bool qjl, bool mixed, int sms, cudaStream_t st);
// One launch: window roll, encode of the staged keys and values, counters.
// k_bits is the key code width (the high channels' width for mixed keys).
cudaError_t launch_append(const RollArgs &r, const EncodeArgs &ka, const EncodeArgs &va, int k_bits, bool k_qjl,
                          bool k_mixed, int v_bits, int sms, cudaStream_t st);

// Launch `kern` on `st`, as a programmatic dependent of the previous kernel on
// the stream when `dependent` (the kernel must call griddep_wait() before it
// reads that kernel's outputs).
template <typename... P, typename... A>
cudaError_t launch_maybe_dependent(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                   bool dependent, A &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}
cudaError_t launch_encode_kv(const EncodeArgs &ka, const EncodeArgs &va, int bits, int sms, cudaStream_t st);
cudaError_t launch_decode(const DecodeArgs &a, int bits, bool qjl, bool mixed, int sms, cudaStream_t st);

// Decode attention pieces (tq_attn_aux.cu and tq_attn_k*.cu).
constexpr int kWinChunk = 32;  // window tokens per window partial
cudaError_t launch_attn_prep(const AttnArgs &a, bool qjl, cudaStream_t st);
cudaError_t launch_attn_merge(const AttnArgs &a, cudaStream_t st);
// Window partials by their own launch (a.win_apart): after the main kernel,
// as its programmatic dependent; no-op without a window.
cudaError_t launch_attn_window(const AttnArgs &a, cudaStream_t st);
// Merge geometry: rows whose (sequence, kv head) average at most
// kWarpMergeMaxPartials partials are merged by one warp each, the others by
// blocks of kMergeWarps warps, kSlicePartials partials per block (slices).
constexpr int kWarpMergeMaxPartials = 24, kMergeWarps = 16, kWideChunk = 10;
constexpr int kSlicePartials = kMergeWarps * kWideChunk, kMaxMergeSlices = 32;
constexpr int kMergePartStride = kD + 4;  // floats per slice result: a multiple of 4 (float4 accesses)
inline bool merge_by_warps(int64_t nw_launch, int64_t units) { return nw_launch <= kWarpMergeMaxPartials * units; }
inline int merge_slices(int64_t nw_launch, int64_t units) {
  if (merge_by_warps(nw_launch, units)) return 1;
  const int64_t avg = (nw_launch + units - 1) / units;
  const int64_t s = (avg + kSlicePartials - 1) / kSlicePartials;
  return (int)(s < 1 ? 1 : (s > kMaxMergeSlices ? kMaxMergeSlices : s));
}
// Main split-KV kernel: returns its per-SM occupancy through *blocks_per_sm
// when `query_only`, else launches `blocks` CTAs.
cudaError_t attn_main_k2(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                         int blocks, cudaStream_t st);
cudaError_t attn_main_k3(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                         int blocks, cudaStream_t st);
cudaError_t attn_main_k4(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                         int blocks, cudaStream_t st);
cudaError_t attn_main_k34(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                         int blocks, cudaStream_t st);
cudaError_t attn_main_k23(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                         int blocks, cudaStream_t st);
// The same with the prep kernel's ready-made key-score query operands.
cudaError_t attn_main_k2_qop(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                             int blocks, cudaStream_t st);
cudaError_t attn_main_k3_qop(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                             int blocks, cudaStream_t st);
cudaError_t attn_main_k4_qop(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                             int blocks, cudaStream_t st);
cudaError_t attn_main_k34_qop(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                              int blocks, cudaStream_t st);
cudaError_t attn_main_k23_qop(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *blocks_per_sm,
                              int blocks, cudaStream_t st);

// Set a kernel's dynamic shared-memory limit once per device (never inside a
// stream capture after the first call on that device).
template <typename K>
cudaError_t set_smem_once(K kernel, int bytes, unsigned long long &done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (__atomic_load_n(&done_mask, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) __atomic_fetch_or(&done_mask, bit, __ATOMIC_ACQ_REL);
  return e;
}

// Threads per CTA of the main attention kernel (one CTA per SM), by the
// number of 8-column n-tiles (NT = 1 for up to 4 query heads per kv head, 2
// for up to 8) and QJL: the register file is shared out as 65536 / threads,
// and the NT = 2 accumulators (and QJL operands) need more per thread.
// 384 threads for NT = 1 measured within 1.5 % of 512 at the Llama-3-8B and
// long-context decode shapes, with a step no faster.
__host__ __device__ constexpr int attn_threads(int nt, bool qjl) {
  return nt == 1 ? 512 : (qjl ? 256 : 384);
}
__host__ __device__ constexpr int attn_warps(int nt, bool qjl) { return attn_threads(nt, qjl) / 32; }

}  // namespace tq
