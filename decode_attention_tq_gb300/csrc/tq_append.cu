// tq_append.cu -- the append of one decode step in one launch (sm_103a).
//
// A cache is compressed pages plus an fp16 recent window of W tokens kept as
// a ring per sequence ("TurboQuant Family Design Study for CPU and Browser
// WASM KV Caches", 'Packed format and complete bit accounting': the last W
// tokens stay fp16; 'Append cost and memory-bandwidth tradeoffs': the append
// runs once per generated token; 'Paging, lifecycle, and cache identity':
// fixed pages filled in order).  Per sequence b:
//
//   * W > 0, window not full: the new token goes to ring slot win_lens[b];
//   * W > 0, window full: the oldest token (ring slot win_head[b]) is encoded
//     at compressed position comp_lens[b] and the new token takes its slot;
//   * W == 0: the new token itself is encoded.
//
// A block owns a group of sequences and does everything for them, in three
// phases separated by block barriers, so that one launch needs no
// cross-block ordering and each phase waits on at most one memory latency:
//   1. loads that depend on nothing: the sequences' counters, their new
//      tokens (into shared memory), both kinds' codebooks and sign flips (and
//      the QJL matrix, into registers);
//   2. the action of each sequence from its counters; side by side, the block
//      table entry of the compressed position it writes and the ring slot of
//      the token that leaves (copied into shared memory); the quantizer
//      tables and the QJL matrix's hi / lo cells are built meanwhile;
//   3. the new tokens into the rings (every leaving token has been read),
//      the counters, and the two encodes from shared memory at once: keys on
//      warps 0-3, values on warps 4-7.
#include "tq_encode_body.cuh"

namespace tq {

namespace {

constexpr int kChunks = kD / 8;    // 16-byte chunks per head vector
constexpr int kMaxSeqPerBlock = 32;
constexpr int kAppendThreads = 256;
// Vectors per kind a block holds: at most 64 sequence-heads, or one sequence
// of up to 128 heads (the largest head count tq_append_window accepts).
constexpr int kAppendMaxVecs = 128;

__device__ __forceinline__ void copy16(__half *dst, const __half *src) {
  *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
}

enum : int { kSkip = 0, kFill = 1, kEvict = 2 };

// Dynamic shared memory of a block: the QJL matrix cells (keys with a sketch)
// at its start, then the new tokens and, with a window, the tokens that leave
// it, each as [kind K, V][sequence][head][d] fp16.
__host__ __device__ constexpr size_t append_cells_bytes(bool kqjl) { return kqjl ? (size_t)kM * kD * 4 : 0; }
__host__ __device__ constexpr size_t append_smem_bytes(bool kqjl, int vecs, bool window) {
  return append_cells_bytes(kqjl) + (size_t)(window ? 2 : 1) * 2 * vecs * kD * sizeof(__half);
}

template <int KBITS, bool KQJL, bool KMIX, int VBITS>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(const RollArgs r, const EncodeArgs ka,
                                                                const EncodeArgs va, int seq_per_block) {
  __shared__ EncodeTables<KMIX> tk;
  __shared__ EncodeTables<false> tv;
  __shared__ int s_len[kMaxSeqPerBlock], s_head[kMaxSeqPerBlock], s_comp[kMaxSeqPerBlock], s_act[kMaxSeqPerBlock];
  __shared__ int32_t s_slot[kMaxSeqPerBlock];
  extern __shared__ __align__(16) uint8_t smem[];
  const int s0 = blockIdx.x * seq_per_block;
  const int ns = min(seq_per_block, r.B - s0);
  const int tid = threadIdx.x;
  const int W = r.W, H = r.H, P = r.P;
  const int nsh = ns * H;                 // vectors per kind
  const int nchunk = 2 * nsh * kChunks;   // 16-byte chunks of one token per (sequence, head, kind)
  const int64_t win_h = (int64_t)W * kD;  // head stride inside a sequence's window
  __half *s_new = reinterpret_cast<__half *>(smem + append_cells_bytes(KQJL));
  __half *s_old = s_new + 2 * nsh * kD;

  // Launched as a programmatic dependent of the kernel before it: nothing is
  // read before that kernel has completed (its launch and block scheduling
  // overlap that kernel's end).
  griddep_wait();
  // A kernel launched after this one as a programmatic dependent (the
  // attention's prep kernel) may start now: before it waits for this grid it
  // reads only the attention call's inputs (query, S, sign flips).
  griddep_launch_dependents();

  // 1. counters, new tokens, tables
  if (tid < ns) {
    const int b = s0 + tid;
    s_len[tid] = W > 0 ? r.win_lens[b] : 0;
    s_head[tid] = W > 0 ? r.win_head[b] : 0;
    s_comp[tid] = r.comp_lens[b];
  }
  for (int i = tid; i < nchunk; i += blockDim.x) {
    const int kind = i >= nsh * kChunks, c = kind ? i - nsh * kChunks : i;
    copy16(s_new + kind * nsh * kD + c * 8, (kind ? r.v_new : r.k_new) + (int64_t)s0 * H * kD + c * 8);
  }
  if (tid < kD) encode_tables_load<KBITS, KMIX>(tk, ka, tid);
  else if (tid < 2 * kD) encode_tables_load<VBITS, false>(tv, va, tid - kD);
  // the QJL matrix: loaded here (one memory latency beside the others),
  // converted into its hi / lo cells in phase 2, where that work overlaps the
  // block-table lookup (256 threads: one batch of kSCellBatch float4 each)
  static_assert(kAppendThreads * kSCellBatch * 4 == kM * kD, "one batch of S per thread");
  float4 sv[KQJL ? kSCellBatch : 1];
  if constexpr (KQJL) encode_s_batch_load(ka, tid, sv);
  __syncthreads();

  // 2. actions, pages and leaving tokens, quantizer tables
  if (tid < ns) {
    const int b = s0 + tid;
    const int len = s_len[tid], head = s_head[tid], comp = s_comp[tid];
    int act = kSkip, slot = -1;
    if (comp < 0 || (W > 0 && (len < 0 || len > W || head < 0 || head >= W))) {
      report(r.err_word, TQ_DEVERR_LENGTH);
    } else if (W > 0 && len < W) {
      act = kFill;
    } else {
      const int pi = comp / P;
      const int64_t page = pi < r.max_pages ? r.block_tables[(int64_t)b * r.max_pages + pi] : -1;
      if (page < 0 || page >= r.num_pages) {
        report(r.err_word, pi < r.max_pages ? TQ_DEVERR_PAGE_RANGE : TQ_DEVERR_LENGTH);
      } else {
        act = kEvict;
        slot = (int32_t)(page * P + comp % P);
      }
    }
    s_act[tid] = act;
    s_slot[tid] = slot;
  }
  if (W > 0) {
    // a full ring with valid counters gives up its oldest token (whether its
    // page turns out valid is decided above; an unused copy is harmless)
    for (int i = tid; i < nchunk; i += blockDim.x) {
      const int kind = i >= nsh * kChunks, c = kind ? i - nsh * kChunks : i;
      const int sl = c / (H * kChunks), h = (c / kChunks) % H, e = (c % kChunks) * 8;
      const int head = s_head[sl];
      if (s_len[sl] != W || head < 0 || head >= W || s_comp[sl] < 0) continue;
      const int64_t vec = (int64_t)(s0 + sl) * H + h;
      copy16(s_old + kind * nsh * kD + c * 8, (kind ? r.v_win : r.k_win) + vec * win_h + (int64_t)head * kD + e);
    }
  }
  encode_tables_build<KBITS, KMIX>(tk);
  encode_tables_build<VBITS, false>(tv);
  if constexpr (KQJL) encode_s_batch_store(tid, sv);
  __syncthreads();

  // 3. rings, counters, encodes (slot -1: nothing to encode for that sequence)
  if (W > 0) {
    for (int i = tid; i < nchunk; i += blockDim.x) {
      const int kind = i >= nsh * kChunks, c = kind ? i - nsh * kChunks : i;
      const int sl = c / (H * kChunks), h = (c / kChunks) % H, e = (c % kChunks) * 8;
      const int act = s_act[sl];
      if (act == kSkip) continue;
      const int ring = act == kFill ? s_len[sl] : s_head[sl];
      const int64_t vec = (int64_t)(s0 + sl) * H + h;
      copy16((kind ? r.v_win : r.k_win) + vec * win_h + (int64_t)ring * kD + e, s_new + kind * nsh * kD + c * 8);
    }
  }
  if (tid < ns) {
    const int b = s0 + tid, act = s_act[tid];
    if (act == kFill) {
      r.win_lens[b] = s_len[tid] + 1;
    } else if (act == kEvict) {
      if (W > 0) r.win_head[b] = s_head[tid] + 1 == W ? 0 : s_head[tid] + 1;
      r.comp_lens[b] = s_comp[tid] + 1;
    }
  }
  const int warp = tid >> 5;
  const __half *x = W > 0 ? s_old : s_new;  // the tokens to encode, [kind][sequence][head][d]
  if (warp < 4) {
    EncodeArgs kl = ka;
    kl.x = x;
    kl.n_tokens = ns;
    kl.slot_mapping = s_slot;
    if (KQJL && nsh <= 8)  // one octet of key vectors: the four warps share its QJL projection
      encode_loop<KBITS, KQJL, KMIX>(tk, kl, 0, 1, warp, 4);
    else
      encode_loop<KBITS, KQJL, KMIX>(tk, kl, warp, 4);
  } else {
    EncodeArgs vl = va;
    vl.x = x + nsh * kD;
    vl.n_tokens = ns;
    vl.slot_mapping = s_slot;
    encode_loop<VBITS, false, false>(tv, vl, warp - 4, 4);
  }
}

template <int KBITS, bool KQJL, bool KMIX, int VBITS>
cudaError_t launch_append_t(const RollArgs &r, const EncodeArgs &ka, const EncodeArgs &va, int sms, cudaStream_t st) {
  auto kern = append_kernel<KBITS, KQJL, KMIX, VBITS>;
  // Sequences per block: as few as keep the grid about one wave of the
  // machine (a block's phases wait on memory latency, not on throughput)
  int spb = (r.B + sms - 1) / (sms > 0 ? sms : 1);
  const int cap = r.H >= 64 ? 1 : (64 / r.H < kMaxSeqPerBlock ? 64 / r.H : kMaxSeqPerBlock);
  if (spb > cap) spb = cap;
  if (spb < 1) spb = 1;
  const int blocks = (r.B + spb - 1) / spb;
  const size_t smem = append_smem_bytes(KQJL, spb * r.H, r.W > 0);
  if (smem > append_smem_bytes(KQJL, kAppendMaxVecs, true)) return cudaErrorInvalidValue;
  static unsigned long long done = 0;
  const cudaError_t e = set_smem_once(kern, (int)append_smem_bytes(KQJL, kAppendMaxVecs, true), done);
  if (e != cudaSuccess) return e;
  const cudaError_t le = launch_maybe_dependent(kern, dim3(blocks), dim3(kAppendThreads), smem, st, true, r, ka, va, spb);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

template <int KBITS, bool KQJL, bool KMIX>
cudaError_t launch_append_v(const RollArgs &r, const EncodeArgs &ka, const EncodeArgs &va, int v_bits, int sms,
                            cudaStream_t st) {
  switch (v_bits) {
    case 2: return launch_append_t<KBITS, KQJL, KMIX, 2>(r, ka, va, sms, st);
    case 3: return launch_append_t<KBITS, KQJL, KMIX, 3>(r, ka, va, sms, st);
    case 4: return launch_append_t<KBITS, KQJL, KMIX, 4>(r, ka, va, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// k_bits: the key code width (the high channels' width for mixed keys)
cudaError_t launch_append(const RollArgs &r, const EncodeArgs &ka, const EncodeArgs &va, int k_bits, bool k_qjl,
                          bool k_mixed, int v_bits, int sms, cudaStream_t st) {
  if (r.B <= 0) return cudaSuccess;
  if (k_mixed) {
    switch (k_bits * 2 + (k_qjl ? 1 : 0)) {
      case 6: return launch_append_v<3, false, true>(r, ka, va, v_bits, sms, st);
      case 7: return launch_append_v<3, true, true>(r, ka, va, v_bits, sms, st);
      case 8: return launch_append_v<4, false, true>(r, ka, va, v_bits, sms, st);
      case 9: return launch_append_v<4, true, true>(r, ka, va, v_bits, sms, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (k_bits * 2 + (k_qjl ? 1 : 0)) {
    case 4: return launch_append_v<2, false, false>(r, ka, va, v_bits, sms, st);
    case 5: return launch_append_v<2, true, false>(r, ka, va, v_bits, sms, st);
    case 6: return launch_append_v<3, false, false>(r, ka, va, v_bits, sms, st);
    case 7: return launch_append_v<3, true, false>(r, ka, va, v_bits, sms, st);
    case 8: return launch_append_v<4, false, false>(r, ka, va, v_bits, sms, st);
    case 9: return launch_append_v<4, true, false>(r, ka, va, v_bits, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq
