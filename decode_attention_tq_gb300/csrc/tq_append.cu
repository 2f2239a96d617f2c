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
// A block owns a group of sequences and does everything for them: it reads
// their counters, copies the tokens that leave into a staging buffer, writes
// the new tokens into the rings, encodes the staged keys, then the staged
// values (each kind with its own format), and last writes the counters.  No
// other block touches these sequences, so one launch needs no cross-block
// ordering.
#include "tq_encode_body.cuh"

namespace tq {

namespace {

constexpr int kChunks = kD / 8;    // 16-byte chunks per head vector
constexpr int kMaxSeqPerBlock = 32;

__device__ __forceinline__ void copy16(__half *dst, const __half *src) {
  *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
}

enum : int { kSkip = 0, kFill = 1, kEvict = 2 };

template <int KBITS, bool KQJL, bool KMIX, int VBITS>
__global__ void __launch_bounds__(256) append_kernel(const RollArgs r, const EncodeArgs ka, const EncodeArgs va,
                                                     int seq_per_block) {
  __shared__ int s_len[kMaxSeqPerBlock], s_head[kMaxSeqPerBlock], s_comp[kMaxSeqPerBlock], s_act[kMaxSeqPerBlock];
  const int s0 = blockIdx.x * seq_per_block;
  const int ns = min(seq_per_block, r.B - s0);
  const int tid = threadIdx.x;
  const int W = r.W, H = r.H, P = r.P;

  // 1. what each sequence does, from its counters
  if (tid < ns) {
    const int b = s0 + tid;
    const int len = W > 0 ? r.win_lens[b] : 0, head = W > 0 ? r.win_head[b] : 0, comp = r.comp_lens[b];
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
    s_len[tid] = len;
    s_head[tid] = head;
    s_comp[tid] = comp;
    s_act[tid] = act;
    r.stage_slots[b] = slot;
  }
  __syncthreads();

  // 2. stage the tokens that leave (or, without a window, the new ones); 3.
  // after every thread has read the ring slots, write the new tokens
  const int per_seq = 2 * H * kChunks;
  const int64_t win_h = (int64_t)W * kD;  // head stride inside a sequence's window
  for (int i = tid; i < ns * per_seq; i += blockDim.x) {
    const int sl = i / per_seq, c = i % per_seq, kind = c >= H * kChunks, cc = kind ? c - H * kChunks : c;
    const int h = cc / kChunks, e = (cc % kChunks) * 8;
    if (s_act[sl] != kEvict) continue;
    const int64_t vec = (int64_t)(s0 + sl) * H + h;
    const __half *src = W == 0 ? (kind ? r.v_new : r.k_new) + vec * kD + e
                               : (kind ? r.v_win : r.k_win) + vec * win_h + (int64_t)s_head[sl] * kD + e;
    copy16((kind ? r.stage_v : r.stage_k) + vec * kD + e, src);
  }
  __syncthreads();
  if (W > 0) {
    for (int i = tid; i < ns * per_seq; i += blockDim.x) {
      const int sl = i / per_seq, c = i % per_seq, kind = c >= H * kChunks, cc = kind ? c - H * kChunks : c;
      const int h = cc / kChunks, e = (cc % kChunks) * 8;
      const int act = s_act[sl];
      if (act == kSkip) continue;
      const int ring = act == kFill ? s_len[sl] : s_head[sl];
      const int64_t vec = (int64_t)(s0 + sl) * H + h;
      copy16((kind ? r.v_win : r.k_win) + vec * win_h + (int64_t)ring * kD + e, (kind ? r.v_new : r.k_new) + vec * kD + e);
    }
  }

  // 4. encode this block's staged keys, then values (slot -1: nothing staged)
  const int64_t warp = tid >> 5, nwarps = blockDim.x >> 5;
  EncodeArgs kl = ka;
  kl.x = r.stage_k + (int64_t)s0 * H * kD;
  kl.n_tokens = ns;
  kl.slot_mapping = r.stage_slots + s0;
  encode_body<KBITS, KQJL, KMIX>(kl, warp, nwarps);
  __syncthreads();  // the two bodies may share their tables
  EncodeArgs vl = va;
  vl.x = r.stage_v + (int64_t)s0 * H * kD;
  vl.n_tokens = ns;
  vl.slot_mapping = r.stage_slots + s0;
  encode_body<VBITS, false, false>(vl, warp, nwarps);

  // 5. the counters, after every thread of the block has used them
  __syncthreads();
  if (tid < ns) {
    const int b = s0 + tid, act = s_act[tid];
    if (act == kFill) {
      r.win_lens[b] = s_len[tid] + 1;
    } else if (act == kEvict) {
      if (W > 0) r.win_head[b] = s_head[tid] + 1 == W ? 0 : s_head[tid] + 1;
      r.comp_lens[b] = s_comp[tid] + 1;
    }
  }
}

template <int KBITS, bool KQJL, bool KMIX, int VBITS>
cudaError_t launch_append_t(const RollArgs &r, const EncodeArgs &ka, const EncodeArgs &va, int sms, cudaStream_t st) {
  auto kern = append_kernel<KBITS, KQJL, KMIX, VBITS>;
  const size_t smem = KQJL ? (size_t)kM * kD * sizeof(float) : 0;  // S cells of the key sketch
  if (KQJL) {
    static unsigned long long done = 0;
    const cudaError_t e = set_smem_once(kern, (int)smem, done);
    if (e != cudaSuccess) return e;
  }
  // Sequences per block: as few as keep the grid about one wave of the
  // machine (each block runs its copies and both encodes one after another)
  int spb = (r.B + sms - 1) / (sms > 0 ? sms : 1);
  const int cap = r.H >= 64 ? 1 : (64 / r.H < kMaxSeqPerBlock ? 64 / r.H : kMaxSeqPerBlock);
  if (spb > cap) spb = cap;
  if (spb < 1) spb = 1;
  const int blocks = (r.B + spb - 1) / spb;
  kern<<<blocks, 256, smem, st>>>(r, ka, va, spb);
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
