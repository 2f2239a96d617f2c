// tq_encode.cu -- encode (append) kernels and the decode (reconstruct)
// kernel.  The encode body lives in tq_encode_body.cuh.  Decode: four
// consecutive lanes (a "quad") own one head vector, lane q holds coordinates
// 32q..32q+31; its codes are b 32-bit words of one stream for every b.
#include "tq_encode_body.cuh"

namespace tq {

// Blocks per SM of the encode without QJL: 3 for 4-bit and 4 for 2- and
// 3-bit codes (measured: 3-bit +6 %, 2-bit +2 % at 4 blocks).
template <int BITS>
constexpr int encode_min_blocks() {
  return BITS == 4 ? kEncodeBlocks4 : 4;
}

template <int BITS, bool MIXED = false>
__global__ void __launch_bounds__(256, encode_min_blocks<BITS>()) encode_kernel(const EncodeArgs a) {
  encode_body<BITS, MIXED>(a);
}

// Keys with QJL: the sketch products on tcgen05 (UmmaQjl in
// tq_encode_body.cuh).  One block of 16 warps per SM: S hi/lo (64 KB) and
// two residual buffers (2 x 64 KB) of 128-row operand tiles, 512 columns of
// tensor memory for three fp32 accumulators.
template <int BITS, bool MIXED>
__global__ void __launch_bounds__(kUmmaThreads, 1) encode_qjl_kernel(const EncodeArgs a) {
  __shared__ EncodeTables<MIXED> T;
  __shared__ uint64_t s_info[kUmmaInfoRing * kUmmaRows];
  __shared__ __align__(8) uint64_t s_mbar[2];  // done(0), done(1)
  __shared__ unsigned s_count[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  extern __shared__ __align__(16) uint4 s_Sq[];  // the operand tiles (1024-byte aligned below)
  const int tid = threadIdx.x;
  const uint32_t dyn = umma::smem_addr(s_Sq);
  const uint32_t pad = (1024u - (dyn & 1023u)) & 1023u;
  uint8_t *tiles = reinterpret_cast<uint8_t *>(s_Sq) + pad;
  if (tid < kD) encode_tables_load<BITS, MIXED>(T, a, tid);
  if (tid == 0) {
    umma::mbar_init(umma::smem_addr(&s_mbar[0]), 1);
    umma::mbar_init(umma::smem_addr(&s_mbar[1]), 1);
    s_count[0] = s_count[1] = 0u;
    s_abort = 0;
    umma::mbar_init_fence();
  }
  if (tid < 32) {
    umma::tmem_alloc(umma::smem_addr(&s_tmem), kUmmaTmemCols);
    umma::tmem_relinquish();
  }
  umma_s_tiles_load(a, tiles);
  umma::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  encode_tables_build<BITS, MIXED>(T);
  __syncthreads();
  UmmaQjl U;
  U.s_tiles = dyn + pad;
  U.r_tiles = dyn + pad + 2 * kUmmaTile;
  U.r_ptr = tiles + 2 * kUmmaTile;
  U.info = s_info;
  U.mbar = umma::smem_addr(&s_mbar[0]);
  U.count = s_count;
  U.tmem = s_tmem;
  U.abort = &s_abort;
  encode_loop<BITS, true, MIXED, true>(T, a, -1, 0, 0, 1, &U);
  umma::fence_before_sync();
  __syncthreads();
  if (tid < 32) {
    umma::fence_after_sync();
    umma::tmem_dealloc(U.tmem, kUmmaTmemCols);
  }
}

// Keys and values of the same tokens in one launch (same bits, keys without
// QJL): blockIdx.y selects the kind.
template <int BITS>
__global__ void __launch_bounds__(256, kEncodeBlocks4) encode_kv_kernel(const EncodeArgs ka, const EncodeArgs va) {
  if (blockIdx.y == 0)
    encode_body<BITS>(ka);
  else
    encode_body<BITS>(va);
}

// 16 codes of W bits from byte `off` of a key stream, as a 64-bit value.
__device__ __forceinline__ uint64_t codes16_bytes(const uint8_t *tok, int off, int W) {
  uint64_t v = 0;
  for (int k = 0; k < 2 * W; k++) v |= (uint64_t)tok[off + k] << (8 * k);
  return v;
}

// MIXED: keys at a fractional rate, BITS on the high channels (j mod 16 < 8)
// and BITS - 1 on the others (as in encode_body).
template <int BITS, bool QJL, bool MIXED = false>
__global__ void __launch_bounds__(256) decode_kernel(const DecodeArgs a) {
  extern __shared__ float s_S[];
  __shared__ float s_cent[MIXED ? 32 : 16];
  __shared__ uint32_t s_dsign[4];
  constexpr int L = 1 << BITS;
  const int tid = threadIdx.x;
  if (tid < L) s_cent[tid] = a.codebook[tid];
  if (MIXED && tid < L / 2) s_cent[16 + tid] = a.codebook[2 * L - 1 + tid];
  if (tid < 4) {
    uint32_t w = 0;
    for (int j = 0; j < 32; j++) w |= (a.signs[32 * tid + j] ? 1u : 0u) << j;
    s_dsign[tid] = w;
  }
  if constexpr (QJL) {
    // float4 loads, four per thread in flight; the swizzle keeps groups of
    // four columns together
    constexpr int N4 = kM * kD / 4;
    const float4 *S4 = reinterpret_cast<const float4 *>(a.S);
    for (int i0 = tid; i0 < N4; i0 += 4 * blockDim.x) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int i4 = i0 + u * blockDim.x;
        v[u] = i4 < N4 ? __ldg(S4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; u++) {
        const int i4 = i0 + u * blockDim.x;
        if (i4 < N4) *reinterpret_cast<float4 *>(&s_S[s_swz((4 * i4) / kD, (4 * i4) % kD)]) = v[u];
      }
    }
  }
  __syncthreads();

  const int lane = tid & 31, q = lane & 3, quad_in_warp = lane >> 2;
  const int warp = (blockIdx.x * blockDim.x + tid) >> 5;
  const int64_t nwarps = (int64_t)gridDim.x * blockDim.x / 32;
  const int64_t NH = a.n_tokens * a.H;
  const uint32_t dsign = s_dsign[q];
  const int64_t pool_slots = a.num_pages * (int64_t)a.P;
  // sqrt(d) * qjl_coef: the QJL term in u units (qjl_coef = sqrt(pi/2) / m
  // for the paper's Gaussian S)
  const float kq = 11.313708498984761f * a.qjl_coef;

  for (int64_t vb = (int64_t)warp * 8; vb < NH; vb += nwarps * 8) {
    const int64_t v = vb + quad_in_warp;
    const bool in_range = v < NH;
    const int64_t vv = in_range ? v : NH - 1;
    const int64_t n = vv / a.H;
    const int h = (int)(vv % a.H);
    const int64_t slot = a.slot_mapping[n];
    bool ok = in_range && slot >= 0;
    if (ok && slot >= pool_slots) {
      if (q == 0) report(a.err_word, TQ_DEVERR_SLOT_RANGE);
      ok = false;
    }
    const int64_t page = ok ? slot / a.P : 0;
    const int64_t off = ok ? slot % a.P : 0;
    const uint8_t *slab = a.pool + page * a.page_bytes + (int64_t)h * a.slab_bytes;

    const float nrm = reinterpret_cast<const float *>(slab + a.norm_off)[off];
    float y[32];
    if constexpr (MIXED) {
      // lane q's channels 32q..32q+31: codes 16q..16q+15 of the high stream
      // (channels with j mod 16 < 8) and of the low stream
      const uint8_t *tok = slab + a.codes_off + off * a.code_bytes;
      const uint64_t hv = codes16_bytes(tok, 2 * BITS * q, BITS);
      const uint64_t lv = codes16_bytes(tok, 8 * BITS + 2 * (BITS - 1) * q, BITS - 1);
#pragma unroll
      for (int j = 0; j < 32; j++) {
        const int k = 8 * (j >> 4) + (j & 7);
        y[j] = (j & 15) < 8 ? s_cent[(int)((hv >> (BITS * k)) & ((1u << BITS) - 1))]
                            : s_cent[16 + (int)((lv >> ((BITS - 1) * k)) & ((1u << (BITS - 1)) - 1))];
      }
    } else {
      uint32_t w[BITS];
      if (!a.grouped)
        load_codes<BITS>(slab + a.codes_off + off * a.code_bytes + q * 4 * BITS, w);
      else if constexpr (value_pairs_interleaved(BITS))
        load_codes_pair<BITS>(slab + a.codes_off, off, q, w);
      else
        load_codes_grouped<BITS>(slab + a.codes_off, off, q, w);
      int idx[32];
      unpack_codes<BITS>(w, idx);
#pragma unroll
      for (int j = 0; j < 32; j++) y[j] = s_cent[idx[j]];
    }
    if constexpr (QJL) {
      const float gamma = reinterpret_cast<const float *>(slab + a.gamma_off)[off];
      const uint4 sb = *reinterpret_cast<const uint4 *>(slab + a.signs_off + off * (kM / 8));
      const uint32_t sw[4] = {sb.x, sb.y, sb.z, sb.w};
      float acc[32];
#pragma unroll
      for (int j = 0; j < 32; j++) acc[j] = 0.f;
#pragma unroll
      for (int wi = 0; wi < 4; wi++) {
        const uint32_t bits = sw[wi];
#pragma unroll 4
        for (int bit = 0; bit < 32; bit++) {
        const int l = 32 * wi + bit;
        const float sg = ((bits >> bit) & 1u) ? 1.f : -1.f;
#pragma unroll
        for (int i4 = 0; i4 < 8; i4++) {
          const float4 sv = *reinterpret_cast<const float4 *>(&s_S[l * kD + 32 * q + ((4 * i4) ^ (8 * q))]);
          acc[4 * i4 + 0] = fmaf(sg, sv.x, acc[4 * i4 + 0]);
          acc[4 * i4 + 1] = fmaf(sg, sv.y, acc[4 * i4 + 1]);
          acc[4 * i4 + 2] = fmaf(sg, sv.z, acc[4 * i4 + 2]);
          acc[4 * i4 + 3] = fmaf(sg, sv.w, acc[4 * i4 + 3]);
        }
        }
      }
      const float gk = gamma * kq;
#pragma unroll
      for (int j = 0; j < 32; j++) y[j] = fmaf(gk, acc[j], y[j]);
    }
    fwht_quad(y, q);
    const float sc = ok ? nrm * (1.0f / (float)kD) : 0.f;
    float o[32];
#pragma unroll
    for (int j = 0; j < 32; j++) o[j] = (((dsign >> j) & 1u) ? -y[j] : y[j]) * sc;
    if (in_range) {
      float4 *dst = reinterpret_cast<float4 *>(a.out + vv * kD + 32 * q);
#pragma unroll
      for (int k = 0; k < 8; k++) dst[k] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
    }
  }
}

// ----------------------------------------------------------------- launch --
template <int BITS, bool QJL, bool MIXED = false>
static cudaError_t launch_encode_t(const EncodeArgs &a, int sms, cudaStream_t st) {
  const int64_t vectors = a.n_tokens * a.H;
  if constexpr (QJL) {
    static unsigned long long done = 0;
    cudaError_t e = set_smem_once(encode_qjl_kernel<BITS, MIXED>, (int)kUmmaDynSmem, done);
    if (e != cudaSuccess) return e;
    int64_t blocks = (vectors + kUmmaRows - 1) / kUmmaRows;  // one batch of 128 vectors per block and pass
    if (blocks > sms) blocks = sms;
    if (blocks < 1) blocks = 1;
    encode_qjl_kernel<BITS, MIXED><<<(unsigned)blocks, kUmmaThreads, kUmmaDynSmem, st>>>(a);
  } else {
    int64_t blocks = (vectors + 63) / 64;
    const int64_t cap = (int64_t)sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    encode_kernel<BITS, MIXED><<<(unsigned)blocks, 256, 0, st>>>(a);
  }
  return cudaGetLastError();
}

template <int BITS, bool QJL, bool MIXED = false>
static cudaError_t launch_decode_t(const DecodeArgs &a, int sms, cudaStream_t st) {
  const size_t smem = QJL ? (size_t)kM * kD * sizeof(float) : 0;
  if (QJL) {
    static unsigned long long done = 0;
    cudaError_t e = set_smem_once(decode_kernel<BITS, QJL, MIXED>, (int)smem, done);
    if (e != cudaSuccess) return e;
  }
  const int64_t quads = a.n_tokens * a.H;
  int64_t blocks = (quads + 63) / 64;
  const int64_t cap = (int64_t)sms * (QJL ? 3 : 8);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  decode_kernel<BITS, QJL, MIXED><<<(unsigned)blocks, 256, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_encode_kv(const EncodeArgs &ka, const EncodeArgs &va, int bits, int sms, cudaStream_t st) {
  const int64_t quads = ka.n_tokens * ka.H;
  int64_t blocks = (quads + 63) / 64;
  const int64_t cap = (int64_t)sms * 4;  // two kinds share the machine
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid((unsigned)blocks, 2);
  switch (bits) {
    case 2: encode_kv_kernel<2><<<grid, 256, 0, st>>>(ka, va); break;
    case 3: encode_kv_kernel<3><<<grid, 256, 0, st>>>(ka, va); break;
    case 4: encode_kv_kernel<4><<<grid, 256, 0, st>>>(ka, va); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// bits: the code width; for mixed-rate keys the high channels' width
cudaError_t launch_encode(const EncodeArgs &a, int bits, bool qjl, bool mixed, int sms, cudaStream_t st) {
  if (mixed) {
    switch (bits * 2 + (qjl ? 1 : 0)) {
      case 6: return launch_encode_t<3, false, true>(a, sms, st);
      case 7: return launch_encode_t<3, true, true>(a, sms, st);
      case 8: return launch_encode_t<4, false, true>(a, sms, st);
      case 9: return launch_encode_t<4, true, true>(a, sms, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (bits * 2 + (qjl ? 1 : 0)) {
    case 4: return launch_encode_t<2, false>(a, sms, st);
    case 5: return launch_encode_t<2, true>(a, sms, st);
    case 6: return launch_encode_t<3, false>(a, sms, st);
    case 7: return launch_encode_t<3, true>(a, sms, st);
    case 8: return launch_encode_t<4, false>(a, sms, st);
    case 9: return launch_encode_t<4, true>(a, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(const DecodeArgs &a, int bits, bool qjl, bool mixed, int sms, cudaStream_t st) {
  if (mixed) {
    switch (bits * 2 + (qjl ? 1 : 0)) {
      case 6: return launch_decode_t<3, false, true>(a, sms, st);
      case 7: return launch_decode_t<3, true, true>(a, sms, st);
      case 8: return launch_decode_t<4, false, true>(a, sms, st);
      case 9: return launch_decode_t<4, true, true>(a, sms, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (bits * 2 + (qjl ? 1 : 0)) {
    case 4: return launch_decode_t<2, false>(a, sms, st);
    case 5: return launch_decode_t<2, true>(a, sms, st);
    case 6: return launch_decode_t<3, false>(a, sms, st);
    case 7: return launch_decode_t<3, true>(a, sms, st);
    case 8: return launch_decode_t<4, false>(a, sms, st);
    case 9: return launch_decode_t<4, true>(a, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq
