// tq_encode.cu -- encode (append) kernel and the decode (reconstruct) kernel.
//
// Work split: four consecutive lanes (a "quad") own one head vector; lane q
// holds coordinates 32q..32q+31, so the Walsh-Hadamard butterflies with
// h = 1..16 run in registers and h = 32, 64 are two shuffle stages.  With 32
// coordinates per lane the packed codes of a lane are exactly b 32-bit words
// for every b, so packing is thread-local and each lane writes its own slice.
#include "tq_internal.cuh"

namespace tq {

// QJL matrix S [m][d] staged in shared memory with columns XOR-swizzled by
// lane slice so the four lanes of a quad read different banks.
__device__ __forceinline__ int s_swz(int l, int j) { return l * kD + (j ^ ((j >> 5) << 3)); }

template <int BITS>
__device__ __forceinline__ void pack_codes(const int (&idx)[32], uint32_t (&w)[BITS]) {
#pragma unroll
  for (int k = 0; k < BITS; k++) w[k] = 0u;
#pragma unroll
  for (int j = 0; j < 32; j++) {
    const int bit = j * BITS, wi = bit >> 5, sh = bit & 31;
    w[wi] |= (uint32_t)idx[j] << sh;
    if (sh + BITS > 32) w[wi + 1] |= (uint32_t)idx[j] >> (32 - sh);
  }
}

template <int BITS>
__device__ __forceinline__ void unpack_codes(const uint32_t (&w)[BITS], int (&idx)[32]) {
  constexpr uint32_t mask = (1u << BITS) - 1u;
#pragma unroll
  for (int j = 0; j < 32; j++) {
    const int bit = j * BITS, wi = bit >> 5, sh = bit & 31;
    uint32_t v = w[wi] >> sh;
    if (sh + BITS > 32) v |= w[wi + 1] << (32 - sh);
    idx[j] = (int)(v & mask);
  }
}

template <int BITS>
__device__ __forceinline__ void store_codes(uint8_t *p, const uint32_t (&w)[BITS]) {
  if constexpr (BITS == 4) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  } else if constexpr (BITS == 2) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
  } else {
#pragma unroll
    for (int k = 0; k < BITS; k++) reinterpret_cast<uint32_t *>(p)[k] = w[k];
  }
}

// The same 4*BITS bytes (chunks 2q and 2q+1 of a token) in a grouped
// value-code section (value_chunk_offset).
template <int BITS>
__device__ __forceinline__ void store_codes_grouped(uint8_t *sec, int64_t off, int q, const uint32_t (&w)[BITS]) {
  uint8_t *c0 = sec + value_chunk_offset(off, 2 * q, BITS);
  uint8_t *c1 = sec + value_chunk_offset(off, 2 * q + 1, BITS);
  if constexpr (BITS == 4) {
    *reinterpret_cast<uint2 *>(c0) = make_uint2(w[0], w[1]);
    *reinterpret_cast<uint2 *>(c1) = make_uint2(w[2], w[3]);
  } else if constexpr (BITS == 2) {
    *reinterpret_cast<uint32_t *>(c0) = w[0];
    *reinterpret_cast<uint32_t *>(c1) = w[1];
  } else {  // 6-byte chunks on 2-byte boundaries
    uint16_t *h0 = reinterpret_cast<uint16_t *>(c0), *h1 = reinterpret_cast<uint16_t *>(c1);
    h0[0] = (uint16_t)w[0];
    h0[1] = (uint16_t)(w[0] >> 16);
    h0[2] = (uint16_t)w[1];
    h1[0] = (uint16_t)(w[1] >> 16);
    h1[1] = (uint16_t)w[2];
    h1[2] = (uint16_t)(w[2] >> 16);
  }
}

template <int BITS>
__device__ __forceinline__ void load_codes_grouped(const uint8_t *sec, int64_t off, int q, uint32_t (&w)[BITS]) {
  const uint8_t *c0 = sec + value_chunk_offset(off, 2 * q, BITS);
  const uint8_t *c1 = sec + value_chunk_offset(off, 2 * q + 1, BITS);
  if constexpr (BITS == 4) {
    const uint2 x = *reinterpret_cast<const uint2 *>(c0), y = *reinterpret_cast<const uint2 *>(c1);
    w[0] = x.x; w[1] = x.y; w[2] = y.x; w[3] = y.y;
  } else if constexpr (BITS == 2) {
    w[0] = *reinterpret_cast<const uint32_t *>(c0);
    w[1] = *reinterpret_cast<const uint32_t *>(c1);
  } else {
    const uint16_t *h0 = reinterpret_cast<const uint16_t *>(c0), *h1 = reinterpret_cast<const uint16_t *>(c1);
    w[0] = (uint32_t)h0[0] | ((uint32_t)h0[1] << 16);
    w[1] = (uint32_t)h0[2] | ((uint32_t)h1[0] << 16);
    w[2] = (uint32_t)h1[1] | ((uint32_t)h1[2] << 16);
  }
}

template <int BITS>
__device__ __forceinline__ void load_codes(const uint8_t *p, uint32_t (&w)[BITS]) {
  if constexpr (BITS == 4) {
    uint4 v = *reinterpret_cast<const uint4 *>(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (BITS == 2) {
    uint2 v = *reinterpret_cast<const uint2 *>(p);
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int k = 0; k < BITS; k++) w[k] = reinterpret_cast<const uint32_t *>(p)[k];
  }
}

// 32 fp16 -> fp32 of this lane's slice.
__device__ __forceinline__ void load_slice_f16(const __half *src, float (&x)[32]) {
  const uint4 *p = reinterpret_cast<const uint4 *>(src);
#pragma unroll
  for (int k = 0; k < 4; k++) {
    uint4 v = p[k];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
      __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
      float2 f = __half22float2(h);
      x[8 * k + 2 * i] = f.x;
      x[8 * k + 2 * i + 1] = f.y;
    }
  }
}

// Unnormalized WHT of a 128-vector spread over a quad (lane slice q).
__device__ __forceinline__ void fwht_quad(float (&x)[32], int q) {
  fwht_local<32>(x);
  fwht_xlane<32>(x, 1, (q & 1) != 0);
  fwht_xlane<32>(x, 2, (q & 2) != 0);
}

template <int BITS, bool QJL>
__global__ void __launch_bounds__(256) encode_kernel(const EncodeArgs a) {
  extern __shared__ float s_S[];  // [m][d] swizzled, QJL only
  __shared__ float s_cent[16];
  __shared__ float s_mid[16];
  __shared__ uint32_t s_dsign[4];
  constexpr int L = 1 << BITS;
  const int tid = threadIdx.x;
  if (tid < L) s_cent[tid] = a.codebook[tid];
  if (tid < L - 1) s_mid[tid] = a.codebook[L + tid];
  if (tid < 4) {
    uint32_t w = 0;
    for (int j = 0; j < 32; j++) w |= (a.signs[32 * tid + j] ? 1u : 0u) << j;
    s_dsign[tid] = w;
  }
  if constexpr (QJL) {
    for (int i = tid; i < kM * kD; i += blockDim.x) s_S[s_swz(i / kD, i % kD)] = a.S[i];
  }
  __syncthreads();

  const int lane = tid & 31, q = lane & 3, quad_in_warp = lane >> 2;
  const int warp = (blockIdx.x * blockDim.x + tid) >> 5;
  const int64_t nwarps = (int64_t)gridDim.x * blockDim.x / 32;
  const int64_t NH = a.n_tokens * a.H;
  const uint32_t dsign = s_dsign[q];
  const int64_t pool_slots = a.num_pages * (int64_t)a.P;

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

    float x[32];
    load_slice_f16(a.x + vv * kD + 32 * q, x);
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 32; j++) ss = fmaf(x[j], x[j], ss);
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    const float nrm = sqrtf(ss);
    const bool zero = !(nrm > 0.f);

#pragma unroll
    for (int j = 0; j < 32; j++) x[j] = ((dsign >> j) & 1u) ? -x[j] : x[j];
    fwht_quad(x, q);
    const float inv = zero ? 0.f : 1.0f / nrm;

    int idx[32];
#pragma unroll
    for (int j = 0; j < 32; j++) {
      const float u = x[j] * inv;
      int k = 0;
#pragma unroll
      for (int s = L / 2; s >= 1; s >>= 1)
        if (u >= s_mid[k + s - 1]) k += s;
      idx[j] = zero ? 0 : k;
      x[j] = u - s_cent[idx[j]];  // residual in u units (QJL only)
    }
    uint32_t w[BITS];
    pack_codes<BITS>(idx, w);

    const int64_t page = ok ? slot / a.P : 0;
    const int64_t off = ok ? slot % a.P : 0;
    uint8_t *slab = a.pool + page * a.page_bytes + (int64_t)h * a.slab_bytes;
    if (ok) {
      if (a.grouped)
        store_codes_grouped<BITS>(slab + a.codes_off, off, q, w);
      else
        store_codes<BITS>(slab + a.codes_off + off * a.code_bytes + q * 4 * BITS, w);
      if (q == 0) reinterpret_cast<float *>(slab + a.norm_off)[off] = nrm;
    }

    if constexpr (QJL) {
      // gamma = ||u - c|| / sqrt(d); the sign of (S e)_l does not depend on the
      // positive factor 1/sqrt(d), so the projection uses u - c directly.
      float g2 = 0.f;
#pragma unroll
      for (int j = 0; j < 32; j++) g2 = fmaf(x[j], x[j], g2);
      g2 += __shfl_xor_sync(0xffffffffu, g2, 1);
      g2 += __shfl_xor_sync(0xffffffffu, g2, 2);
      const float gamma = zero ? 0.f : sqrtf(g2) * 0.08838834764831845f;
      uint32_t word = 0u;
#pragma unroll 1
      for (int c = 0; c < 4; c++) {
        // rows l = 32k + 8c + i, partial index p = 8k + i
        float part[32];
#pragma unroll
        for (int p = 0; p < 32; p++) {
          const int l = 32 * (p >> 3) + 8 * c + (p & 7);
          float acc = 0.f;
#pragma unroll
          for (int i4 = 0; i4 < 8; i4++) {
            const float4 sv = *reinterpret_cast<const float4 *>(&s_S[l * kD + 32 * q + ((4 * i4) ^ (8 * q))]);
            acc = fmaf(sv.x, x[4 * i4 + 0], acc);
            acc = fmaf(sv.y, x[4 * i4 + 1], acc);
            acc = fmaf(sv.z, x[4 * i4 + 2], acc);
            acc = fmaf(sv.w, x[4 * i4 + 3], acc);
          }
          part[p] = acc;
        }
        // reduce-scatter over the quad: stage 1 keeps k in {b, b+2}, stage 2 keeps k = q
        const int bq = q & 1, aq = q >> 1;
        float r1[16];
#pragma unroll
        for (int i = 0; i < 8; i++) {
          // keep groups k = bq and k = bq + 2; send k = 1-bq and k = 3-bq
          const float keep0 = bq ? part[8 + i] : part[i];
          const float keep1 = bq ? part[24 + i] : part[16 + i];
          const float send0 = bq ? part[i] : part[8 + i];
          const float send1 = bq ? part[16 + i] : part[24 + i];
          r1[i] = keep0 + __shfl_xor_sync(0xffffffffu, send0, 1);
          r1[8 + i] = keep1 + __shfl_xor_sync(0xffffffffu, send1, 1);
        }
        uint32_t byte = 0u;
#pragma unroll
        for (int i = 0; i < 8; i++) {
          const float keep = aq ? r1[8 + i] : r1[i];
          const float send = aq ? r1[i] : r1[8 + i];
          const float tot = keep + __shfl_xor_sync(0xffffffffu, send, 2);
          byte |= (tot >= 0.f ? 1u : 0u) << i;
        }
        word |= byte << (8 * c);
      }
      if (zero) word = 0u;
      if (ok) {
        reinterpret_cast<uint32_t *>(slab + a.signs_off + off * (kM / 8))[q] = word;
        if (q == 0) reinterpret_cast<float *>(slab + a.gamma_off)[off] = gamma;
      }
    }
  }
}

template <int BITS, bool QJL>
__global__ void __launch_bounds__(256) decode_kernel(const DecodeArgs a) {
  extern __shared__ float s_S[];
  __shared__ float s_cent[16];
  __shared__ uint32_t s_dsign[4];
  constexpr int L = 1 << BITS;
  const int tid = threadIdx.x;
  if (tid < L) s_cent[tid] = a.codebook[tid];
  if (tid < 4) {
    uint32_t w = 0;
    for (int j = 0; j < 32; j++) w |= (a.signs[32 * tid + j] ? 1u : 0u) << j;
    s_dsign[tid] = w;
  }
  if constexpr (QJL) {
    for (int i = tid; i < kM * kD; i += blockDim.x) s_S[s_swz(i / kD, i % kD)] = a.S[i];
  }
  __syncthreads();

  const int lane = tid & 31, q = lane & 3, quad_in_warp = lane >> 2;
  const int warp = (blockIdx.x * blockDim.x + tid) >> 5;
  const int64_t nwarps = (int64_t)gridDim.x * blockDim.x / 32;
  const int64_t NH = a.n_tokens * a.H;
  const uint32_t dsign = s_dsign[q];
  const int64_t pool_slots = a.num_pages * (int64_t)a.P;
  // sqrt(d) * sqrt(pi/2) / m: the QJL term in u units
  const float kq = 11.313708498984761f * 1.2533141373155003f / (float)kM;

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

    uint32_t w[BITS];
    if (a.grouped)
      load_codes_grouped<BITS>(slab + a.codes_off, off, q, w);
    else
      load_codes<BITS>(slab + a.codes_off + off * a.code_bytes + q * 4 * BITS, w);
    const float nrm = reinterpret_cast<const float *>(slab + a.norm_off)[off];
    int idx[32];
    unpack_codes<BITS>(w, idx);
    float y[32];
#pragma unroll
    for (int j = 0; j < 32; j++) y[j] = s_cent[idx[j]];
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
template <int BITS, bool QJL>
static cudaError_t launch_encode_t(const EncodeArgs &a, int sms, cudaStream_t st) {
  const size_t smem = QJL ? (size_t)kM * kD * sizeof(float) : 0;
  if (QJL) {
    static unsigned long long done = 0;
    cudaError_t e = set_smem_once(encode_kernel<BITS, QJL>, (int)smem, done);
    if (e != cudaSuccess) return e;
  }
  const int64_t quads = a.n_tokens * a.H;
  int64_t blocks = (quads + 63) / 64;
  const int64_t cap = (int64_t)sms * (QJL ? 3 : 8);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  encode_kernel<BITS, QJL><<<(unsigned)blocks, 256, smem, st>>>(a);
  return cudaGetLastError();
}

template <int BITS, bool QJL>
static cudaError_t launch_decode_t(const DecodeArgs &a, int sms, cudaStream_t st) {
  const size_t smem = QJL ? (size_t)kM * kD * sizeof(float) : 0;
  if (QJL) {
    static unsigned long long done = 0;
    cudaError_t e = set_smem_once(decode_kernel<BITS, QJL>, (int)smem, done);
    if (e != cudaSuccess) return e;
  }
  const int64_t quads = a.n_tokens * a.H;
  int64_t blocks = (quads + 63) / 64;
  const int64_t cap = (int64_t)sms * (QJL ? 3 : 8);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  decode_kernel<BITS, QJL><<<(unsigned)blocks, 256, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_encode(const EncodeArgs &a, int bits, bool qjl, int sms, cudaStream_t st) {
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

cudaError_t launch_decode(const DecodeArgs &a, int bits, bool qjl, int sms, cudaStream_t st) {
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
