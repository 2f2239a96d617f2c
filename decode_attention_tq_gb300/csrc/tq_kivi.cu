// tq_kivi.cu -- the KIVI-style control arm: asymmetric (scale, zero) integer
// quantization of keys per channel over a page and of values per token, and
// split-KV decode attention on such a cache ("TurboQuant Family Design Study
// for CPU and Browser WASM KV Caches", 'Candidate key and value algorithms',
// item 1: the control baseline arm).  No rotation: the codes quantize the
// raw-domain vectors, so decode attention needs no centroid tables: integer
// codes become exact fp16 tensor-core operands with one lop3 per code pair.
//
//   scores:  l_i = (sum_j q_j s_j c_ij + sum_j q_j z_j) / sqrt(d), s, z the
//            channel scales and zeros of the token's page: the B operand is
//            q * s per page (hi/lo fp16 split), A the codes of 16 tokens;
//   values:  sum_i p_i v_hat_i = sum_i (p_i s_i) c_i + (sum_i p_i z_i) 1, s_i,
//            z_i the token's scale and zero: A the codes (coordinate pairs x
//            token slots), B the weights p_i s_i / nu in fp16.
// The work split, online softmax, partial layout and merge are those of the
// TurboQuant attention (tq_attn_main.cuh, tq_attn_aux.cu in raw mode).
#include "tq_attn_main.cuh"

namespace tq {

// ---------------------------------------------------------------- quantizer --
// The stored (scale, zero) of a group with fp32 minimum mn and maximum mx.
__device__ __forceinline__ __half2 kivi_params(float mn, float mx, int top) {
  const float s32 = __fdiv_rn(__fsub_rn(mx, mn), (float)top);
  __half sh = __float2half_rn(s32);
  if (__half2float(sh) > 65504.f) sh = __float2half_rn(65504.f);  // an infinite range
  return __halves2half2(sh, __float2half_rn(__fadd_rn(mn, 0.0f)));  // a zero minimum as +0
}

// The code of x, decided in fp32 with the stored zero z and scale s.
__device__ __forceinline__ int kivi_code(float x, float z, float s, int top) {
  if (!(s > 0.f)) return 0;
  const float r = floorf(__fadd_rn(__fdiv_rn(__fsub_rn(x, z), s), 0.5f));
  return r >= 0.f ? (r > (float)top ? top : (int)r) : 0;
}

__device__ __forceinline__ void half4_to_float(uint2 raw, float (&f)[4]) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
  f[0] = a.x;
  f[1] = a.y;
  f[2] = b.x;
  f[3] = b.y;
}

// One warp per (page group, head): lane l owns channels 4l .. 4l+3.
template <int BITS>
__global__ void __launch_bounds__(128) kivi_encode_keys_kernel(const KiviEncodeArgs a) {
  constexpr int top = (1 << BITS) - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n_groups = (a.n_tokens + a.P - 1) / a.P;
  const int64_t unit = (int64_t)blockIdx.x * 4 + warp;
  if (unit >= n_groups * a.H) return;
  const int64_t g = unit / a.H;
  const int h = (int)(unit % a.H);
  const int n = (int)min((int64_t)a.P, a.n_tokens - g * a.P);
  const int32_t page = a.page_ids[g];
  if (page < 0 || (int64_t)page >= a.num_pages) {
    if (lane == 0) report(a.err_word, TQ_DEVERR_PAGE_RANGE);
    return;
  }
  uint8_t *slab = a.pool + (int64_t)page * a.page_bytes + (int64_t)h * a.slab_bytes;
  const int64_t tstride = (int64_t)a.H * kD;  // halves between consecutive tokens
  const __half *x0 = a.x + (g * a.P * a.H + h) * kD + 4 * lane;
  float mn[4], mx[4];
#pragma unroll
  for (int c = 0; c < 4; c++) {
    mn[c] = INFINITY;
    mx[c] = -INFINITY;
  }
  for (int i = 0; i < n; i++) {
    float f[4];
    half4_to_float(*reinterpret_cast<const uint2 *>(x0 + i * tstride), f);
#pragma unroll
    for (int c = 0; c < 4; c++) {
      if (f[c] < mn[c]) mn[c] = f[c];
      if (f[c] > mx[c]) mx[c] = f[c];
    }
  }
  __half2 prm[4];
  float sf[4], zf[4];
#pragma unroll
  for (int c = 0; c < 4; c++) {
    prm[c] = kivi_params(mn[c], mx[c], top);
    sf[c] = __low2float(prm[c]);
    zf[c] = __high2float(prm[c]);
  }
  *reinterpret_cast<uint4 *>(slab + a.params_off + 16 * lane) =
      make_uint4(*reinterpret_cast<uint32_t *>(&prm[0]), *reinterpret_cast<uint32_t *>(&prm[1]),
                 *reinterpret_cast<uint32_t *>(&prm[2]), *reinterpret_cast<uint32_t *>(&prm[3]));
  uint8_t *codes = slab + a.codes_off;
  for (int i = 0; i < n; i++) {
    float f[4];
    half4_to_float(*reinterpret_cast<const uint2 *>(x0 + i * tstride), f);
    uint32_t w = 0;
#pragma unroll
    for (int c = 0; c < 4; c++) w |= (uint32_t)kivi_code(f[c], zf[c], sf[c], top) << (BITS * c);
    if constexpr (BITS == 4)
      reinterpret_cast<uint16_t *>(codes + (int64_t)i * (kD / 2))[lane] = (uint16_t)w;
    else
      codes[(int64_t)i * (kD / 4) + lane] = (uint8_t)w;
  }
}

// One warp per (token, head): lane l owns channels 4l .. 4l+3.
template <int BITS>
__global__ void __launch_bounds__(128) kivi_encode_values_kernel(const KiviEncodeArgs a) {
  constexpr int top = (1 << BITS) - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t unit = (int64_t)blockIdx.x * 4 + warp;
  if (unit >= a.n_tokens * a.H) return;
  const int64_t n = unit / a.H;
  const int h = (int)(unit % a.H);
  const int32_t slot = a.slot_mapping[n];
  if (slot < 0) return;
  if ((int64_t)slot >= a.num_pages * a.P) {
    if (lane == 0) report(a.err_word, TQ_DEVERR_SLOT_RANGE);
    return;
  }
  const int64_t page = slot / a.P, off = slot % a.P;
  uint8_t *slab = a.pool + page * a.page_bytes + (int64_t)h * a.slab_bytes;
  float f[4];
  half4_to_float(*reinterpret_cast<const uint2 *>(a.x + (n * a.H + h) * kD + 4 * lane), f);
  float mn = fminf(fminf(f[0], f[1]), fminf(f[2], f[3]));
  float mx = fmaxf(fmaxf(f[0], f[1]), fmaxf(f[2], f[3]));
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, m));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
  }
  const __half2 prm = kivi_params(mn, mx, top);
  const float sf = __low2float(prm), zf = __high2float(prm);
  uint32_t w = 0;
#pragma unroll
  for (int c = 0; c < 4; c++) w |= (uint32_t)kivi_code(f[c], zf, sf, top) << (BITS * c);
  // chunk lane/4 (coordinates 16 (lane/4) ..) of the grouped value section
  uint8_t *chunk = slab + a.codes_off + value_chunk_offset(off, lane >> 2, BITS);
  if constexpr (BITS == 4)
    reinterpret_cast<uint16_t *>(chunk)[lane & 3] = (uint16_t)w;
  else
    chunk[lane & 3] = (uint8_t)w;
  if (lane == 0) *reinterpret_cast<__half2 *>(slab + a.params_off + 4 * off) = prm;
}

// Reconstruction z + s * code of one (slot, head) per warp (tests).
template <int BITS>
__global__ void __launch_bounds__(128) kivi_decode_kernel(const KiviDecodeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t unit = (int64_t)blockIdx.x * 4 + warp;
  if (unit >= a.n_tokens * a.H) return;
  const int64_t n = unit / a.H;
  const int h = (int)(unit % a.H);
  float *o = a.out + (n * a.H + h) * kD + 4 * lane;
  const int32_t slot = a.slot_mapping[n];
  if (slot < 0 || (int64_t)slot >= a.num_pages * a.P) {
    if (slot >= 0 && lane == 0) report(a.err_word, TQ_DEVERR_SLOT_RANGE);
    *reinterpret_cast<float4 *>(o) = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int64_t page = slot / a.P, off = slot % a.P;
  const uint8_t *slab = a.pool + page * a.page_bytes + (int64_t)h * a.slab_bytes;
  uint32_t w;
  if (a.kind == TQ_KIND_K)
    w = BITS == 4 ? reinterpret_cast<const uint16_t *>(slab + a.codes_off + off * (kD / 2))[lane]
                  : slab[a.codes_off + off * (kD / 4) + lane];
  else {
    const uint8_t *chunk = slab + a.codes_off + value_chunk_offset(off, lane >> 2, BITS);
    w = BITS == 4 ? reinterpret_cast<const uint16_t *>(chunk)[lane & 3] : chunk[lane & 3];
  }
  float r[4];
#pragma unroll
  for (int c = 0; c < 4; c++) {
    float s, z;
    if (a.kind == TQ_KIND_K) {
      const __half2 p = reinterpret_cast<const __half2 *>(slab + a.params_off)[4 * lane + c];
      s = __low2float(p);
      z = __high2float(p);
    } else {
      const __half2 p = reinterpret_cast<const __half2 *>(slab + a.params_off)[off];
      s = __low2float(p);
      z = __high2float(p);
    }
    r[c] = fmaf(s, (float)((w >> (BITS * c)) & ((1u << BITS) - 1)), z);
  }
  *reinterpret_cast<float4 *>(o) = make_float4(r[0], r[1], r[2], r[3]);
}

cudaError_t launch_kivi_encode(const KiviEncodeArgs &a, int kind, int bits, cudaStream_t st) {
  const int64_t units = kind == TQ_KIND_K ? ((a.n_tokens + a.P - 1) / a.P) * a.H : a.n_tokens * a.H;
  const dim3 grid((unsigned)((units + 3) / 4));
  if (kind == TQ_KIND_K) {
    if (bits == 4) kivi_encode_keys_kernel<4><<<grid, 128, 0, st>>>(a);
    else kivi_encode_keys_kernel<2><<<grid, 128, 0, st>>>(a);
  } else {
    if (bits == 4) kivi_encode_values_kernel<4><<<grid, 128, 0, st>>>(a);
    else kivi_encode_values_kernel<2><<<grid, 128, 0, st>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_kivi_decode(const KiviDecodeArgs &a, int bits, cudaStream_t st) {
  const dim3 grid((unsigned)((a.n_tokens * a.H + 3) / 4));
  if (bits == 4) kivi_decode_kernel<4><<<grid, 128, 0, st>>>(a);
  else kivi_decode_kernel<2><<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------- attention --
// Integer codes as exact fp16 tensor-core operands: fp16 1024 + n has the
// integer n in its low mantissa bits, so a lop3 of the code word with a mask
// and 0x6400 gives (1024 + n) or (1024 + 2^k n) in each half, and one
// subtraction of 1024 leaves n * 2^k exactly.  The pairs that come out of one
// 32-bit word are codes (i, i + 4) of 4-bit codes or (i, i + 8) of 2-bit
// codes; the power-of-two factor 2^k of a pair is divided out of its B
// operand (keys) or its output row (values).
__device__ __forceinline__ uint32_t magic_pair(uint32_t w, uint32_t mask) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(mask), "r"(0x64006400u));  // (w & mask) | magic
  const __half2 h = __hsub2(*reinterpret_cast<__half2 *>(&r), __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
  return *reinterpret_cast<const uint32_t *>(&h);
}

// Code pair q (0 .. 4 for 4-bit words, 0 .. 8 for 2-bit) of a word: the
// integer values times kivi_pair_scale<BITS>(q).
template <int BITS>
__device__ __forceinline__ uint32_t kivi_pair(uint32_t w, int q) {
  if constexpr (BITS == 4) {  // pairs (n_i, n_i+4), i = kivi_pair_code<4>(q)
    const uint32_t x = (q & 2) ? (w >> 8) : w;
    return magic_pair(x, (q & 1) ? 0x00F000F0u : 0x000F000Fu);
  } else {
    const uint32_t x = (q & 4) ? (w >> 8) : w;
    return magic_pair(x, 0x00030003u << (2 * (q & 3)));
  }
}
// First code index of pair q of a word (the second is + 4 or + 8) and the
// power of two the pair's values carry.
template <int BITS>
__host__ __device__ constexpr int kivi_pair_code(int q) {
  return BITS == 4 ? ((q & 2) ? 2 : 0) + (q & 1) : ((q & 4) ? 4 : 0) + (q & 3);
}
template <int BITS>
__host__ __device__ constexpr float kivi_pair_scale(int q) {
  return BITS == 4 ? ((q & 1) ? 16.f : 1.f) : (float)(1 << (2 * (q & 3)));
}

template <int KB>
struct KiviKeyRegs {
  uint32_t k0[KB], k1[KB];  // key code slice t (channels 32t .. 32t+31) of tokens r, r+8
  bool ok0, ok1, page0;     // live tokens r / r+8; the tile opens a page (B rebuilt)
  const uint8_t *slab;      // the tile's page slab
};
struct KiviValRegs {
  uint32_t v[8];            // chunk r of tokens 2t, 2t+1, 2t+8, 2t+9 (4-bit: two words each; 2-bit: one)
  __half2 p0, p1;           // (scale, zero) of tokens r, r+8
};


// Per warp: the raw query of its G heads, fp32 [8][kD], scaled by
// 2^(eq - 14): with |q| 2^eq < 2^13 and a stored scale s < 2^16 the B
// operand q s 2^(eq - 14) stays below 2^15.
template <int KB, int VB, int NT>
__global__ void __launch_bounds__(kivi_threads(NT), 1) kivi_main_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) float kq_smem[];
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31, r = lane >> 2, t = lane & 3, wib = threadIdx.x >> 5;
  float *qs = kq_smem + wib * (8 * kD);  // this warp's scaled queries [g][j]
  const int64_t wg = (int64_t)blockIdx.x * (kivi_threads(NT) / 32) + wib;
  const int64_t T = a.hdr->total_tiles;
  const int64_t NW = a.hdr->active_warps;
  if (wg >= NW) return;
  const int64_t ts = T * wg / NW, te = T * (wg + 1) / NW;
  if (ts >= te) return;
  const int H = a.H, G = a.G, Hq = a.Hq;
  const int tpp = a.P >> 4;
  const uint32_t selW_lo = r < 4 ? 0x4410u : 0x1044u, selW_hi = r < 4 ? 0x4432u : 0x3244u;
  constexpr int KW = KB;  // code words per token slice (32 channels)
  constexpr int VW = VB == 4 ? 2 : 1;  // code words per token chunk (16 coordinates)

  int b = 0;
  {
    int lo = 0, hi = a.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (H * a.pre[mid] <= ts) lo = mid; else hi = mid;
    }
    b = lo;
  }
  int tb = (int)(a.pre[b + 1] - a.pre[b]);
  int h = (int)((ts - H * a.pre[b]) / tb);
  int j = (int)((ts - H * a.pre[b]) - (int64_t)h * tb);
  int64_t pos = ts;

  while (pos < te) {
    const int seg_tiles = (int)min(te - pos, (int64_t)(tb - j));
    // ---- segment: scaled queries of the G heads into shared memory
    __syncwarp();
    for (int e = lane; e < 8 * kD; e += 32) {
      const int g = e / kD;
      float v = 0.f;
      if (g < G) {
        const int64_t row = (int64_t)b * Hq + (int64_t)h * G + g;
        v = ldexpf(a.q_rot[row * kD + (e % kD)], a.q_exp[row * 2] - 14);
      }
      qs[e] = v;
    }
    __syncwarp();
    float cL[NT];  // logit factor of this lane's head 4nt + t: log2(e)/sqrt(d) 2^(14 - eq)
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      const int g = 4 * nt + t;
      const int64_t row = (int64_t)b * Hq + (int64_t)h * G + (g < G ? g : 0);
      cL[nt] = ldexpf(kLog2e * 0.08838834764831845f, 14 - a.q_exp[row * 2]);
    }

    float mu[NT], lsum[NT], zsum[NT];
    float acc[4][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      mu[nt] = -INFINITY;
      lsum[nt] = 0.f;
      zsum[nt] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 4; mt++)
#pragma unroll
        for (int i = 0; i < 4; i++) acc[mt][nt][i] = 0.f;
    }
    float nu = 0.f, inv_nu = 0.f;
    uint32_t qb[NT][8][2];  // B operand of the page: q s 2^(eq-14) / pair factor, hi or lo part
    float bias[NT];         // sum_j q_j z_j 2^(eq-14) of this lane's head

    TileCursor cur;
    cur.pool = a.pool;
    cur.btrow = a.block_tables + (int64_t)b * a.max_pages;
    cur.num_pages = a.num_pages;
    cur.page_bytes = a.page_bytes;
    cur.slab_off = (int64_t)h * a.slab_bytes;
    cur.P = a.P;
    cur.pidx = j / tpp;
    cur.o0 = (j - cur.pidx * tpp) * 16;
    cur.tok0 = j * 16;
    cur.clen = a.clen[b];
    cur.last_page = (j + seg_tiles - 1) / tpp;
    cur.begin(a.err_word, lane == 0, (uint32_t)a.slab_bytes);
    bool first_tile = true;

    // B operand and bias of the page a tile opens: lane (r, t) builds column
    // r (head 4nt + r/2, hi part for even r, lo part for odd r) for its
    // channels 32t .. 32t+31 in the order of its code pairs
    auto build_page = [&](const uint8_t *slab) {
      const __half2 *prm = reinterpret_cast<const __half2 *>(slab + a.k_norm_o) + 32 * t;
#pragma unroll
      for (int nt = 0; nt < NT; nt++) {
        const int gcol = 4 * nt + (r >> 1);
        const float *qrow = qs + (gcol < 8 ? gcol : 0) * kD + 32 * t;
        const bool lo_part = (r & 1) != 0;
        float bz = 0.f;
#pragma unroll
        for (int w = 0; w < KW; w++) {
          // word w of the slice: 32/KW channels; its pairs q give k-steps
#pragma unroll
          for (int q = 0; q < 8 / KW * 2; q += 2) {
            // k-step kk = (8/KW) w + q/2: A registers pairs q (slots 2t, 2t+1), q+1 (slots 2t+8, 2t+9)
            const int kk = (8 / KW) * w + q / 2;
            uint32_t bw[2];
#pragma unroll
            for (int e = 0; e < 2; e++) {
              const int qq = q + e;
              const int c0 = w * (32 / KW) + kivi_pair_code<KB>(qq), c1 = c0 + (KB == 4 ? 4 : 8);
              const float2 p0 = __half22float2(prm[c0]), p1 = __half22float2(prm[c1]);
              const float inv = 1.0f / kivi_pair_scale<KB>(qq);
              const float y0 = qrow[c0] * p0.x * inv, y1 = qrow[c1] * p1.x * inv;
              bz = fmaf(qrow[c0], p0.y, fmaf(qrow[c1], p1.y, bz));
              __half h0, l0, h1, l1;
              split_half(y0, h0, l0);
              split_half(y1, h1, l1);
              bw[e] = lo_part ? pack_half2_raw(l0, l1) : pack_half2_raw(h0, h1);
            }
            qb[nt][kk][0] = bw[0];
            qb[nt][kk][1] = bw[1];
          }
        }
        // bias of head 4nt + r/2 over channels 32t.. -> summed over t, then
        // this lane's own head 4nt + t taken from lane 8t (r = 2t)
        bz += __shfl_xor_sync(0xffffffffu, bz, 1);
        bz += __shfl_xor_sync(0xffffffffu, bz, 2);
        bias[nt] = __shfl_sync(0xffffffffu, bz, 8 * t);
      }
    };

    auto load_keys = [&](KiviKeyRegs<KB> &R) {
      const int live = cur.live();
      R.ok0 = r < live;
      R.ok1 = r + 8 < live;
      R.page0 = first_tile || cur.o0 == 0;
      R.slab = cur.slab;
      const uint8_t *kc = cur.slab + a.k_codes_o + t * 4 * KB;
      ldg_words<KB>(kc + (cur.o0 + r) * (16 * KB), R.k0);
      ldg_words<KB>(kc + (cur.o0 + r + 8) * (16 * KB), R.k1);
    };
    auto load_vals = [&](KiviValRegs &V) {
      const __half2 *vp = reinterpret_cast<const __half2 *>(cur.slab + a.v_norm_o) + cur.o0;
      V.p0 = vp[r];
      V.p1 = vp[r + 8];
      const uint8_t *vc = cur.slab + a.v_codes_o + (int64_t)cur.o0 * (16 * VB) + r * (16 * 2 * VB) + t * (4 * 2 * VB);
      if constexpr (VB == 4) {
        ldna32B(vc, V.v);
      } else {
        const uint4 x = ldna(reinterpret_cast<const uint4 *>(vc));
        V.v[0] = x.x; V.v[1] = x.y; V.v[2] = x.z; V.v[3] = x.w;
#pragma unroll
        for (int i = 4; i < 8; i++) V.v[i] = 0u;
      }
    };

    auto process = [&](const KiviKeyRegs<KB> &R, const KiviValRegs &V) {
      if (!__any_sync(0xffffffffu, R.ok0)) return;  // a page outside the pool
      if (R.page0) build_page(R.slab);
      // ---- scores: rows r / r+8 = tokens r / r+8
      float sc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int i = 0; i < 4; i++) sc[nt][i] = 0.f;
#pragma unroll
      for (int w = 0; w < KW; w++)
#pragma unroll
        for (int q = 0; q < 8 / KW * 2; q += 2) {
          const int kk = (8 / KW) * w + q / 2;
          const uint32_t A0 = kivi_pair<KB>(R.k0[w], q), A2 = kivi_pair<KB>(R.k0[w], q + 1);
          const uint32_t A1 = kivi_pair<KB>(R.k1[w], q), A3 = kivi_pair<KB>(R.k1[w], q + 1);
#pragma unroll
          for (int nt = 0; nt < NT; nt++) mma_16816(sc[nt], A0, A1, A2, A3, qb[nt][kk][0], qb[nt][kk][1]);
        }
      // ---- online softmax (log2 domain), lazy running (mu, nu) as in the
      // TurboQuant kernel; nu bounds the value scales s_i
      const float vs0 = R.ok0 ? __low2float(V.p0) : 0.f, vs1 = R.ok1 ? __low2float(V.p1) : 0.f;
      const float vz0 = __high2float(V.p0), vz1 = __high2float(V.p1);
      float lg0[NT], lg1[NT];
      bool big = vs0 > kLazyNu * nu || vs1 > kLazyNu * nu;
#pragma unroll
      for (int nt = 0; nt < NT; nt++) {
        lg0[nt] = R.ok0 ? (sc[nt][0] + sc[nt][1] + bias[nt]) * cL[nt] : -INFINITY;
        lg1[nt] = R.ok1 ? (sc[nt][2] + sc[nt][3] + bias[nt]) * cL[nt] : -INFINITY;
        big |= fmaxf(lg0[nt], lg1[nt]) > mu[nt] + kLazyLog2;
      }
      if (__any_sync(0xffffffffu, big)) {
        const float tnu = warp_max_xor(fmaxf(vs0, vs1), 4 | 8 | 16);
        const float nu_new = fmaxf(nu, tnu);
        const float nu_ratio = nu_new > 0.f ? nu / nu_new : 1.f;
        inv_nu = nu_new > 0.f ? kWeightScale / nu_new : 0.f;
        nu = nu_new;
        float beta[NT];
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
          const float mnew = fmaxf(mu[nt], warp_max_xor(fmaxf(lg0[nt], lg1[nt]), 4 | 8 | 16));
          const float alpha = mnew == -INFINITY ? 1.f : fast_exp2(mu[nt] - mnew);
          lsum[nt] *= alpha;
          zsum[nt] *= alpha;
          mu[nt] = mnew;
          beta[nt] = alpha * nu_ratio;
        }
        const int l0 = (lane & ~3) | (2 * (t & 1));
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
          const float bA = __shfl_sync(0xffffffffu, beta[nt], l0), bB = __shfl_sync(0xffffffffu, beta[nt], l0 + 1);
#pragma unroll
          for (int mt = 0; mt < 4; mt++) {
            acc[mt][nt][0] *= bA;
            acc[mt][nt][1] *= bB;
            acc[mt][nt][2] *= bA;
            acc[mt][nt][3] *= bB;
          }
        }
      }
      uint32_t wb[NT][2][2];
#pragma unroll
      for (int nt = 0; nt < NT; nt++) {
        const float p0 = fast_exp2(lg0[nt] - mu[nt]), p1 = fast_exp2(lg1[nt] - mu[nt]);
        lsum[nt] += p0 + p1;
        zsum[nt] = fmaf(p0, R.ok0 ? vz0 : 0.f, fmaf(p1, R.ok1 ? vz1 : 0.f, zsum[nt]));
        const uint32_t Wh = pack_half2(p0 * vs0 * inv_nu, p1 * vs1 * inv_nu);  // tokens r, r+8 of head 4nt + t
        const int src0 = 4 * (2 * t) + (r & 3), src1 = src0 + 4;
        const uint32_t h0 = __shfl_sync(0xffffffffu, Wh, src0);  // tokens 2t, 2t+8
        const uint32_t h1 = __shfl_sync(0xffffffffu, Wh, src1);  // tokens 2t+1, 2t+9
        wb[nt][0][0] = __byte_perm(h0, 0u, selW_lo);
        wb[nt][0][1] = __byte_perm(h1, 0u, selW_lo);
        wb[nt][1][0] = __byte_perm(h0, 0u, selW_hi);
        wb[nt][1][1] = __byte_perm(h1, 0u, selW_hi);
      }
      // ---- values: K index (token slot, pair half); A row r / r+8 = code
      // pair 2mt / 2mt+1 of this lane's chunk; slots t / t+4 = tokens
      // 2t + 8s / 2t + 1 + 8s (chunk words of token u at V.v[u * VW ..])
#pragma unroll
      for (int s = 0; s < 2; s++)
#pragma unroll
        for (int mt = 0; mt < 4; mt++) {
          const int pa = 2 * mt, pb = 2 * mt + 1;  // pair indices within the chunk
          const int wa = pa / (VB == 4 ? 4 : 8), wbi = pb / (VB == 4 ? 4 : 8);
          const int qa = pa % (VB == 4 ? 4 : 8), qbp = pb % (VB == 4 ? 4 : 8);
          const uint32_t a0 = kivi_pair<VB>(V.v[(2 * s) * VW + wa], qa);
          const uint32_t a1 = kivi_pair<VB>(V.v[(2 * s) * VW + wbi], qbp);
          const uint32_t a2 = kivi_pair<VB>(V.v[(2 * s + 1) * VW + wa], qa);
          const uint32_t a3 = kivi_pair<VB>(V.v[(2 * s + 1) * VW + wbi], qbp);
#pragma unroll
          for (int nt = 0; nt < NT; nt++) mma_16816(acc[mt][nt], a0, a1, a2, a3, wb[nt][s][0], wb[nt][s][1]);
        }
    };

    auto step_cursor = [&]() {
      first_tile = false;
      cur.step(a.err_word, lane == 0, (uint32_t)a.slab_bytes);
    };
    {
      KiviKeyRegs<KB> ka, kb;
      KiviValRegs v;
      load_keys(ka);
      for (int k = 0;;) {
        load_vals(v);
        if (k + 1 < seg_tiles) {
          step_cursor();
          load_keys(kb);
        }
        process(ka, v);
        if (++k == seg_tiles) break;
        load_vals(v);
        if (k + 1 < seg_tiles) {
          step_cursor();
          load_keys(ka);
        }
        process(kb, v);
        if (++k == seg_tiles) break;
      }
    }

    // ---- segment partial (raw domain): slot = warp + unit
    const int64_t slot = wg + (int64_t)b * H + h;
    const float vscale = nu / kWeightScale;
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      const float ltot = warp_sum_xor(lsum[nt], 4 | 8 | 16);
      const float ztot = warp_sum_xor(zsum[nt], 4 | 8 | 16);  // sum p z of head 4nt + t
      const int g = 4 * nt + t;
      if (g < G && r == 0) {
        a.seg_ml[(slot * G + g) * 2] = mu[nt];
        a.seg_ml[(slot * G + g) * 2 + 1] = ltot;
      }
      const int gA = 4 * nt + 2 * (t & 1);
      const float zA = __shfl_sync(0xffffffffu, ztot, (lane & ~3) | (2 * (t & 1)));
      const float zB = __shfl_sync(0xffffffffu, ztot, (lane & ~3) | (2 * (t & 1) + 1));
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        if (gA + hh < G) {
          float *row = a.seg_acc + (slot * G + gA + hh) * kD + 16 * r;
          const float zz = hh ? zB : zA;
#pragma unroll
          for (int mt = 0; mt < 4; mt++) {
            // rows r / r+8: pairs 2mt / 2mt+1; column parity t/2 selects the
            // first or second code of the pair
            const int pa = 2 * mt, pb = 2 * mt + 1;
            const int wa = pa / (VB == 4 ? 4 : 8), wbi = pb / (VB == 4 ? 4 : 8);
            const int qa = pa % (VB == 4 ? 4 : 8), qbp = pb % (VB == 4 ? 4 : 8);
            const int step = VB == 4 ? 4 : 8;
            const int ca = wa * (VB == 4 ? 8 : 16) + kivi_pair_code<VB>(qa) + (t >> 1) * step;
            const int cb = wbi * (VB == 4 ? 8 : 16) + kivi_pair_code<VB>(qbp) + (t >> 1) * step;
            row[ca] = fmaf(acc[mt][nt][hh], vscale / kivi_pair_scale<VB>(qa), zz);
            row[cb] = fmaf(acc[mt][nt][hh + 2], vscale / kivi_pair_scale<VB>(qbp), zz);
          }
        }
      }
    }

    pos += seg_tiles;
    if (pos < te) {
      j = 0;
      if (++h == H) {
        h = 0;
        do { ++b; } while (a.pre[b + 1] == a.pre[b]);
        tb = (int)(a.pre[b + 1] - a.pre[b]);
      }
    }
  }
}

template <int KB, int VB, int NT>
cudaError_t kivi_main_launch_t(const AttnArgs &a, bool query_only, int *blocks_per_sm, int blocks, cudaStream_t st) {
  auto kern = kivi_main_kernel<KB, VB, NT>;
  constexpr size_t smem_bytes = (size_t)(kivi_threads(NT) / 32) * 8 * kD * sizeof(float);
  static unsigned long long done = 0;
  cudaError_t e = set_smem_once(kern, (int)smem_bytes, done);
  if (e != cudaSuccess) return e;
  if (query_only) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, kern, kivi_threads(NT), smem_bytes);
  return launch_maybe_dependent(kern, dim3(blocks), dim3(kivi_threads(NT)), smem_bytes, st, a.pdl, a);
}

cudaError_t kivi_main(const AttnArgs &a, int k_bits, int v_bits, int nt, bool query_only, int *blocks_per_sm, int blocks,
                      cudaStream_t st) {
#define TQ_KCASE(KB, VB, N) \
  if (k_bits == KB && v_bits == VB && nt == N) return kivi_main_launch_t<KB, VB, N>(a, query_only, blocks_per_sm, blocks, st);
  TQ_KCASE(4, 4, 1) TQ_KCASE(4, 4, 2) TQ_KCASE(2, 2, 1) TQ_KCASE(2, 2, 2)
  TQ_KCASE(4, 2, 1) TQ_KCASE(4, 2, 2) TQ_KCASE(2, 4, 1) TQ_KCASE(2, 4, 2)
#undef TQ_KCASE
  return cudaErrorInvalidValue;
}

}  // namespace tq
