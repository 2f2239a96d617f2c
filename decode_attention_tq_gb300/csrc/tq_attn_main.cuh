// tq_attn_main.cuh -- split-KV fused decode attention over the packed cache.
//
// Work split.  The compressed cache of one layer is a flat list of 16-token
// tiles ordered by (sequence b, kv head h, tile j).  Warp w of the launch owns
// the contiguous tile range [T*w/NW, T*(w+1)/NW): every warp streams the same
// number of tiles (+-1), independent of sequence lengths, with no atomics and
// no block-level synchronisation in the hot loop.  Where a range crosses a
// (b, h) boundary the warp emits one partial (running max, sum, rotated value
// accumulator) per piece into slot w + (b*H + h), which is unique because both
// w and the unit index grow monotonically along the list.
//
// Per tile (16 tokens, one (b, h)) a warp does, on the tensor cores
// (mma.sync m16n8k16, fp16 operands, fp32 accumulation):
//   scores[16 x 2G] = Kcodes[16 x 128] * Qrot[128 x 2G]
//     A: centroid of each code pair from a shared-memory table (fp16 hi and lo
//        parts, two MMAs); B: the rotated query, hi/lo split over the 2G
//        columns, so the product is exact to ~2^-22;
//   QJL (keys): + signs[16 x 128] * (S q_rot)[128 x 2G], the +-1 operands are
//        exact in fp16;
//   online softmax in fp32 (log2 domain);
//   acc[128 x 2G] += Vcodes^T[128 x 16] * W[16 x 2G], W = p_i * n_i / nu
//        (nu = running max value norm) split hi/lo over the columns.
// Thread (r = lane/4, t = lane%4) of the MMA layout owns head 4*nt + t of
// n-tile nt, tokens r and r+8 of a tile for the scores, and output
// coordinates 16r..16r+15 of the value accumulator.
#pragma once

#include "tq_internal.cuh"

namespace tq {

template <int KB, int VB, bool QJL>
struct TileRegs {
  uint32_t k0[KB], k1[KB];  // key code slice (coords 32t..32t+31) of tokens r, r+8
  float nk0, nk1;           // key norms of tokens r, r+8
  float g0, g1;             // QJL gammas
  uint32_t s0, s1;          // QJL sign word t of tokens r, r+8
  float nv0, nv1;           // value norms of tokens r, r+8
  uint32_t vlo[4], vhi[4];  // value code bits of coords 16r..16r+15 of tokens 2t, 2t+1, 2t+8, 2t+9
  bool ok0, ok1;            // token r / r+8 is a live compressed token
};

// Code pair p (coordinates 32t+2p, 32t+2p+1) of a key slice.
template <int KB>
__device__ __forceinline__ uint32_t key_pair(const uint32_t (&w)[KB], int p) {
  if constexpr (KB == 4) {
    return (w[p >> 2] >> ((p & 3) * 8)) & 0xFFu;
  } else if constexpr (KB == 2) {
    return (w[p >> 3] >> ((p & 7) * 4)) & 0xFu;
  } else {
    const int bit = 6 * p, wi = bit >> 5, sh = bit & 31;
    if (sh <= 26) return (w[wi] >> sh) & 63u;
    return __funnelshift_r(w[wi], w[wi + 1], sh) & 63u;
  }
}

// Code pair mt (coordinates 16r+2mt, 16r+2mt+1) of a value slice.
template <int VB>
__device__ __forceinline__ uint32_t value_pair(uint32_t lo, uint32_t hi, int mt) {
  constexpr uint32_t mask = (1u << (2 * VB)) - 1u;
  const int bit = 2 * VB * mt;
  if (bit + 2 * VB <= 32) return (lo >> bit) & mask;
  if (bit >= 32) return (hi >> (bit - 32)) & mask;
  return __funnelshift_r(lo, hi, bit) & mask;
}

// +-1 fp16 pair from sign bits p and p+16 of a word (bit set -> +1).
__device__ __forceinline__ uint32_t sign_pair(uint32_t w, int p) {
  return 0xBC00BC00u ^ ((w << (15 - p)) & 0x80008000u);
}

template <int NB>
__device__ __forceinline__ void ldg_words(const uint8_t *p, uint32_t (&w)[NB]) {
  if constexpr (NB == 4) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (NB == 2) {
    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int k = 0; k < NB; k++) w[k] = __ldg(reinterpret_cast<const uint32_t *>(p) + k);
  }
}

template <int KB, int VB, bool QJL>
__device__ __forceinline__ void load_tile(const AttnArgs &a, int b, int h, int64_t j, int clen, int r, int t,
                                          TileRegs<KB, VB, QJL> &R) {
  constexpr int KCB = 16 * KB, VCB = 16 * VB;
  const int tpp = a.P >> 4;
  const int64_t pidx = j / tpp;
  const int o0 = (int)(j - pidx * tpp) * 16;
  int32_t page = __ldg(a.block_tables + (int64_t)b * a.max_pages + pidx);
  const bool pok = page >= 0 && (int64_t)page < a.num_pages;
  if (!pok) {
    if (r == 0 && t == 0) report(a.err_word, TQ_DEVERR_PAGE_RANGE);
    page = 0;
  }
  const uint8_t *slab = a.pool + (int64_t)page * a.page_bytes + (int64_t)h * a.slab_bytes;
  const int64_t tok0 = j * 16;
  R.ok0 = pok && (tok0 + r < clen);
  R.ok1 = pok && (tok0 + r + 8 < clen);
  const uint8_t *kc = slab + a.k_codes_o + t * 4 * KB;
  ldg_words<KB>(kc + (o0 + r) * KCB, R.k0);
  ldg_words<KB>(kc + (o0 + r + 8) * KCB, R.k1);
  const float *kn = reinterpret_cast<const float *>(slab + a.k_norm_o) + o0;
  R.nk0 = __ldg(kn + r);
  R.nk1 = __ldg(kn + r + 8);
  if constexpr (QJL) {
    const float *kg = reinterpret_cast<const float *>(slab + a.k_gamma_o) + o0;
    R.g0 = __ldg(kg + r);
    R.g1 = __ldg(kg + r + 8);
    const uint32_t *ks = reinterpret_cast<const uint32_t *>(slab + a.k_signs_o) + o0 * (kM / 32) + t;
    R.s0 = __ldg(ks + r * (kM / 32));
    R.s1 = __ldg(ks + (r + 8) * (kM / 32));
  }
  const float *vn = reinterpret_cast<const float *>(slab + a.v_norm_o) + o0;
  R.nv0 = __ldg(vn + r);
  R.nv1 = __ldg(vn + r + 8);
  const uint8_t *vc = slab + a.v_codes_o;
  const int vt[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    const uint8_t *row = vc + (o0 + vt[i]) * VCB;
    if constexpr (VB == 4) {
      const uint2 v = __ldg(reinterpret_cast<const uint2 *>(row + 8 * r));
      R.vlo[i] = v.x;
      R.vhi[i] = v.y;
    } else if constexpr (VB == 2) {
      R.vlo[i] = __ldg(reinterpret_cast<const uint32_t *>(row + 4 * r));
      R.vhi[i] = 0u;
    } else {
      // 48 bits starting at byte 6r: two aligned words, then shift by 0 or 16
      const int w0 = (6 * r) >> 2;
      const uint32_t x0 = __ldg(reinterpret_cast<const uint32_t *>(row) + w0);
      const uint32_t x1 = __ldg(reinterpret_cast<const uint32_t *>(row) + w0 + 1);
      const int sh = ((6 * r) & 3) * 8;
      R.vlo[i] = __funnelshift_r(x0, x1, sh);
      R.vhi[i] = x1 >> sh;
    }
  }
}

template <int KB, int VB, bool QJL, int NT>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_main_kernel(const AttnArgs a) {
  constexpr int EK = 1 << (2 * KB), EV = 1 << (2 * VB);
  extern __shared__ __align__(16) uint8_t smem[];
  uint2 *lutK = reinterpret_cast<uint2 *>(smem);            // [EK][32] (hi, lo) x256
  uint32_t *lutV = reinterpret_cast<uint32_t *>(lutK + EK * 32);  // [EV][32] x256

  // Bank-private centroid-pair tables: entry e of lane l lives in bank l.
  for (int i = threadIdx.x; i < EK * 32; i += blockDim.x) {
    const int e = i >> 5;
    __half h0, l0, h1, l1;
    split_half(__ldg(a.k_cb + (e & ((1 << KB) - 1))) * kCentScale, h0, l0);
    split_half(__ldg(a.k_cb + (e >> KB)) * kCentScale, h1, l1);
    lutK[i] = make_uint2(pack_half2_raw(h0, h1), pack_half2_raw(l0, l1));
  }
  for (int i = threadIdx.x; i < EV * 32; i += blockDim.x) {
    const int e = i >> 5;
    lutV[i] = pack_half2(__ldg(a.v_cb + (e & ((1 << VB) - 1))) * kCentScale, __ldg(a.v_cb + (e >> VB)) * kCentScale);
  }
  __syncthreads();

  const int lane = threadIdx.x & 31, r = lane >> 2, t = lane & 3;
  const int64_t wg = (int64_t)blockIdx.x * kAttnWarps + (threadIdx.x >> 5);
  const int64_t T = a.hdr->total_tiles;
  const int64_t NW = a.hdr->active_warps;
  if (wg >= NW) return;
  const int64_t ts = T * wg / NW, te = T * (wg + 1) / NW;
  if (ts >= te) return;
  const uint2 *lutK_l = lutK + lane;
  const uint32_t *lutV_l = lutV + lane;
  const int H = a.H, G = a.G, Hq = a.Hq;

  // locate the first tile: largest b with H * pre[b] <= ts
  int b = 0;
  {
    int lo = 0, hi = a.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (H * a.pre[mid] <= ts) lo = mid; else hi = mid;
    }
    b = lo;
  }
  int64_t tb = a.pre[b + 1] - a.pre[b];
  int h = (int)((ts - H * a.pre[b]) / tb);
  int64_t j = (ts - H * a.pre[b]) - (int64_t)h * tb;
  int64_t pos = ts;

  while (pos < te) {
    const int64_t seg_tiles = min(te - pos, tb - j);
    const int clen = a.clen[b];

    // ---- segment setup: query operands for the G heads of (b, h)
    uint32_t qb[NT][8][2];
    uint32_t sb[NT][QJL ? 8 : 1][2];
    float cK[NT], cQ[NT];
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      const int gcol = 4 * nt + (r >> 1);
      const bool lo_part = (r & 1) != 0;
      const bool gval = gcol < G;
      const int64_t qrow = ((int64_t)b * Hq + (int64_t)h * G + (gval ? gcol : 0));
      const int ecol = gval ? a.q_exp[qrow * 2] : 0;
      const float sc = ldexpf(1.0f, ecol);
      const float *qr = a.q_rot + qrow * kD + 32 * t;
#pragma unroll
      for (int kk = 0; kk < 8; kk++) {
        float4 v = gval ? *reinterpret_cast<const float4 *>(qr + 4 * kk) : make_float4(0.f, 0.f, 0.f, 0.f);
        __half hx, lx, hy, ly, hz, lz, hw, lw;
        split_half(v.x * sc, hx, lx);
        split_half(v.y * sc, hy, ly);
        split_half(v.z * sc, hz, lz);
        split_half(v.w * sc, hw, lw);
        qb[nt][kk][0] = lo_part ? pack_half2_raw(lx, ly) : pack_half2_raw(hx, hy);
        qb[nt][kk][1] = lo_part ? pack_half2_raw(lz, lw) : pack_half2_raw(hz, hw);
      }
      if constexpr (QJL) {
        const int es = gval ? a.q_exp[qrow * 2 + 1] : 0;
        const float ss = ldexpf(1.0f, es);
        const float *qs = a.q_s + qrow * kM + 32 * t;
        float v[32];
#pragma unroll
        for (int k4 = 0; k4 < 8; k4++) {
          const float4 f = gval ? *reinterpret_cast<const float4 *>(qs + 4 * k4) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[4 * k4] = f.x * ss; v[4 * k4 + 1] = f.y * ss; v[4 * k4 + 2] = f.z * ss; v[4 * k4 + 3] = f.w * ss;
        }
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          __half h0, l0, h1, l1, h2, l2, h3, l3;
          split_half(v[2 * kk], h0, l0);
          split_half(v[2 * kk + 16], h1, l1);
          split_half(v[2 * kk + 1], h2, l2);
          split_half(v[2 * kk + 17], h3, l3);
          sb[nt][kk][0] = lo_part ? pack_half2_raw(l0, l1) : pack_half2_raw(h0, h1);
          sb[nt][kk][1] = lo_part ? pack_half2_raw(l2, l3) : pack_half2_raw(h2, h3);
        }
      }
      // score constants of this thread's own head g = 4nt + t (log2 domain)
      const int gown = 4 * nt + t;
      const int64_t orow = ((int64_t)b * Hq + (int64_t)h * G + (gown < G ? gown : 0));
      const int eq = a.q_exp[orow * 2];
      cK[nt] = ldexpf(kLog2e / (float)kD, -(eq + 8));
      if constexpr (QJL) {
        const int es = a.q_exp[orow * 2 + 1];
        // sqrt(pi/2) / (m sqrt(d))
        cQ[nt] = ldexpf(kLog2e * 1.2533141373155003f / ((float)kM * 11.313708498984761f), -es);
      } else {
        cQ[nt] = 0.f;
      }
    }

    float mu[NT], lsum[NT];
    float acc[8][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      mu[nt] = -INFINITY;
      lsum[nt] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 8; mt++)
#pragma unroll
        for (int i = 0; i < 4; i++) acc[mt][nt][i] = 0.f;
    }
    float nu = 0.f;

    TileRegs<KB, VB, QJL> cur, nxt;
    load_tile<KB, VB, QJL>(a, b, h, j, clen, r, t, cur);
    for (int64_t k = 0; k < seg_tiles; k++) {
      if (k + 1 < seg_tiles) load_tile<KB, VB, QJL>(a, b, h, j + k + 1, clen, r, t, nxt);
      if (__any_sync(0xffffffffu, cur.ok0 || cur.ok1)) {
        // ---- scores
        float sk[NT][4], sq[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
          for (int i = 0; i < 4; i++) { sk[nt][i] = 0.f; sq[nt][i] = 0.f; }
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const uint2 L00 = lutK_l[key_pair<KB>(cur.k0, 2 * kk) << 5];
          const uint2 L10 = lutK_l[key_pair<KB>(cur.k1, 2 * kk) << 5];
          const uint2 L01 = lutK_l[key_pair<KB>(cur.k0, 2 * kk + 1) << 5];
          const uint2 L11 = lutK_l[key_pair<KB>(cur.k1, 2 * kk + 1) << 5];
#pragma unroll
          for (int nt = 0; nt < NT; nt++) {
            mma_16816(sk[nt], L00.x, L10.x, L01.x, L11.x, qb[nt][kk][0], qb[nt][kk][1]);
            mma_16816(sk[nt], L00.y, L10.y, L01.y, L11.y, qb[nt][kk][0], qb[nt][kk][1]);
          }
          if constexpr (QJL) {
            const uint32_t a0 = sign_pair(cur.s0, 2 * kk), a1 = sign_pair(cur.s1, 2 * kk);
            const uint32_t a2 = sign_pair(cur.s0, 2 * kk + 1), a3 = sign_pair(cur.s1, 2 * kk + 1);
#pragma unroll
            for (int nt = 0; nt < NT; nt++) mma_16816(sq[nt], a0, a1, a2, a3, sb[nt][kk][0], sb[nt][kk][1]);
          }
        }
        // ---- online softmax (log2 domain) and value weights
        float vn0 = cur.ok0 ? cur.nv0 : 0.f, vn1 = cur.ok1 ? cur.nv1 : 0.f;
        const float tnu = warp_max_xor(fmaxf(vn0, vn1), 4 | 8 | 16);
        const float nu_new = fmaxf(nu, tnu);
        const float nu_ratio = nu_new > 0.f ? nu / nu_new : 1.f;
        const float inv_nu = nu_new > 0.f ? kWeightScale / nu_new : 0.f;
        nu = nu_new;
        uint32_t wb[NT][2];
        bool rescale = false;
        float beta[NT];
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
          float l0 = (sk[nt][0] + sk[nt][1]) * cK[nt];
          float l1 = (sk[nt][2] + sk[nt][3]) * cK[nt];
          if constexpr (QJL) {
            l0 = fmaf(cur.g0 * (sq[nt][0] + sq[nt][1]), cQ[nt], l0);
            l1 = fmaf(cur.g1 * (sq[nt][2] + sq[nt][3]), cQ[nt], l1);
          }
          l0 = cur.ok0 ? cur.nk0 * l0 : -INFINITY;
          l1 = cur.ok1 ? cur.nk1 * l1 : -INFINITY;
          const float tmax = warp_max_xor(fmaxf(l0, l1), 4 | 8 | 16);
          const float mnew = fmaxf(mu[nt], tmax);
          const float alpha = exp2f(mu[nt] - mnew);
          const float p0 = exp2f(l0 - mnew), p1 = exp2f(l1 - mnew);
          lsum[nt] = fmaf(lsum[nt], alpha, p0 + p1);
          mu[nt] = mnew;
          beta[nt] = alpha * nu_ratio;
          rescale |= beta[nt] != 1.f;
          const float w0 = p0 * vn0 * inv_nu, w1 = p1 * vn1 * inv_nu;
          __half wh0, wl0, wh1, wl1;
          split_half(w0, wh0, wl0);
          split_half(w1, wh1, wl1);
          const uint32_t Wh = pack_half2_raw(wh0, wh1), Wl = pack_half2_raw(wl0, wl1);
          const int src0 = 4 * (2 * t) + (r >> 1), src1 = src0 + 4;
          const uint32_t h0 = __shfl_sync(0xffffffffu, Wh, src0), q0 = __shfl_sync(0xffffffffu, Wl, src0);
          const uint32_t h1 = __shfl_sync(0xffffffffu, Wh, src1), q1 = __shfl_sync(0xffffffffu, Wl, src1);
          const uint32_t x0 = (r & 1) ? q0 : h0, x1 = (r & 1) ? q1 : h1;
          wb[nt][0] = __byte_perm(x0, x1, 0x5410);
          wb[nt][1] = __byte_perm(x0, x1, 0x7632);
        }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
          for (int mt = 0; mt < 8; mt++)
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
#pragma unroll
              for (int i = 0; i < 4; i++) acc[mt][nt][i] *= beta[nt];
        }
        // ---- values
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
          const uint32_t V0 = lutV_l[value_pair<VB>(cur.vlo[0], cur.vhi[0], mt) << 5];
          const uint32_t V1 = lutV_l[value_pair<VB>(cur.vlo[1], cur.vhi[1], mt) << 5];
          const uint32_t V2 = lutV_l[value_pair<VB>(cur.vlo[2], cur.vhi[2], mt) << 5];
          const uint32_t V3 = lutV_l[value_pair<VB>(cur.vlo[3], cur.vhi[3], mt) << 5];
          const uint32_t a0 = __byte_perm(V0, V1, 0x5410), a1 = __byte_perm(V0, V1, 0x7632);
          const uint32_t a2 = __byte_perm(V2, V3, 0x5410), a3 = __byte_perm(V2, V3, 0x7632);
#pragma unroll
          for (int nt = 0; nt < NT; nt++) mma_16816(acc[mt][nt], a0, a1, a2, a3, wb[nt][0], wb[nt][1]);
        }
      }
      cur = nxt;
    }

    // ---- segment partial: slot = warp + unit
    const int64_t slot = wg + (int64_t)b * H + h;
    const float vscale = nu / (kWeightScale * kCentScale);
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      const float ltot = warp_sum_xor(lsum[nt], 4 | 8 | 16);
      const int g = 4 * nt + t;
      if (g < G) {
        const int64_t base = slot * G + g;
        if (r == 0) {
          a.seg_ml[base * 2] = mu[nt];
          a.seg_ml[base * 2 + 1] = ltot;
        }
        float o[16];
#pragma unroll
        for (int mt = 0; mt < 8; mt++) {
          o[2 * mt] = (acc[mt][nt][0] + acc[mt][nt][1]) * vscale;
          o[2 * mt + 1] = (acc[mt][nt][2] + acc[mt][nt][3]) * vscale;
        }
        float4 *dst = reinterpret_cast<float4 *>(a.seg_acc + base * kD + 16 * r);
#pragma unroll
        for (int k4 = 0; k4 < 4; k4++) dst[k4] = make_float4(o[4 * k4], o[4 * k4 + 1], o[4 * k4 + 2], o[4 * k4 + 3]);
      }
    }

    pos += seg_tiles;
    if (pos < te) {  // next non-empty (b, h)
      j = 0;
      if (++h == H) {
        h = 0;
        do { ++b; } while (a.pre[b + 1] == a.pre[b]);
        tb = a.pre[b + 1] - a.pre[b];
      }
    }
  }
}

template <int KB, int VB, bool QJL, int NT>
cudaError_t attn_main_launch_t(const AttnArgs &a, bool query_only, int *blocks_per_sm, int blocks, cudaStream_t st) {
  constexpr int EK = 1 << (2 * KB), EV = 1 << (2 * VB);
  constexpr size_t smem = (size_t)EK * 32 * 8 + (size_t)EV * 32 * 4;
  auto kern = attn_main_kernel<KB, VB, QJL, NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (query_only) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, kern, kAttnThreads, smem);
  kern<<<blocks, kAttnThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int KB>
cudaError_t attn_main_dispatch(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *bps, int blocks,
                               cudaStream_t st) {
#define TQ_CASE(VB, Q, N) \
  if (v_bits == VB && qjl == Q && nt == N) return attn_main_launch_t<KB, VB, Q, N>(a, query_only, bps, blocks, st);
  TQ_CASE(2, false, 1) TQ_CASE(2, false, 2) TQ_CASE(2, true, 1) TQ_CASE(2, true, 2)
  TQ_CASE(3, false, 1) TQ_CASE(3, false, 2) TQ_CASE(3, true, 1) TQ_CASE(3, true, 2)
  TQ_CASE(4, false, 1) TQ_CASE(4, false, 2) TQ_CASE(4, true, 1) TQ_CASE(4, true, 2)
#undef TQ_CASE
  return cudaErrorInvalidValue;
}

}  // namespace tq
