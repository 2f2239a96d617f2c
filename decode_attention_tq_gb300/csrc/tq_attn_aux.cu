// tq_attn_aux.cu -- the small kernels around the split-KV main kernel:
//   prep   : rotate each query once into the key basis (q_rot = H (D_K . q)/sqrt(d)),
//            project it for the QJL term (q_s = S q_rot), choose power-of-two
//            operand scales, clamp the lengths and build the tile prefix sums;
//   window : attention partial over the raw fp16 recent-token window;
//   merge  : log-sum-exp merge of all partials of a (sequence, query head),
//            one inverse rotation of the value accumulator (D_V . H acc / d),
//            plus the window part, normalised.
#include "tq_internal.cuh"

namespace tq {

__global__ void __launch_bounds__(128) attn_prep_kernel(const AttnArgs a, bool qjl) {
  __shared__ float s_q[4][kD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const int64_t cap = (int64_t)a.max_pages * a.P;
    int64_t acc = 0;
    a.pre[0] = 0;
    for (int b = 0; b < a.B; b++) {
      int64_t c = a.comp_lens[b];
      if (c < 0 || c > cap) {
        report(a.err_word, TQ_DEVERR_LENGTH);
        c = c < 0 ? 0 : cap;
      }
      a.clen[b] = (int32_t)c;
      acc += (c + kTile - 1) / kTile;
      a.pre[b + 1] = acc;
      int32_t wl = 0;
      if (a.window > 0 && a.win_lens) {
        wl = a.win_lens[b];
        if (wl < 0 || wl > a.window) {
          report(a.err_word, TQ_DEVERR_LENGTH);
          wl = wl < 0 ? 0 : a.window;
        }
      }
      a.wlen[b] = wl;
    }
    const int64_t total = acc * a.H;
    int64_t nw = (total + a.min_tiles - 1) / a.min_tiles;
    if (nw > a.nw_launch) nw = a.nw_launch;
    a.hdr->total_tiles = total;
    a.hdr->active_warps = total > 0 ? nw : 0;
  }

  const int64_t row = (int64_t)blockIdx.x * 4 + warp;  // b * Hq + qh
  if (row >= (int64_t)a.B * a.Hq) return;
  // lane holds coordinates 4*lane .. 4*lane+3
  const uint2 raw = *reinterpret_cast<const uint2 *>(a.q + row * kD + 4 * lane);
  const float2 f01 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
  const float2 f23 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
  float x[4] = {f01.x, f01.y, f23.x, f23.y};
#pragma unroll
  for (int i = 0; i < 4; i++)
    if (a.k_signs[4 * lane + i]) x[i] = -x[i];
  fwht_local<4>(x);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) fwht_xlane<4>(x, m, (lane & m) != 0);
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < 4; i++) {
    x[i] *= 0.08838834764831845f;  // 1/sqrt(128)
    mx = fmaxf(mx, fabsf(x[i]));
  }
  *reinterpret_cast<float4 *>(a.q_rot + row * kD + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
  mx = warp_max_xor(mx, 31);
  // largest |value| lands in [2^12, 2^13) after scaling by 2^e
  const int eq = mx > 0.f ? 12 - ilogbf(mx) : 0;
  int es = 0;
  if (qjl) {
#pragma unroll
    for (int i = 0; i < 4; i++) s_q[warp][4 * lane + i] = x[i];
    __syncwarp();
    float ys[4];
    float my = 0.f;
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const float4 *srow = reinterpret_cast<const float4 *>(a.S + (int64_t)(4 * lane + i) * kD);
      float acc = 0.f;
#pragma unroll 8
      for (int k = 0; k < kD / 4; k++) {
        const float4 s = __ldg(srow + k);
        acc = fmaf(s.x, s_q[warp][4 * k], acc);
        acc = fmaf(s.y, s_q[warp][4 * k + 1], acc);
        acc = fmaf(s.z, s_q[warp][4 * k + 2], acc);
        acc = fmaf(s.w, s_q[warp][4 * k + 3], acc);
      }
      ys[i] = acc;
      my = fmaxf(my, fabsf(acc));
    }
    *reinterpret_cast<float4 *>(a.q_s + row * kM + 4 * lane) = make_float4(ys[0], ys[1], ys[2], ys[3]);
    my = warp_max_xor(my, 31);
    es = my > 0.f ? 12 - ilogbf(my) : 0;
  }
  if (lane == 0) {
    a.q_exp[row * 2] = eq;
    a.q_exp[row * 2 + 1] = es;
  }
}

// One block (256 threads) per (b, kv head) over the raw fp16 window, in
// chunks of 128 tokens: (1) scores, two threads per token (64 coordinates
// each, 16-byte loads); (2) per-head max / exp / sum with warp reductions;
// (3) values, thread = (coordinate pair, head group) streaming half2 rows.
__global__ void __launch_bounds__(256) attn_window_kernel(const AttnArgs a) {
  __shared__ float s_q[8][kD];
  __shared__ float s_p[8][128];
  __shared__ float s_mu[8], s_l[8], s_alpha[8];
  const int b = blockIdx.x / a.H, h = blockIdx.x % a.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G;
  const int wl = a.wlen[b];
  for (int i = tid; i < G * kD; i += 256) s_q[i / kD][i % kD] = __half2float(a.q[((int64_t)b * a.Hq + h * G) * kD + i]);
  if (tid < G) {
    s_mu[tid] = -INFINITY;
    s_l[tid] = 0.f;
  }
  const int cpair = tid & 63, hg = tid >> 6;  // value phase: coordinates 2*cpair, 2*cpair+1; heads hg, hg+4
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  __syncthreads();
  const float sscale = kLog2e * 0.08838834764831845f;  // log2(e)/sqrt(d)
  const __half *kbase = a.k_win + ((int64_t)b * a.H + h) * a.window * kD;
  const __half *vbase = a.v_win + ((int64_t)b * a.H + h) * a.window * kD;
  for (int c0 = 0; c0 < wl; c0 += 128) {
    const int n = min(128, wl - c0);
    {  // (1) scores
      const int i = tid >> 1, half = tid & 1;
      float part[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (i < n) {
        const uint4 *src = reinterpret_cast<const uint4 *>(kbase + (int64_t)(c0 + i) * kD + 64 * half);
        uint4 raw[8];
#pragma unroll
        for (int k = 0; k < 8; k++) raw[k] = src[k];
#pragma unroll
        for (int k = 0; k < 8; k++) {
          const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
          for (int e = 0; e < 4; e++) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[e]));
            const int c = 64 * half + 8 * k + 2 * e;
#pragma unroll
            for (int g = 0; g < 8; g++)
              if (g < G) part[g] = fmaf(f.x, s_q[g][c], fmaf(f.y, s_q[g][c + 1], part[g]));
          }
        }
      }
#pragma unroll
      for (int g = 0; g < 8; g++) {
        const float tot = part[g] + __shfl_xor_sync(0xffffffffu, part[g], 1);
        if (g < G && half == 0 && i < n) s_p[g][i] = tot * sscale;
      }
    }
    __syncthreads();
    for (int g = warp; g < G; g += 8) {  // (2) softmax statistics, one warp per head
      float v[4], m = -INFINITY;
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int i = lane + 32 * k;
        v[k] = i < n ? s_p[g][i] : -INFINITY;
        m = fmaxf(m, v[k]);
      }
      m = warp_max_xor(m, 31);
      const float mnew = fmaxf(s_mu[g], m);
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int i = lane + 32 * k;
        const float p = i < n ? exp2f(v[k] - mnew) : 0.f;
        if (i < n) s_p[g][i] = p;
        sum += p;
      }
      sum = warp_sum_xor(sum, 31);
      if (lane == 0) {
        const float alpha = exp2f(s_mu[g] - mnew);
        s_alpha[g] = alpha;
        s_l[g] = s_l[g] * alpha + sum;
        s_mu[g] = mnew;
      }
    }
    __syncthreads();
    {  // (3) values
#pragma unroll
      for (int gi = 0; gi < 2; gi++) {
        const int g = hg + 4 * gi;
        if (g < G) {
          acc[gi][0] *= s_alpha[g];
          acc[gi][1] *= s_alpha[g];
        }
      }
      const __half2 *vrow = reinterpret_cast<const __half2 *>(vbase + (int64_t)c0 * kD) + cpair;
      int i = 0;
      for (; i + 8 <= n; i += 8) {
        __half2 vv[8];
#pragma unroll
        for (int k = 0; k < 8; k++) vv[k] = vrow[(i + k) * (kD / 2)];
#pragma unroll
        for (int k = 0; k < 8; k++) {
          const float2 f = __half22float2(vv[k]);
#pragma unroll
          for (int gi = 0; gi < 2; gi++) {
            const int g = hg + 4 * gi;
            if (g < G) {
              const float p = s_p[g][i + k];
              acc[gi][0] = fmaf(p, f.x, acc[gi][0]);
              acc[gi][1] = fmaf(p, f.y, acc[gi][1]);
            }
          }
        }
      }
      for (; i < n; i++) {
        const float2 f = __half22float2(vrow[i * (kD / 2)]);
#pragma unroll
        for (int gi = 0; gi < 2; gi++) {
          const int g = hg + 4 * gi;
          if (g < G) {
            const float p = s_p[g][i];
            acc[gi][0] = fmaf(p, f.x, acc[gi][0]);
            acc[gi][1] = fmaf(p, f.y, acc[gi][1]);
          }
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int gi = 0; gi < 2; gi++) {
    const int g = hg + 4 * gi;
    if (g < G) {
      const int64_t row = (int64_t)b * a.Hq + h * G + g;
      if (cpair == 0) {
        a.win_ml[row * 2] = s_mu[g];
        a.win_ml[row * 2 + 1] = s_l[g];
      }
      *reinterpret_cast<float2 *>(a.win_acc + row * kD + 2 * cpair) = make_float2(acc[gi][0], acc[gi][1]);
    }
  }
}

// Warp that owns tile x: largest w in [0, NW) with floor(T*w/NW) <= x.
__device__ __forceinline__ int64_t tile_owner(int64_t x, int64_t T, int64_t NW) {
  const int64_t w = (NW * (x + 1) + T - 1) / T - 1;
  return w < NW - 1 ? w : NW - 1;
}

__global__ void __launch_bounds__(128) attn_merge_kernel(const AttnArgs a) {
  __shared__ float s_x[kD];
  const int64_t row = blockIdx.x;  // b * Hq + qh
  const int b = (int)(row / a.Hq), qh = (int)(row % a.Hq);
  const int h = qh / a.G, g = qh % a.G;
  const int j = threadIdx.x;
  const int64_t T = a.hdr->total_tiles, NW = a.hdr->active_warps;
  float mu = -INFINITY, l = 0.f, A = 0.f;
  const int64_t tb = a.pre[b + 1] - a.pre[b];
  if (tb > 0 && NW > 0) {
    const int64_t o = a.H * a.pre[b] + h * tb;
    const int64_t w0 = tile_owner(o, T, NW), w1 = tile_owner(o + tb - 1, T, NW);
    const int64_t unit = (int64_t)b * a.H + h;
    for (int64_t w = w0; w <= w1; w++) {
      if (T * w / NW >= T * (w + 1) / NW) continue;  // empty range
      const int64_t base = (w + unit) * a.G + g;
      const float ms = a.seg_ml[base * 2], ls = a.seg_ml[base * 2 + 1];
      const float As = a.seg_acc[base * kD + j];
      const float mn = fmaxf(mu, ms);
      if (mn == -INFINITY) continue;
      const float sa = exp2f(mu - mn), sb = exp2f(ms - mn);
      l = l * sa + ls * sb;
      A = A * sa + As * sb;
      mu = mn;
    }
  }
  // inverse rotation of the rotated-domain accumulator: D_V . (H A) / d
  float x = A;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, x, m);
    x = (j & m) ? (o - x) : (x + o);
  }
#pragma unroll
  for (int m = 32; m < kD; m <<= 1) {
    s_x[j] = x;
    __syncthreads();
    const float o = s_x[j ^ m];
    __syncthreads();
    x = (j & m) ? (o - x) : (x + o);
  }
  x = (a.v_signs[j] ? -x : x) * (1.0f / (float)kD);

  float mw = -INFINITY, lw = 0.f, Aw = 0.f;
  if (a.window > 0 && a.wlen[b] > 0) {
    mw = a.win_ml[row * 2];
    lw = a.win_ml[row * 2 + 1];
    Aw = a.win_acc[row * kD + j];
  }
  const float M = fmaxf(mu, mw);
  float o = 0.f;
  if (M != -INFINITY) {
    const float sc = exp2f(mu - M), sw = exp2f(mw - M);
    const float den = l * sc + lw * sw;
    o = den > 0.f ? (x * sc + Aw * sw) / den : 0.f;
  }
  a.out[row * kD + j] = o;
}

cudaError_t launch_attn_prep(const AttnArgs &a, bool qjl, cudaStream_t st) {
  const int64_t rows = (int64_t)a.B * a.Hq;
  const unsigned blocks = (unsigned)((rows + 3) / 4);
  attn_prep_kernel<<<blocks, 128, 0, st>>>(a, qjl);
  return cudaGetLastError();
}

cudaError_t launch_attn_window(const AttnArgs &a, cudaStream_t st) {
  attn_window_kernel<<<(unsigned)((int64_t)a.B * a.H), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_attn_merge(const AttnArgs &a, cudaStream_t st) {
  attn_merge_kernel<<<(unsigned)((int64_t)a.B * a.Hq), 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tq
