// tq_attn_aux.cu -- the small kernels around the split-KV main kernel:
//   prep   : (one launch, three kinds of block) tile prefix sums and clamped
//            lengths; each query rotated once into the key basis
//            (q_rot = H (D_K . q)/sqrt(d)), projected for the QJL term
//            (S q_rot, one block per row), with power-of-two operand scales,
//            written as the main kernel's fp16 hi/lo operands; and
//            attention partials over the raw fp16 recent-token window, one
//            per 32-token chunk;
//   merge  : log-sum-exp merge of the compressed partials of a (sequence,
//            query head), one inverse rotation of their value accumulator
//            (D_V . H acc / d), then the window partials, normalised; one
//            warp per (sequence, query head) when they have few partials,
//            blocks of 16 warps sharing them otherwise (several blocks per
//            row, the last one to finish merging their results).
#include "tq_internal.cuh"

namespace tq {

// Block 0, warp 0: clamped lengths and tile prefix sums, 32 sequences at a
// time (a warp scan), then the header the main and merge kernels read.
__device__ void prep_lengths(const AttnArgs &a, int lane) {
  const int64_t cap = (int64_t)a.max_pages * a.P;
  int64_t carry = 0;
  if (lane == 0) a.pre[0] = 0;
  for (int b0 = 0; b0 < a.B; b0 += 32) {
    const int b = b0 + lane;
    int64_t tiles = 0;
    if (b < a.B) {
      int64_t c = a.comp_lens[b];
      if (c < 0 || c > cap) {
        report(a.err_word, TQ_DEVERR_LENGTH);
        c = c < 0 ? 0 : cap;
      }
      a.clen[b] = (int32_t)c;
      tiles = (c + kTile - 1) / kTile;
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
    int64_t inc = tiles;  // inclusive scan over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    if (b < a.B) a.pre[b + 1] = carry + inc;
    carry += __shfl_sync(0xffffffffu, inc, 31);
  }
  if (lane == 0) {
    const int64_t total = carry * a.H;
    int64_t nw = (total + a.min_tiles - 1) / a.min_tiles;
    if (nw > a.nw_launch) nw = a.nw_launch;
    a.hdr->total_tiles = total;
    a.hdr->active_warps = total > 0 ? nw : 0;
  }
}

// The query row rotated into the key basis, q_rot = H (D_K . q) / sqrt(d)
// (a raw-domain KIVI cache takes the query as it is): lane holds
// coordinates 4 lane .. 4 lane + 3.
__device__ __forceinline__ void rotate_query(const AttnArgs &a, int64_t row, int lane, float (&x)[4]) {
  const uint2 raw = __ldcg(reinterpret_cast<const uint2 *>(a.q + row * kD + 4 * lane));
  const float2 f01 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
  const float2 f23 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
  x[0] = f01.x;
  x[1] = f01.y;
  x[2] = f23.x;
  x[3] = f23.y;
  if (!a.raw) {
#pragma unroll
    for (int i = 0; i < 4; i++)
      if (__ldcg(a.k_signs + 4 * lane + i)) x[i] = -x[i];
    fwht_local<4>(x);
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) fwht_xlane<4>(x, m, (lane & m) != 0);
#pragma unroll
    for (int i = 0; i < 4; i++) x[i] *= 0.08838834764831845f;  // 1/sqrt(128)
  }
}

// Power-of-two operand scale: the largest |value| lands in [2^12, 2^13).
__device__ __forceinline__ int operand_exponent(float mx) { return mx > 0.f ? 12 - ilogbf(mx) : 0; }

// Stores q_rot, its exponent and (rotated-domain caches) its operand parts
// and key score constant (one warp).
__device__ __forceinline__ void store_query(const AttnArgs &a, int64_t row, int lane, const float (&x)[4]) {
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < 4; i++) mx = fmaxf(mx, fabsf(x[i]));
  *reinterpret_cast<float4 *>(a.q_rot + row * kD + 4 * lane) = make_float4(x[0], x[1], x[2], x[3]);
  mx = warp_max_xor(mx, 31);
  const int eq = operand_exponent(mx);
  if (lane == 0) a.q_exp[row * 2] = eq;
  if (!a.raw) {
    // words 2 lane, 2 lane + 1 of parts 0 (hi) and 1 (lo): coordinates 4 lane .. 4 lane + 3
    const float sc = ldexpf(1.0f, eq);
    __half h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; i++) split_half(x[i] * sc, h[i], l[i]);
    uint32_t *op = a.q_op + row * 256;
    *reinterpret_cast<uint2 *>(op + 2 * lane) = make_uint2(pack_half2_raw(h[0], h[1]), pack_half2_raw(h[2], h[3]));
    *reinterpret_cast<uint2 *>(op + 64 + 2 * lane) = make_uint2(pack_half2_raw(l[0], l[1]), pack_half2_raw(l[2], l[3]));
    if (lane == 0) a.q_cst[row].x = ldexpf(kLog2e / (float)kD, -(eq + 8));
  }
}

// Without QJL: one warp per query row.
__device__ void prep_query(const AttnArgs &a, int64_t row, int lane) {
  float x[4];
  rotate_query(a, row, lane, x);
  store_query(a, row, lane, x);
  if (lane == 0) {
    a.q_exp[row * 2 + 1] = 0;
    a.q_cst[row].y = 0.f;
  }
}

// With QJL: one block of NW warps per query row (NW = 4 or 8).  Every warp
// rotates the row (a few shuffles); warp w projects it on S rows R w ..
// R w + R - 1 (R = 128 / NW), S q_rot: lane holds coordinates 4 lane ..
// 4 lane + 3 and reads the same coordinates of each S row (one coalesced
// 512-byte row per load, all R loads issued before the rotation).  The R
// per-lane partial dots are summed over the warp by a transposing butterfly,
// after which lane l holds row R w + l (R = 32), or lanes 2i, 2i+1 hold row
// R w + i (R = 16).
template <int NW>
__device__ void prep_query_qjl(const AttnArgs &a, int64_t row, int warp, int lane, float *s_red) {
  constexpr int R = kM / NW;
  float4 sv[R];
  const float4 *S4 = reinterpret_cast<const float4 *>(a.S + (int64_t)(R * warp) * kD) + lane;
#pragma unroll
  for (int i = 0; i < R; i++) sv[i] = __ldcg(S4 + i * (kD / 4));
  float x[4];
  rotate_query(a, row, lane, x);
  if (warp == 0) store_query(a, row, lane, x);
  float v[R];
#pragma unroll
  for (int i = 0; i < R; i++) v[i] = fmaf(sv[i].x, x[0], fmaf(sv[i].y, x[1], fmaf(sv[i].z, x[2], sv[i].w * x[3])));
#pragma unroll
  for (int m = 16, n = R / 2; n >= 1; m >>= 1, n >>= 1) {
    // keep the half of the n pairs (v[i], v[i + n]) selected by lane bit m,
    // add the partner's copy of it
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < n; i++) {
      const float keep = up ? v[i + n] : v[i], send = up ? v[i] : v[i + n];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  constexpr int kRest = R == 32 ? 0 : 1;  // lane bits not yet summed (bit 0 for R = 16)
  if (kRest) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
  const int i_row = R == 32 ? lane : (lane >> 1);  // this lane's row within the warp's R
  const float my = warp_max_xor(fabsf(v[0]), 31);
  if (lane == 0) s_red[warp] = my;
  __syncthreads();
  float mx = 0.f;
#pragma unroll
  for (int w = 0; w < NW; w++) mx = fmaxf(mx, s_red[w]);
  const int es = operand_exponent(mx);
  // slice t of parts 2 (hi) and 3 (lo): S rows 32t .. 32t + 31, value i (qop_qjl_half)
  __half hi, lo;
  split_half(v[0] * ldexpf(1.0f, es), hi, lo);
  const int srow = R * warp + i_row, t = srow >> 5, i = srow & 31;
  if (R == 32 || (lane & 1) == 0) {
    __half *op = reinterpret_cast<__half *>(a.q_op + row * 256);
    op[2 * (128 + 16 * t) + qop_qjl_half(i)] = hi;
    op[2 * (192 + 16 * t) + qop_qjl_half(i)] = lo;
  }
  if (threadIdx.x == 0) {
    a.q_exp[row * 2 + 1] = es;
    // qjl_coef / sqrt(d) (qjl_coef = sqrt(pi/2) / m for the paper's Gaussian S)
    a.q_cst[row].y = ldexpf(kLog2e * a.qjl_coef / 11.313708498984761f, -es);
  }
}

// Attention partial of the G query heads of (b, h) over window chunk c
// (tokens 32c .. 32c+31 of the raw fp16 window), 128 threads:
// (1) scores, four threads per token (32 coordinates each);
// (2) per-head max / exp / sum, one warp per head, lane = token;
// (3) values, thread = coordinate.
// Window queries in shared memory: head g, coordinate c at g * kQRow +
// (c / 32) * 34 + c % 32, so the four 32-coordinate parts read by the four
// threads of a token start in different banks (and stay 8-byte aligned).
constexpr int kQPart = 34, kQRow = 4 * kQPart;

// GM: 4 or 8, the largest head count the unrolled loops cover (G <= GM).
template <int GM>
__device__ void prep_window(const AttnArgs &a, int64_t unit, int c, float *s_q, float (*s_p)[kWinChunk]) {
  const int b = (int)(unit / a.H), h = (int)(unit % a.H);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G;
  int wl = a.win_lens ? a.win_lens[b] : 0;  // clamped here as in prep_lengths (which reports)
  wl = wl < 0 ? 0 : (wl > a.window ? a.window : wl);
  const int t0 = c * kWinChunk;
  const int n = min(kWinChunk, wl - t0);
  if (n <= 0) return;  // block-uniform (the caller's barriers follow for all threads)
  const __half *kbase = a.k_win + (((int64_t)b * a.H + h) * a.window + t0) * kD;
  const __half *vbase = a.v_win + (((int64_t)b * a.H + h) * a.window + t0) * kD;
  // every load of the block is issued before the first barrier: this
  // thread's key row part (token tid/4, coordinates 32 (tid%4) ..) and its
  // coordinate of every value row
  const int i = tid >> 2, part = tid & 3;
  uint4 raw[4] = {};
  if (i < n) {
    const uint4 *src = reinterpret_cast<const uint4 *>(kbase + (int64_t)i * kD + 32 * part);
#pragma unroll
    for (int k = 0; k < 4; k++) raw[k] = src[k];
  }
  __half vrow[kWinChunk];
#pragma unroll
  for (int k = 0; k < kWinChunk; k++) vrow[k] = k < n ? vbase[(int64_t)k * kD + tid] : __float2half(0.f);
  for (int e = tid; e < G * kD; e += blockDim.x)
    s_q[(e / kD) * kQRow + ((e % kD) >> 5) * kQPart + (e & 31)] = __half2float(a.q[((int64_t)b * a.Hq + h * G) * kD + e]);
  __syncthreads();
  {  // (1) scores
    float acc[GM];
#pragma unroll
    for (int g = 0; g < GM; g++) acc[g] = 0.f;
    if (i < n) {
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[e]));
          const int cc = 32 * part + 8 * k + 2 * e;
#pragma unroll
          for (int g = 0; g < GM; g++)
            if (g < G) {
              const float2 qq = *reinterpret_cast<const float2 *>(s_q + g * kQRow + part * kQPart + (cc & 31));
              acc[g] = fmaf(f.x, qq.x, fmaf(f.y, qq.y, acc[g]));
            }
        }
      }
    }
    const float sscale = kLog2e * 0.08838834764831845f;  // log2(e)/sqrt(d)
#pragma unroll
    for (int g = 0; g < GM; g++) {
      float v = acc[g] + __shfl_xor_sync(0xffffffffu, acc[g], 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      if (g < G && part == 0 && i < n) s_p[g][i] = v * sscale;
    }
  }
  __syncthreads();
  const int64_t nch = (a.window + kWinChunk - 1) / kWinChunk;
  for (int g = warp; g < G; g += 4) {  // (2) softmax statistics of the chunk
    const float v = lane < n ? s_p[g][lane] : -INFINITY;
    const float m = warp_max_xor(v, 31);
    const float p = lane < n ? exp2f(v - m) : 0.f;
    s_p[g][lane] = p;
    const float l = warp_sum_xor(p, 31);
    if (lane == 0) {
      const int64_t part = ((int64_t)b * a.Hq + h * G + g) * nch + c;
      a.win_ml[part * 2] = m;
      a.win_ml[part * 2 + 1] = l;
    }
  }
  __syncthreads();
  {  // (3) values (s_p is 0 past n)
    float acc[GM];
#pragma unroll
    for (int g = 0; g < GM; g++) acc[g] = 0.f;
#pragma unroll
    for (int k = 0; k < kWinChunk; k++) {
      const float v = __half2float(vrow[k]);
#pragma unroll
      for (int g = 0; g < GM; g++)
        if (g < G) acc[g] = fmaf(s_p[g][k], v, acc[g]);
    }
#pragma unroll
    for (int g = 0; g < GM; g++)
      if (g < G) a.win_acc[(((int64_t)b * a.Hq + h * G + g) * nch + c) * kD + tid] = acc[g];
  }
}

__global__ void __launch_bounds__(256) attn_prep_kernel(const AttnArgs a, bool qjl, int row_blocks) {
  __shared__ __align__(16) float s_q[8 * kQRow];
  __shared__ float s_p[8][kWinChunk];
  // Launched as a programmatic dependent of the kernel before it in the
  // stream (the append).
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (blockIdx.x >= row_blocks) {  // window chunk blocks: they read the rings the append writes
    griddep_wait();
    griddep_launch_dependents();  // the main kernel may start building its tables
    const int64_t nch = (a.window + kWinChunk - 1) / kWinChunk;
    const int64_t k = blockIdx.x - row_blocks;
    if (a.G <= 4)
      prep_window<4>(a, k / nch, (int)(k % nch), s_q, s_p);
    else
      prep_window<8>(a, k / nch, (int)(k % nch), s_q, s_p);
    return;
  }
  // Query rows before the grid wait, beside the kernel before this one: they
  // read only the call's inputs (q, S, the key sign flips, through L2), which
  // no kernel of this library writes, and write q_rot, q_op, q_exp and q_cst,
  // which only this call's main kernel reads (it waits for this grid; the
  // previous call's main kernel completed before the kernel before this one
  // let it launch).
  if (qjl) {  // one row per block (b * Hq + qh)
    if (blockDim.x == 256)
      prep_query_qjl<8>(a, blockIdx.x, warp, lane, s_q);
    else
      prep_query_qjl<4>(a, blockIdx.x, warp, lane, s_q);
  } else {
    const int64_t row = (int64_t)blockIdx.x * 4 + warp;  // b * Hq + qh
    if (row < (int64_t)a.B * a.Hq) prep_query(a, row, lane);
  }
  // After the grid wait: the lengths the append updates, and the merge
  // counters, which the previous call's merge may still be using until then.
  // The main kernel launches from here (launched earlier, beside the
  // append, its blocks measured slower once they ran).
  griddep_wait();
  griddep_launch_dependents();  // the main kernel may start building its tables
  if (blockIdx.x == 0 && warp == 0) prep_lengths(a, lane);
  if (qjl) {
    if (threadIdx.x == 0) a.merge_cnt[blockIdx.x] = 0;
  } else {
    const int64_t row = (int64_t)blockIdx.x * 4 + warp;
    if (lane == 0 && row < (int64_t)a.B * a.Hq) a.merge_cnt[row] = 0;
  }
}

// Window partials in a launch of their own, after the main kernel as its
// programmatic dependent: it starts once the main kernel is past its grid
// wait (so the append before the prep kernel has completed and the window
// rings are final) and runs beside it on the SMs the main grid leaves free.
// Every thread waits for the main kernel before it exits, so the merge
// launched after this kernel sees the main kernel's partials too.
__global__ void __launch_bounds__(128) attn_window_kernel(const AttnArgs a) {
  __shared__ __align__(16) float s_q[8 * kQRow];
  __shared__ float s_p[8][kWinChunk];
  griddep_launch_dependents();  // the merge may launch; it waits for this grid
  const int64_t nch = (a.window + kWinChunk - 1) / kWinChunk;
  const int64_t k = blockIdx.x;
  if (a.G <= 4)
    prep_window<4>(a, k / nch, (int)(k % nch), s_q, s_p);
  else
    prep_window<8>(a, k / nch, (int)(k % nch), s_q, s_p);
  griddep_wait();
}

// Warp that owns tile x: largest w in [0, NW) with floor(T*w/NW) <= x.
__device__ __forceinline__ int64_t tile_owner(int64_t x, int64_t T, int64_t NW) {
  const int64_t num = NW * (x + 1) + T - 1;
  const int64_t w = (num <= 0xffffffffll ? (int64_t)((uint32_t)num / (uint32_t)T) : num / T) - 1;  // 32-bit when it fits
  return w < NW - 1 ? w : NW - 1;
}

// kWarpMergeMaxPartials: partials per chunk of the warp merge (32 float4
// accumulators would spill).

// One chunk of up to 32 partials merged into the running (M, L, A) of a
// warp: lane i holds the (max m, sum l) of partial i, v[u] the accumulator
// coordinates 4 lane .. 4 lane + 3 of partial i0 + u.
__device__ __forceinline__ float chunk_weight(float m, float l, float &M, float &L, float4 &A, float &lsum) {
  const float Mn = fmaxf(M, warp_max_xor(m, 31));
  const float w = m == -INFINITY ? 0.f : exp2f(m - Mn);
  lsum = warp_sum_xor(l * w, 31);
  const float sold = Mn == -INFINITY ? 1.f : exp2f(M - Mn);
  A.x *= sold;
  A.y *= sold;
  A.z *= sold;
  A.w *= sold;
  L *= sold;
  M = Mn;
  return w;
}
template <int N>
__device__ __forceinline__ void chunk_accumulate(float w, int i0, const float4 (&v)[N], float4 &A) {
#pragma unroll
  for (int u = 0; u < N; u++) {
    const float wu = __shfl_sync(0xffffffffu, w, (i0 + u) & 31);
    A.x = fmaf(wu, v[u].x, A.x);
    A.y = fmaf(wu, v[u].y, A.y);
    A.z = fmaf(wu, v[u].z, A.z);
    A.w = fmaf(wu, v[u].w, A.w);
  }
}

// Online log-sum-exp merge of n partials (max, sum, accumulator) into the
// running (M, L, A) of one warp; lane l holds accumulator coordinates
// 4l .. 4l+3.  kChunk (<= 32) partials at a time: their accumulators
// (kChunk float4 loads per lane) are issued together with their (max, sum)
// pairs (one per lane), so a chunk costs one memory latency.
template <int kChunk, class ML, class ACC>
__device__ __forceinline__ void merge_partials(int64_t n, ML ml, ACC acc_of, float &M, float &L, float4 &A, int lane) {
  for (int64_t c0 = 0; c0 < n; c0 += kChunk) {
    const int cn = (int)min((int64_t)kChunk, n - c0);
    float4 v[kChunk];
#pragma unroll
    for (int u = 0; u < kChunk; u++)
      v[u] = u < cn ? reinterpret_cast<const float4 *>(acc_of(c0 + u))[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    float m = -INFINITY, l = 0.f;
    if (lane < cn) {
      const float2 p = ml(c0 + lane);
      m = p.x;
      l = p.y;
    }
    float lsum;
    const float w = chunk_weight(m, l, M, L, A, lsum);  // w = 0 past cn
    chunk_accumulate(w, 0, v, A);
    L += lsum;
  }
}

// The compressed partials of (b, h): warps w0 .. w0 + n - 1 of the main
// kernel, slot w + unit; n = 0 when the sequence has no compressed token.
struct RowParts {
  int64_t w0, n, unit, T, NW;
};
__device__ __forceinline__ RowParts row_parts(const AttnArgs &a, int b, int h) {
  RowParts r;
  r.T = a.hdr->total_tiles;
  r.NW = a.hdr->active_warps;
  r.unit = (int64_t)b * a.H + h;
  r.w0 = 0;
  r.n = 0;
  const int64_t tb = a.pre[b + 1] - a.pre[b];
  if (tb > 0 && r.NW > 0) {
    const int64_t o = a.H * a.pre[b] + h * tb;
    r.w0 = tile_owner(o, r.T, r.NW);
    r.n = tile_owner(o + tb - 1, r.T, r.NW) - r.w0 + 1;
  }
  return r;
}

// Merge of partials k0 .. k1 - 1 of a row into the running (M, L, A) of a
// warp, kChunk at a time.
template <int kChunk>
__device__ __forceinline__ void merge_row_range(const AttnArgs &a, const RowParts &r, int g, int64_t k0, int64_t k1, float &M,
                                                float &L, float4 &A, int lane) {
  merge_partials<kChunk>(
      k1 - k0,
      [&](int64_t k) {
        const int64_t w = r.w0 + k0 + k;
        // a warp's range can only be empty when there are fewer tiles than warps
        if (r.T < r.NW && r.T * w / r.NW >= r.T * (w + 1) / r.NW) return make_float2(-INFINITY, 0.f);
        return *reinterpret_cast<const float2 *>(a.seg_ml + ((w + r.unit) * a.G + g) * 2);
      },
      [&](int64_t k) { return a.seg_acc + ((r.w0 + k0 + k + r.unit) * a.G + g) * kD; }, M, L, A, lane);
}

// Window partials of a row: up to kWinPre chunks are loaded before the
// compressed merge (they do not depend on it); longer windows are merged
// from memory at the end.
constexpr int kWinPre = 8;
struct RowWindow {
  float4 v[kWinPre];
  float m, l;
  int64_t n, nch;
};
__device__ __forceinline__ void row_window_load(const AttnArgs &a, int64_t row, int b, int lane, RowWindow &w) {
  w.nch = (a.window + kWinChunk - 1) / kWinChunk;
  w.n = a.window > 0 ? (a.wlen[b] + kWinChunk - 1) / kWinChunk : 0;
  w.m = -INFINITY;
  w.l = 0.f;
  if (w.n <= kWinPre) {
#pragma unroll
    for (int u = 0; u < kWinPre; u++)
      w.v[u] = u < w.n ? reinterpret_cast<const float4 *>(a.win_acc + (row * w.nch + u) * kD)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane < w.n) {
      const float2 v = *reinterpret_cast<const float2 *>(a.win_ml + (row * w.nch + lane) * 2);
      w.m = v.x;
      w.l = v.y;
    }
  }
}

// The end of a row's merge, one warp: inverse rotation of the compressed
// accumulator, the window partials, normalisation, the output row.
__device__ __forceinline__ void row_finish(const AttnArgs &a, int64_t row, int lane, const RowWindow &win, float M, float L,
                                           float4 A) {
  // inverse rotation of the rotated-domain accumulator: D_V . (H A) / d
  // (a raw-domain KIVI accumulator is used as it is)
  if (!a.raw) {
    float x[4] = {A.x, A.y, A.z, A.w};
    fwht_local<4>(x);
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) fwht_xlane<4>(x, m, (lane & m) != 0);
#pragma unroll
    for (int i = 0; i < 4; i++) x[i] = (a.v_signs[4 * lane + i] ? -x[i] : x[i]) * (1.0f / (float)kD);
    A = make_float4(x[0], x[1], x[2], x[3]);
  }
  // window partials (raw domain), merged onto the compressed part
  if (win.n > 0 && win.n <= kWinPre) {
    float lsum;
    const float w = chunk_weight(win.m, win.l, M, L, A, lsum);
    chunk_accumulate(w, 0, win.v, A);
    L += lsum;
  } else if (win.n > kWinPre) {
    const int64_t nch = win.nch;
    merge_partials<kWinPre>(
        win.n, [&](int64_t k) { return *reinterpret_cast<const float2 *>(a.win_ml + (row * nch + k) * 2); },
        [&](int64_t k) { return a.win_acc + (row * nch + k) * kD; }, M, L, A, lane);
  }
  const bool ok = M != -INFINITY && L > 0.f;
  const float inv = ok ? 1.0f / L : 0.f;  // no token: a zero row
  float *o = a.out + row * kD + 4 * lane;  // out is 4-byte aligned
  o[0] = A.x * inv;
  o[1] = A.y * inv;
  o[2] = A.z * inv;
  o[3] = A.w * inv;
}

// Warp variant (rows with few partials): one warp per (sequence, query head)
// row, four rows per block; no shared memory and no block barriers.
// Both merge kernels read the prep kernel's outputs (tile counts, clamped
// lengths) before their grid wait: a merge block starts only after the main
// kernel is past its own grid wait, i.e. after the prep kernel has completed.
// The partials (main kernel) and the window partials are read after it.
__global__ void __launch_bounds__(128) attn_merge_warp_kernel(const AttnArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);  // b * Hq + qh
  const bool live = row < (int64_t)a.B * a.Hq;
  const int b = live ? (int)(row / a.Hq) : 0, qh = live ? (int)(row % a.Hq) : 0;
  const int h = qh / a.G, g = qh % a.G;
  RowParts r;
  if (live) r = row_parts(a, b, h);
  griddep_wait();  // the main kernel's partials
  griddep_launch_dependents();  // a dependent (the next append) may launch; it waits for this grid
  if (!live) return;
  RowWindow win;
  row_window_load(a, row, b, lane, win);
  float M = -INFINITY, L = 0.f;
  float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
  merge_row_range<kWarpMergeMaxPartials>(a, r, g, 0, r.n, M, L, A, lane);
  row_finish(a, row, lane, win, M, L, A);
}

// Wide variant (rows with many partials): blocks of kMergeWarps warps; a row
// is cut into up to merge_slices slices of about kSlicePartials partials, one
// block each.  Warp w of a block merges the w-th share of its slice
// kWideChunk partials at a time (a chunk's loads issued together: one memory
// latency), then warp 0 merges the warps' results from shared memory.  With
// one slice it finishes the row; otherwise it stores the slice result, and
// the block that completes a row's last slice (a per-row counter the prep
// kernel zeroed) merges the slice results and finishes the row.  The window
// partials are copied to shared memory asynchronously meanwhile.
__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_wide_kernel(const AttnArgs a) {
  __shared__ float4 s_acc[kMergeWarps][kD / 4];
  __shared__ float2 s_ml[kMergeWarps];
  __shared__ float4 s_wacc[kWinPre][kD / 4];
  __shared__ float2 s_wml[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = blockIdx.x / a.merge_slices;  // b * Hq + qh
  const int slice = (int)(blockIdx.x - row * a.merge_slices);
  const int b = (int)(row / a.Hq), qh = (int)(row % a.Hq);
  const int h = qh / a.G, g = qh % a.G;
  const RowParts r = row_parts(a, b, h);  // prep outputs: before the grid wait
  const int64_t nch = (a.window + kWinChunk - 1) / kWinChunk;
  const int64_t nwin = a.window > 0 ? (a.wlen[b] + kWinChunk - 1) / kWinChunk : 0;
  griddep_wait();  // the main kernel's partials
  griddep_launch_dependents();  // a dependent (the next append) may launch; it waits for this grid
  // slices this row uses (the same in every block of the row)
  int64_t ns = (r.n + kSlicePartials - 1) / kSlicePartials;
  ns = ns < 1 ? 1 : (ns > a.merge_slices ? a.merge_slices : ns);
  if (slice >= ns) return;  // block-uniform
  if (warp == kMergeWarps - 1 && nwin <= kWinPre) {
    for (int u = 0; u < nwin; u++) cp_async16(&s_wacc[u][lane], a.win_acc + (row * nch + u) * kD + 4 * lane);
    if (lane < nwin) cp_async8(&s_wml[lane], a.win_ml + (row * nch + lane) * 2);
  }
  const int64_t k0 = r.n * slice / ns, kn = r.n * (slice + 1) / ns - k0;
  float M = -INFINITY, L = 0.f;
  float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
  merge_row_range<kWideChunk>(a, r, g, k0 + kn * warp / kMergeWarps, k0 + kn * (warp + 1) / kMergeWarps, M, L, A, lane);
  s_acc[warp][lane] = A;
  if (lane == 0) s_ml[warp] = make_float2(M, L);
  cp_async_wait_all();
  __syncthreads();
  if (warp != 0) return;
  M = -INFINITY;
  L = 0.f;
  A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int h8 = 0; h8 < kMergeWarps; h8 += 8) {  // eight warps' results at a time
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; u++) v[u] = s_acc[h8 + u][lane];
    const float2 ml = lane < 8 ? s_ml[h8 + lane] : make_float2(-INFINITY, 0.f);
    float lsum;
    const float w = chunk_weight(ml.x, ml.y, M, L, A, lsum);
    chunk_accumulate(w, 0, v, A);
    L += lsum;
  }
  if (ns > 1) {
    float *part = a.merge_part + (row * a.merge_slices + slice) * kMergePartStride;
    reinterpret_cast<float4 *>(part)[lane] = A;
    if (lane == 0) *reinterpret_cast<float2 *>(part + kD) = make_float2(M, L);
    __threadfence();
    int done = 0;
    if (lane == 0) done = atomicAdd(a.merge_cnt + row, 1);
    done = __shfl_sync(0xffffffffu, done, 0);
    if (done != ns - 1) return;  // another block finishes the row
    __threadfence();
    // the row's slice results (written by other blocks: read past L1)
    M = -INFINITY;
    L = 0.f;
    A = make_float4(0.f, 0.f, 0.f, 0.f);
    const float *rp = a.merge_part + row * a.merge_slices * kMergePartStride;
    for (int s0 = 0; s0 < ns; s0 += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; u++)
        v[u] = s0 + u < ns ? __ldcg(reinterpret_cast<const float4 *>(rp + (s0 + u) * kMergePartStride) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float2 ml = s0 + lane < ns && lane < 8 ? __ldcg(reinterpret_cast<const float2 *>(rp + (s0 + lane) * kMergePartStride + kD))
                                                   : make_float2(-INFINITY, 0.f);
      float lsum;
      const float w = chunk_weight(ml.x, ml.y, M, L, A, lsum);
      chunk_accumulate(w, 0, v, A);
      L += lsum;
    }
  }
  RowWindow win;
  win.nch = nch;
  win.n = nwin;
  win.m = -INFINITY;
  win.l = 0.f;
  if (nwin <= kWinPre) {
#pragma unroll
    for (int u = 0; u < kWinPre; u++) win.v[u] = u < nwin ? s_wacc[u][lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane < nwin) {
      win.m = s_wml[lane].x;
      win.l = s_wml[lane].y;
    }
  }
  row_finish(a, row, lane, win, M, L, A);
}

cudaError_t launch_attn_prep(const AttnArgs &a, bool qjl, cudaStream_t st) {
  const int64_t rows = (int64_t)a.B * a.Hq;
  const int64_t row_blocks = qjl ? rows : (rows + 3) / 4;
  const int64_t win_blocks =
      a.window > 0 && !a.win_apart ? (int64_t)a.B * a.H * ((a.window + kWinChunk - 1) / kWinChunk) : 0;
  // QJL rows without window blocks in the launch: 8 warps per row (the window
  // blocks need 128 threads: thread = coordinate)
  const int threads = qjl && win_blocks == 0 ? 256 : 128;
  const cudaError_t e = launch_maybe_dependent(attn_prep_kernel, dim3((unsigned)(row_blocks + win_blocks)), dim3(threads),
                                               0, st, a.pdl, a, qjl, (int)row_blocks);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attn_window(const AttnArgs &a, cudaStream_t st) {
  if (!a.win_apart || a.window <= 0) return cudaSuccess;
  const int64_t blocks = (int64_t)a.B * a.H * ((a.window + kWinChunk - 1) / kWinChunk);
  const cudaError_t e = launch_maybe_dependent(attn_window_kernel, dim3((unsigned)blocks), dim3(128), 0, st, a.pdl, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attn_merge(const AttnArgs &a, cudaStream_t st) {
  // warp rows when a (sequence, kv head) averages at most 24 partials (one
  // chunk of the warp merge); blocks of kMergeWarps warps per row slice
  // otherwise
  const int64_t rows = (int64_t)a.B * a.Hq, units = (int64_t)a.B * a.H;
  const cudaError_t e =
      merge_by_warps(a.nw_launch, units)
          ? launch_maybe_dependent(attn_merge_warp_kernel, dim3((unsigned)((rows + 3) / 4)), dim3(128), 0, st, a.pdl, a)
          : launch_maybe_dependent(attn_merge_wide_kernel, dim3((unsigned)(rows * a.merge_slices)), dim3(kMergeWarps * 32), 0,
                                   st, a.pdl, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace tq
