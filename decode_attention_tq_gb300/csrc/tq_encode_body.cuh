// tq_encode_body.cuh -- device code of the encode (append): the per-warp
// encode body (sign flips, H_4 (x) H_32 rotation on the tensor cores,
// one-compare quantizer, packing, QJL sketch) and the code-stream helpers the
// decode kernel shares.  Included by the encode kernels and by the fused
// append kernels.
#pragma once

#include "tq_internal.cuh"
#include "tq_umma.cuh"

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

// Chunks 2q and 2q+1 of a token (4*BITS bytes of its stream) in a grouped
// value-code section whose chunks are whole (3-bit codes: 6-byte chunks,
// 4-byte aligned for even page offsets, 2 bytes past that for odd ones).
template <int BITS>
__device__ __forceinline__ void load_codes_grouped(const uint8_t *sec, int64_t off, int q, uint32_t (&w)[BITS]) {
  static_assert(BITS == 3, "2- and 4-bit value codes are pair-interleaved (load_codes_pair)");
  const uint16_t *h0 = reinterpret_cast<const uint16_t *>(sec + value_chunk_offset(off, 2 * q, BITS));
  const uint16_t *h1 = reinterpret_cast<const uint16_t *>(sec + value_chunk_offset(off, 2 * q + 1, BITS));
  w[0] = (uint32_t)h0[0] | ((uint32_t)h0[1] << 16);
  w[1] = (uint32_t)h0[2] | ((uint32_t)h1[0] << 16);
  w[2] = (uint32_t)h1[1] | ((uint32_t)h1[2] << 16);
}

// Pair-interleaved value codes (value_pairs_interleaved): the bits of a
// 32-bit word of the pair's even- or odd-coordinate stream that belong to
// the token at offset parity m.
template <int BITS>
__host__ __device__ constexpr uint32_t pair_mask(int m) {
  constexpr uint32_t lo = BITS == 4 ? 0x0F0F0F0Fu : 0x33333333u;
  return m ? ~lo : lo;
}
// Word i of a token's own chunk stream (16 coordinates, LSB-first) from words
// i of the pair's even (E) and odd (O) coordinate streams.
template <int BITS>
__device__ __forceinline__ uint32_t pair_split(uint32_t E, uint32_t O, int m) {
  constexpr uint32_t lo = pair_mask<BITS>(0);
  return m ? (((E >> BITS) & lo) | (O & ~lo)) : ((E & lo) | ((O & lo) << BITS));
}
// The inverse: a token's chunk-stream word T to its bits of E and O.
template <int BITS>
__device__ __forceinline__ void pair_merge(uint32_t T, int m, uint32_t &e, uint32_t &o) {
  constexpr uint32_t lo = pair_mask<BITS>(0);
  e = m ? ((T << BITS) & ~lo) : (T & lo);
  o = m ? (T & ~lo) : ((T >> BITS) & lo);
}

// Chunks 2q and 2q+1 of the token at page offset `off` (4*BITS bytes of its
// own stream) from a pair-interleaved value-code section.
template <int BITS>
__device__ __forceinline__ void load_codes_pair(const uint8_t *sec, int64_t off, int q, uint32_t (&w)[BITS]) {
  const int m = (int)(off & 1);
#pragma unroll
  for (int i = 0; i < 2; i++) {
    const uint8_t *pr = sec + value_chunk_offset(off & ~(int64_t)1, 2 * q + i, BITS);
    if constexpr (BITS == 4) {
      const uint4 x = *reinterpret_cast<const uint4 *>(pr);  // E0 E1 O0 O1
      w[2 * i] = pair_split<4>(x.x, x.z, m);
      w[2 * i + 1] = pair_split<4>(x.y, x.w, m);
    } else {
      const uint2 x = *reinterpret_cast<const uint2 *>(pr);  // E O
      w[i] = pair_split<2>(x.x, x.y, m);
    }
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

// QJL matrix for the encode projection on the tensor cores: S split into
// fp16 hi and lo parts, one 16-byte cell per (row l, lane slice t, k-step ks)
// holding S[l][32t+4ks .. 32t+4ks+3] as {hi pair, hi pair, lo pair, lo pair};
// the cell position inside its 128-byte row is XOR-swizzled by (t, l&1) so
// the 8 lanes of each load phase read 8 different bank groups.
__device__ __forceinline__ int sq_cell(int l, int t, int ks) { return (l * 4 + t) * 8 + (ks ^ (t + 4 * (l & 1))); }

// Quantizer lookup.  Bucket k = 48 + round(4u) covers 4u in [k-48.5, k-47.5]
// (both ends closed); since |u| <= sqrt(d) (||u||^2 = d), k stays in [2, 94].
// Entry k = (number of thresholds below the bucket, the single threshold
// inside it or +inf), so idx = #{t <= u} = base + [u >= thr] exactly, as long
// as no bucket holds two thresholds (checked when the table is built; the
// binary search is used otherwise).
constexpr int kQBuckets = 96;
constexpr float kQMagic = 12582912.0f + 48.0f;  // 1.5 * 2^23: the integer part lands in the low mantissa bits

__device__ __forceinline__ int quant_bucket(float u) {
  return __float_as_int(fmaf(u, 4.0f, kQMagic)) - __float_as_int(12582912.0f);
}

// Encode layout.  A warp encodes 8 vectors; thread (g, t) = (lane/4, lane%4)
// holds vector g at coordinates 32c + 8t + i (block c = 0..3, i = 0..7).
// With i = 32c + b the Sylvester matrix factors as H_128 = H_4 (x) H_32, so
// the transform is one tensor-core product per block (z = x_c H_32, rows of
// the A operand are (vector g, block 2m) and (vector g, block 2m+1)) and a
// 4-point butterfly across the blocks a thread already holds.  The k and n
// indices of the MMA are permuted so that a thread's operand words are its
// own loaded fp16 pairs and its outputs are again coordinates 8t .. 8t+7.
//   k (per k-step ks): 2t+e -> 8t+4ks+e, 2t+8+e -> 8t+4ks+2+e
//   n (per n-tile nt): 8nt+2t'+e -> 8t'+2nt+e
__device__ __forceinline__ uint32_t had_pair(int i0, int i1, int j) {
  // fp16 pair (H32[i0][j], H32[i1][j]) of the unnormalized Sylvester matrix
  const uint32_t s0 = (uint32_t)(__popc(i0 & j) & 1) << 15, s1 = (uint32_t)(__popc(i1 & j) & 1) << 31;
  return 0x3C003C00u | s0 | s1;
}

// Blocks per SM of the 4-bit encode without QJL (80 registers a thread).
// Measured: 2 blocks (128 registers, no spills) 0.330 of the HBM peak
// against 0.342 with 3.
constexpr int kEncodeBlocks4 = 3;
// MIXED (keys at a fractional rate): BITS is the width of the high channels
// (j mod 16 < 8), BITS - 1 that of the others; the codebook argument holds
// the BITS-bit device codebook, then the (BITS - 1)-bit one.  The quad lanes
// q = 0, 2 hold high channels (32c + 8q + i), q = 1, 3 low ones, so each lane
// quantizes with one codebook set: set 0 (high) or set 1 (low).
//
// The encode runs in three parts: encode_tables_load (global loads of the
// codebook and sign flips into shared memory; the kernels with a QJL sketch
// also stage S, as hi/lo cells or as tcgen05 operand tiles), then after a
// block barrier encode_tables_build (the quantizer's bucket table), then
// after another barrier encode_loop (the vectors).  A kernel
// that encodes two kinds keeps two table sets and overlaps their loads.
template <bool MIXED>
struct EncodeTables {
  static constexpr int NSET = MIXED ? 2 : 1;
  float cent[NSET * 16];
  float mid[NSET * 16];
  uint32_t dsign[4];
  uint2 qlut[NSET * kQBuckets];
  float2 qcen[NSET * kQBuckets];  // centroids of codes base and base+1 (QJL residual)
  int lut_bad;                    // bit per set
};

// Table loads by the 128 threads i = 0..127 (whole warps) of a block.
template <int BITS, bool MIXED>
__device__ __forceinline__ void encode_tables_load(EncodeTables<MIXED> &T, const EncodeArgs &a, int i) {
  constexpr int L = 1 << BITS;
  if (i < L) T.cent[i] = a.codebook[i];
  if (i < L - 1) T.mid[i] = a.codebook[L + i];
  if constexpr (MIXED) {
    const float *cb_lo = a.codebook + 2 * L - 1;
    if (i < L / 2) T.cent[16 + i] = cb_lo[i];
    if (i < L / 2 - 1) T.mid[16 + i] = cb_lo[L / 2 + i];
  }
  if (i == 0) T.lut_bad = 0;
  // sign words: one load per coordinate, packed by a ballot
  const uint32_t w = __ballot_sync(0xffffffffu, a.signs[i] != 0);
  if ((i & 31) == 0) T.dsign[i >> 5] = w;
}

// QJL: the matrix S staged as fp16 hi/lo cells in dynamic shared memory, by
// every thread of the block.
// cell (l, t, ks) holds S[l][32(ks/2) + 8t + 4(ks%2) + 0..3]: the
// coordinates thread t contributes at k-step ks of the projection.  Four
// consecutive coordinates share a cell: float4 loads, sixteen per thread in
// flight (all of them for 256 threads: one memory latency), and one 8-byte
// store each for the hi and lo halves.
constexpr int kSCellBatch = 16;
__device__ __forceinline__ void encode_s_batch_load(const EncodeArgs &a, int i0, float4 (&v)[kSCellBatch]) {
  constexpr int N4 = kM * kD / 4;
  const float4 *S4 = reinterpret_cast<const float4 *>(a.S);
#pragma unroll
  for (int u = 0; u < kSCellBatch; u++) {
    const int i4 = i0 + u * blockDim.x;
    v[u] = i4 < N4 ? __ldg(S4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}
__device__ __forceinline__ void encode_s_batch_store(int i0, const float4 (&v)[kSCellBatch]) {
  extern __shared__ __align__(16) uint4 s_Sq[];  // [m][4][8] cells
  constexpr int N4 = kM * kD / 4;
  uint2 *cells = reinterpret_cast<uint2 *>(s_Sq);
#pragma unroll
  for (int u = 0; u < kSCellBatch; u++) {
    const int i4 = i0 + u * blockDim.x;
    if (i4 < N4) {
      const int l = (4 * i4) / kD, j = (4 * i4) % kD;
      __half h0, l0, h1, l1, h2, l2, h3, l3;
      split_half(v[u].x, h0, l0);
      split_half(v[u].y, h1, l1);
      split_half(v[u].z, h2, l2);
      split_half(v[u].w, h3, l3);
      const int cell = sq_cell(l, (j & 31) >> 3, 2 * (j >> 5) + ((j >> 2) & 1));
      cells[2 * cell] = make_uint2(pack_half2_raw(h0, h1), pack_half2_raw(h2, h3));
      cells[2 * cell + 1] = make_uint2(pack_half2_raw(l0, l1), pack_half2_raw(l2, l3));
    }
  }
}

// Quantizer bucket table from the loaded codebook (every thread of the block).
template <int BITS, bool MIXED>
__device__ __forceinline__ void encode_tables_build(EncodeTables<MIXED> &T) {
  constexpr int L = 1 << BITS;
  for (int e = threadIdx.x; e < EncodeTables<MIXED>::NSET * kQBuckets; e += blockDim.x) {
    const int set = e / kQBuckets, bk = e % kQBuckets, Ls = set ? L / 2 : L;
    const float *mid = T.mid + 16 * set, *cen = T.cent + 16 * set;
    const float lo = ((float)(bk - 48) - 0.5f) * 0.25f, hi = ((float)(bk - 48) + 0.5f) * 0.25f;
    int base = 0, inside = 0;
    float thr = __int_as_float(0x7f800000);  // +inf
    for (int k = 0; k < Ls - 1; k++) {
      const float t = mid[k];
      if (t < lo) base++;
      else if (t <= hi) { thr = t; inside++; }
    }
    if (inside > 1 || (bk == 0 && base > 0) || (bk == kQBuckets - 1 && inside + base < Ls - 1))
      atomicOr(&T.lut_bad, 1 << set);
    T.qlut[set * kQBuckets + bk] = make_uint2((uint32_t)base, __float_as_uint(thr));
    T.qcen[set * kQBuckets + bk] = make_float2(cen[base], cen[base + 1 < Ls ? base + 1 : base]);
  }
}

// ------------------------------------------------ QJL sketch on tcgen05 --
// The bulk key encode with QJL computes the sketch products (S e)_l of a
// batch of 128 vectors as one 128 x 128 x 128 contraction on the tensor cores:
// D[v][l] = sum_j e_v[j] S[l][j], A = the residuals (rows = vectors), B = S
// (rows = l), both fp16 hi/lo split in shared memory (K-major, 128-byte
// swizzle: two 16 KB column blocks of 64 coordinates per 128-row tile), the
// fp32 accumulator in tensor memory.  Three products (hi.hi, lo.hi, hi.lo)
// give the same precision as the register path (the lo.lo term, ~2^-22 of
// the product, is left out).  A CTA of 16 warps encodes 128 vectors per
// iteration (8 per warp); warp w's vector g is row umma_row(w, g), which
// puts the two vectors of every 8-lane store phase 4 rows apart (so their
// swizzled chunks fall in different banks).  Batch t's MMAs are issued by
// lane 0 of the last warp to finish its rows of residual buffer t&1 (so
// that no thread waits for the others) into accumulator t mod 3, and run
// while the warps encode batches t+1 and t+2.  In iteration t+2 each warp
// waits for them (their residual buffer is then free again) and reads batch
// t's sign words back: the warps of a block may drift up to two batches
// apart before one waits.
constexpr int kUmmaThreads = 512;
constexpr int kUmmaRows = 128;                         // vectors per batch (MMA M)
constexpr uint32_t kUmmaTile = 32768;                  // one 128 x 128 fp16 operand tile
constexpr uint32_t kUmmaDynSmem = 6 * kUmmaTile + 1024;  // S hi/lo, 2 x residual hi/lo, alignment
constexpr uint32_t kUmmaTmemCols = 512;                // 3 accumulators of 128 fp32 columns (a power of 2)
constexpr int kUmmaInfoRing = 8;                       // batches of sign-word addresses kept
constexpr uint64_t kUmmaWaitNs = 1000000000ull;        // bounded waits: one second

__device__ __forceinline__ int umma_row(int warp_in_block, int g) { return 8 * warp_in_block + ((g >> 1) | ((g & 1) << 2)); }

// Byte offset of coordinates j .. j+7 (j a multiple of 8) of row r inside a
// 128 x 128 fp16 tile: column block j / 64, chunk (j mod 64) / 8 swizzled by r.
__device__ __forceinline__ uint32_t umma_tile_off(int r, int j) {
  return (uint32_t)((j >> 6) * 16384 + r * 128 + ((((j & 63) >> 3) ^ (r & 7)) << 4));
}

struct UmmaQjl {
  uint32_t s_tiles;   // S hi at +0, S lo at +kUmmaTile (shared-window address)
  uint32_t r_tiles;   // residual buffer b at +2 kUmmaTile b: hi at +0, lo at +kUmmaTile
  uint8_t *r_ptr;     // generic pointer of r_tiles
  uint64_t *info;     // [kUmmaInfoRing][128]: sign-word address of each row | 1 for a zero
                      // vector; 0 = not stored
  uint32_t mbar;      // two mbarriers, 8 bytes apart: done(b) = mbar + 8 b, the MMAs
                      // reading residual buffer b completed (tcgen05.commit)
  unsigned *count;    // [2]: warps that have written their rows of buffer b (a running
                      // count; the warp that makes it a multiple of 16 issues the MMAs)
  __device__ __forceinline__ uint32_t done(int b) const { return mbar + 8u * (uint32_t)b; }
  uint32_t tmem;      // accumulator base: batch t at column 128 (t mod 3)
  int *abort;         // set when a bounded wait ran out; every warp then stops
};

// S as fp16 hi/lo B-operand tiles (every thread of the block).
__device__ __forceinline__ void umma_s_tiles_load(const EncodeArgs &a, uint8_t *tiles) {
  constexpr int N4 = kM * kD / 4;
  const float4 *S4 = reinterpret_cast<const float4 *>(a.S);
  for (int i0 = threadIdx.x; i0 < N4; i0 += 8 * blockDim.x) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int i4 = i0 + u * blockDim.x;
      v[u] = i4 < N4 ? __ldg(S4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int i4 = i0 + u * blockDim.x;
      if (i4 < N4) {
        const int l = i4 / (kD / 4), j = 4 * (i4 % (kD / 4));
        __half h0, l0, h1, l1, h2, l2, h3, l3;
        split_half(v[u].x, h0, l0);
        split_half(v[u].y, h1, l1);
        split_half(v[u].z, h2, l2);
        split_half(v[u].w, h3, l3);
        const uint32_t o = umma_tile_off(l, j & ~7) + 2 * (j & 7);
        *reinterpret_cast<uint2 *>(tiles + o) = make_uint2(pack_half2_raw(h0, h1), pack_half2_raw(h2, h3));
        *reinterpret_cast<uint2 *>(tiles + kUmmaTile + o) = make_uint2(pack_half2_raw(l0, l1), pack_half2_raw(l2, l3));
      }
    }
  }
}

__device__ __forceinline__ uint32_t umma_acc_col(int64_t t) { return 128u * (uint32_t)(t % 3); }

// The 24 MMAs of batch t (K = 128 in 8 steps of 16, three hi/lo products),
// then the commit that arrives on done(t & 1).  One thread.
__device__ __forceinline__ void umma_qjl_issue(const UmmaQjl &U, int64_t t) {
  constexpr uint32_t idesc = umma::idesc_f16_f32<kUmmaRows, kM>();
  const int buf = (int)(t & 1);
  const uint32_t d = U.tmem + umma_acc_col(t);
  const uint32_t ra = U.r_tiles + 2u * kUmmaTile * (uint32_t)buf;
#pragma unroll
  for (int part = 0; part < 3; part++) {
    const uint32_t a0 = ra + (part == 1 ? kUmmaTile : 0u);           // e hi, e lo, e hi
    const uint32_t b0 = U.s_tiles + (part == 2 ? kUmmaTile : 0u);    // S hi, S hi, S lo
#pragma unroll
    for (int ks = 0; ks < 8; ks++) {
      const uint32_t ko = (uint32_t)((ks >> 2) * 16384 + (ks & 3) * 32);  // 16 coordinates = 32 bytes
      umma::mma_f16_ss(d, umma::desc_sw128_kmajor(a0 + ko), umma::desc_sw128_kmajor(b0 + ko), idesc,
                       (part | ks) ? 1u : 0u);
    }
  }
  umma::commit(U.done(buf));
}

// Waits until batch t's MMAs have completed (its residual buffer is free and
// its accumulator ready).  Warp-uniform; false when the wait ran out here or
// another warp had already given up.
__device__ __forceinline__ bool umma_qjl_wait(const UmmaQjl &U, int64_t t, int32_t *err_word) {
  bool ok = *reinterpret_cast<volatile int *>(U.abort) == 0;
  if (ok && !umma::mbar_wait_bounded(U.done((int)(t & 1)), (uint32_t)((t >> 1) & 1), kUmmaWaitNs)) {
    *reinterpret_cast<volatile int *>(U.abort) = 1;
    report(err_word, TQ_DEVERR_TIMEOUT);
    ok = false;
  }
  ok = __all_sync(0xffffffffu, ok);
  if (ok) umma::fence_after_sync();
  return ok;
}

// Sign words of batch t (after umma_qjl_wait): warp w reads accumulator
// lanes 32 (w mod 4) .. +31 (its sub-partition: one row = one vector per
// thread) and columns 32 (w / 4) .. +31, i.e. sign word w / 4 of each of its
// 32 vectors: bit i is [(S e)_{32 (w/4) + i} >= 0], gathered MSB first by
// funnel shifts of the fp32 sign bits and inverted.
__device__ __forceinline__ void umma_qjl_signs(const UmmaQjl &U, int64_t t) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t v[32];
  umma::ld_32x32b_x32(U.tmem + ((uint32_t)(32 * (w & 3)) << 16) + umma_acc_col(t) + 32u * (uint32_t)(w >> 2), v);
  uint32_t neg = 0u;
#pragma unroll
  for (int i = 31; i >= 0; i--) neg = __funnelshift_l(v[i], neg, 1);
  const uint64_t inf = U.info[(t & (kUmmaInfoRing - 1)) * kUmmaRows + 32 * (w & 3) + lane];
  if (inf) reinterpret_cast<uint32_t *>(inf & ~(uint64_t)1)[w >> 2] = (inf & 1) ? 0u : ~neg;
  umma::fence_before_sync();
}

// The vectors [n_tokens][H] of a.x (global or shared memory), 8 per warp and
// step: warps [warp0, warp0 + nwarps) of the grid share them (a grid-stride
// loop); the default is every warp of the grid.
// part / parts (QJL): several warps encoding the same vectors (a batch that
// fills fewer octets than there are warps) share the projection: this warp
// computes n-tiles [16 part / parts, 16 (part + 1) / parts) and stores only
// the sign words they fill; part 0 stores codes, norm and gamma.
// UMMA (QJL, a block of kUmmaThreads, the default warp range): the
// projection runs on tcgen05 through U (see UmmaQjl); every warp of the block
// runs the same number of iterations (whole batches of 128 vectors).
template <int BITS, bool QJL, bool MIXED = false, bool UMMA = false>
__device__ __forceinline__ void encode_loop(const EncodeTables<MIXED> &T, const EncodeArgs &a, int64_t warp0 = -1,
                                            int64_t nwarps_in = 0, int part = 0, int parts = 1,
                                            const UmmaQjl *U = nullptr) {
  static_assert(!UMMA || QJL, "the tensor-core path is the QJL projection");
  extern __shared__ __align__(16) uint4 s_Sq[];  // QJL only
  constexpr int L = 1 << BITS;
  const int tid = threadIdx.x;
  const int lane = tid & 31, q = lane & 3, quad_in_warp = lane >> 2;
  const int64_t warp = warp0 >= 0 ? warp0 : (int64_t)((blockIdx.x * blockDim.x + tid) >> 5);
  const int64_t nwarps = warp0 >= 0 ? nwarps_in : (int64_t)gridDim.x * blockDim.x / 32;
  const int64_t NH = a.n_tokens * a.H;
  const int64_t pool_slots = a.num_pages * (int64_t)a.P;
  // this lane's codebook set (mixed keys: odd quad lanes hold low channels)
  const int set = MIXED ? (q & 1) : 0;
  const float *cent = T.cent + 16 * set, *midp = T.mid + 16 * set;
  const uint2 *qlut = T.qlut + set * kQBuckets;
  // shared-window addresses of the bucket tables, offset so that the bucket
  // entry of the magic-number sum s (quant_bucket) is at base + 8 * bits(s)
  // (one shift-add per coordinate; the sums wrap mod 2^32 as addresses do)
  const uint32_t kMagicBits = (uint32_t)__float_as_int(12582912.0f);
  // (the centroid pairs qcen follow qlut: the same entry is kQcenOff bytes on)
  const uint32_t qlut_at = (uint32_t)__cvta_generic_to_shared(qlut) - 8u * kMagicBits;
  constexpr int kQcenOff = (int)(sizeof(uint2) * EncodeTables<MIXED>::NSET * kQBuckets);
  static_assert(offsetof(EncodeTables<MIXED>, qcen) - offsetof(EncodeTables<MIXED>, qlut) == kQcenOff,
                "qcen directly after qlut");
  const bool lut_bad = (T.lut_bad >> set) & 1;
  const bool small = NH <= 0x7fffffff;
  // sign masks of this thread's fp16 pairs (coordinates 32c + 8q + 2p, +1)
  uint32_t smask[4][4];
#pragma unroll
  for (int c = 0; c < 4; c++) {
    const uint32_t byte = (T.dsign[c] >> (8 * q)) & 0xFFu;
#pragma unroll
    for (int p = 0; p < 4; p++) smask[c][p] = ((byte >> (2 * p)) & 1u) << 15 | ((byte >> (2 * p + 1)) & 1u) << 31;
  }
  // B fragments of H_32 (k and n permuted as above), constant over the loop
  uint32_t hb[2][4][2];
#pragma unroll
  for (int ks = 0; ks < 2; ks++)
#pragma unroll
    for (int nt = 0; nt < 4; nt++) {
      const int j = 8 * (quad_in_warp >> 1) + 2 * nt + (quad_in_warp & 1);  // permuted column of n = 8nt + g
      hb[ks][nt][0] = had_pair(8 * q + 4 * ks, 8 * q + 4 * ks + 1, j);
      hb[ks][nt][1] = had_pair(8 * q + 4 * ks + 2, 8 * q + 4 * ks + 3, j);
    }

  // Pair-interleaved value codes: vectors in pair-major order, quads 2i and
  // 2i+1 of a warp holding tokens 2k and 2k+1 of one head, so that the two
  // tokens of an offset pair, where they come in order, sit in neighbouring
  // quads and one of them writes the words they share.
  constexpr bool kPairCodes = !MIXED && value_pairs_interleaved(BITS);
  const bool pairs = kPairCodes && a.grouped;
  const int64_t NV = pairs ? ((a.n_tokens + 1) & ~(int64_t)1) * a.H : NH;
  int64_t t = 0;  // iteration (UMMA: batch of the block)
  for (int64_t vb = (int64_t)warp * 8; (UMMA ? (vb & ~(int64_t)(kUmmaRows - 1)) : vb) < NV; vb += nwarps * 8, t++) {
    if constexpr (UMMA) {
      if (__any_sync(0xffffffffu, *reinterpret_cast<volatile int *>(U->abort) != 0)) break;
    }
    const int64_t v = vb + quad_in_warp;
    int64_t n;
    int h;
    bool in_range;
    if (pairs) {
      const int64_t H2 = 2 * (int64_t)a.H;
      const int64_t k = small ? (int64_t)((uint32_t)v / (uint32_t)H2) : v / H2;
      const int rem = (int)(v - k * H2);
      n = 2 * k + (rem & 1);
      h = rem >> 1;
      in_range = n < a.n_tokens;
      if (!in_range) n = a.n_tokens - 1;
    } else {
      in_range = v < NH;
      const int64_t vc = in_range ? v : NH - 1;
      if (small) {  // 32-bit division for the common sizes
        n = (uint32_t)vc / (uint32_t)a.H;
        h = (int)((uint32_t)vc - (uint32_t)n * (uint32_t)a.H);
      } else {
        n = vc / a.H;
        h = (int)(vc % a.H);
      }
    }
    const int64_t vv = n * a.H + h;
    const int64_t slot = a.slot_mapping[n];
    bool ok = in_range && slot >= 0;
    if (ok && slot >= pool_slots) {
      if (q == 0) report(a.err_word, TQ_DEVERR_SLOT_RANGE);
      ok = false;
    }

    // fp16 pairs of coordinates 32c + 8q + 2p, +1, sign-flipped by D
    uint32_t xw[4][4];
#pragma unroll
    for (int c = 0; c < 4; c++) {
      const uint4 raw = *reinterpret_cast<const uint4 *>(a.x + vv * kD + 32 * c + 8 * q);
      const uint32_t r4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int p = 0; p < 4; p++) xw[c][p] = r4[p] ^ smask[c][p];
    }

    // z = x_c H_32 on the tensor cores, then the H_4 butterfly over blocks
    float z[4][8];
#pragma unroll
    for (int mt = 0; mt < 2; mt++)
#pragma unroll
      for (int nt = 0; nt < 4; nt++) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(d, xw[2 * mt][0], xw[2 * mt + 1][0], xw[2 * mt][1], xw[2 * mt + 1][1], hb[0][nt][0], hb[0][nt][1]);
        mma_16816(d, xw[2 * mt][2], xw[2 * mt + 1][2], xw[2 * mt][3], xw[2 * mt + 1][3], hb[1][nt][0], hb[1][nt][1]);
        z[2 * mt][2 * nt] = d[0];
        z[2 * mt][2 * nt + 1] = d[1];
        z[2 * mt + 1][2 * nt] = d[2];
        z[2 * mt + 1][2 * nt + 1] = d[3];
      }
    float x[32];  // x[8c + i]: coordinate 32c + 8q + i of H (D . x)
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const float s01 = z[0][i] + z[1][i], d01 = z[0][i] - z[1][i];
      const float s23 = z[2][i] + z[3][i], d23 = z[2][i] - z[3][i];
      x[i] = s01 + s23;
      x[8 + i] = d01 + d23;
      x[16 + i] = s01 - s23;
      x[24 + i] = d01 - d23;
    }
    // ||x||^2 from the rotated coordinates (||H y||^2 = d ||y||^2 for the
    // unnormalised Sylvester H; the products of the transform are exact).
    // A NaN or infinite coordinate (finite fp16 vectors cannot overflow ss)
    // stores the norm as computed and a zero block, and never reaches the
    // quantizer's bucket table with a NaN.
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 32; j++) ss = fmaf(x[j], x[j], ss);
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    ss *= 1.0f / (float)kD;
    const float nrm = sqrtf(ss);
    const bool bad = !(ss <= 3.0e38f);
    const bool zero = !(nrm > 0.f) || bad;
    if (bad) {
#pragma unroll
      for (int j = 0; j < 32; j++) x[j] = 0.f;
    }
    const float inv = zero ? 0.f : 1.0f / nrm;

    int idx[32];
    if (!lut_bad) {
#pragma unroll
      for (int j = 0; j < 32; j++) {
        const float u = x[j] * inv;
        const uint32_t sb = (uint32_t)__float_as_int(fmaf(u, 4.0f, kQMagic)) << 3;  // 8 x bits of quant_bucket's sum
        uint2 e;
        asm("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(e.x), "=r"(e.y) : "r"(qlut_at + sb));
        const bool up = u >= __uint_as_float(e.y);
        idx[j] = (int)e.x + (up ? 1 : 0);  // a zero vector's codes are cleared when packed
        if constexpr (QJL) {
          float2 c;
          asm("ld.shared.v2.f32 {%0,%1}, [%2+%3];" : "=f"(c.x), "=f"(c.y) : "r"(qlut_at + sb), "n"(kQcenOff));
          x[j] = u - (up ? c.y : c.x);  // residual in u units (unused for a zero vector: gamma, bits 0)
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; j++) {
        const float u = x[j] * inv;
        int k = 0;
        const int Lq = set ? L / 2 : L;
        for (int s = Lq / 2; s >= 1; s >>= 1)
          if (u >= midp[k + s - 1]) k += s;
        idx[j] = zero ? 0 : k;
        x[j] = u - cent[idx[j]];  // residual in u units (QJL only)
      }
    }

    // Norm correction (no QJL): store n / ||y_hat|| with y_hat = c[idx] / sqrt(d),
    // i.e. n sqrt(d) / ||c[idx]||, so that the reconstruction keeps ||x||.
    float nstore = nrm;
    if (!QJL && a.norm_correct) {
      float c2 = 0.f;
#pragma unroll
      for (int j = 0; j < 32; j++) {
        const float cj = cent[idx[j]];
        c2 = fmaf(cj, cj, c2);
      }
      c2 += __shfl_xor_sync(0xffffffffu, c2, 1);
      c2 += __shfl_xor_sync(0xffffffffu, c2, 2);
      nstore = (zero || !(c2 > 0.f)) ? nrm : nrm * 11.313708498984761f / sqrtf(c2);
    }

    const int64_t page = ok ? slot / a.P : 0;
    const int64_t off = ok ? slot % a.P : 0;
    uint8_t *slab = a.pool + page * a.page_bytes + (int64_t)h * a.slab_bytes;
    const bool okc = ok && part == 0;  // this warp stores the codes and the norm
    if (MIXED && okc) {
      // high stream (channels j mod 16 < 8) at BITS bits, then the low stream
      // at BITS - 1: this lane's 8 codes of block c are group 2c + q/2 of its
      // stream
      const int W = set ? BITS - 1 : BITS;
      uint8_t *tok = slab + a.codes_off + off * a.code_bytes;
#pragma unroll
      for (int c = 0; c < 4; c++) {
        uint32_t w = 0u;
#pragma unroll
        for (int i = 0; i < 8; i++) w |= (uint32_t)idx[8 * c + i] << (W * i);
        if (zero) w = 0u;
        const int g = 2 * c + (q >> 1);
        uint8_t *dst = set ? tok + 8 * BITS + g * (BITS - 1) : tok + g * BITS;
        if (W == 4) {
          *reinterpret_cast<uint32_t *>(dst) = w;
        } else if (W == 2) {
          *reinterpret_cast<uint16_t *>(dst) = (uint16_t)w;
        } else {
          dst[0] = (uint8_t)w;
          dst[1] = (uint8_t)(w >> 8);
          dst[2] = (uint8_t)(w >> 16);
        }
      }
      if (q == 0) reinterpret_cast<float *>(slab + a.norm_off)[off] = nstore;
    } else if (kPairCodes && pairs) {
      // this lane's 8 codes of block c are half q&1 of chunk 2c + q/2, i.e.
      // BITS bytes at byte (q&1)*BITS of each of the pair's two streams.  The
      // offset partner in the neighbouring quad: the even-offset token writes
      // both tokens' words; otherwise each token sets its own bits atomically
      // (its partner may be written by another warp of this launch).
      const int64_t pslot = __shfl_xor_sync(0xffffffffu, ok ? slot : (int64_t)-1, 4);
      const bool paired = ok && pslot == (slot ^ 1);
      const int m = (int)(off & 1), hq = q & 1;
#pragma unroll
      for (int c = 0; c < 4; c++) {
        uint32_t w = 0u;
#pragma unroll
        for (int i = 0; i < 8; i++) w += (uint32_t)idx[8 * c + i] << (BITS * i);
        if (zero) w = 0u;
        uint32_t e, o;
        pair_merge<BITS>(BITS == 4 ? w : w << (16 * hq), m, e, o);
        const uint32_t pe = __shfl_xor_sync(0xffffffffu, e, 4), po = __shfl_xor_sync(0xffffffffu, o, 4);
        uint8_t *pr = slab + a.codes_off + value_chunk_offset(off & ~(int64_t)1, 2 * c + (q >> 1), BITS);
        if (paired) {
          if (m == 0) {
            if constexpr (BITS == 4) {
              reinterpret_cast<uint32_t *>(pr)[hq] = e | pe;
              reinterpret_cast<uint32_t *>(pr + 8)[hq] = o | po;
            } else {
              reinterpret_cast<uint16_t *>(pr)[hq] = (uint16_t)((e | pe) >> (16 * hq));
              reinterpret_cast<uint16_t *>(pr + 4)[hq] = (uint16_t)((o | po) >> (16 * hq));
            }
          }
        } else if (ok) {
          unsigned *E = reinterpret_cast<unsigned *>(pr + (BITS == 4 ? 4 * hq : 0));
          unsigned *O = reinterpret_cast<unsigned *>(pr + 2 * BITS + (BITS == 4 ? 4 * hq : 0));
          const uint32_t own = pair_mask<BITS>(m) & (BITS == 4 ? 0xFFFFFFFFu : 0xFFFFu << (16 * hq));
          atomicAnd(E, ~own);
          atomicOr(E, e);
          atomicAnd(O, ~own);
          atomicOr(O, o);
        }
      }
      if (ok && q == 0) reinterpret_cast<float *>(slab + a.norm_off)[off] = nstore;
    } else if (okc) {
#pragma unroll
      for (int c = 0; c < 4; c++) {
        // codes of coordinates 32c + 8q .. +7: 8 * BITS bits, LSB first
        uint32_t w = 0u;
#pragma unroll
        for (int i = 0; i < 8; i++) w += (uint32_t)idx[8 * c + i] << (BITS * i);  // disjoint fields: + is |
        if (zero) w = 0u;
        uint8_t *dst = a.grouped ? slab + a.codes_off + value_chunk_offset(off, 2 * c + (q >> 1), BITS) + (q & 1) * BITS
                                 : slab + a.codes_off + off * a.code_bytes + c * 4 * BITS + q * BITS;
        if constexpr (BITS == 4) {
          *reinterpret_cast<uint32_t *>(dst) = w;
        } else if constexpr (BITS == 2) {
          *reinterpret_cast<uint16_t *>(dst) = (uint16_t)w;
        } else if (!a.grouped) {
          // the quad's 4 x 3 bytes are 12 contiguous bytes: lanes 0..2 write
          // one aligned word each, taking the neighbour's bytes by a shuffle
          const uint32_t wn = __shfl_down_sync(0xfu << (lane & ~3), w, 1, 4);
          if (q < 3) *reinterpret_cast<uint32_t *>(dst - q * BITS + 4 * q) = (w >> (8 * q)) | (wn << (24 - 8 * q));
        } else {
          // a 6-byte chunk is lanes (2k, 2k+1): the even lane writes it,
          // 4-byte aligned for even page offsets, 2 bytes past that for odd
          const uint32_t wn = __shfl_xor_sync(0xfu << (lane & ~3), w, 1);
          if ((q & 1) == 0) {
            const uint32_t lo = w | (wn << 24), hi = wn >> 8;  // 48 bits: lo (4 bytes) then hi (2 bytes)
            if ((off & 1) == 0) {
              *reinterpret_cast<uint32_t *>(dst) = lo;
              *reinterpret_cast<uint16_t *>(dst + 4) = (uint16_t)hi;
            } else {
              *reinterpret_cast<uint16_t *>(dst) = (uint16_t)lo;
              *reinterpret_cast<uint32_t *>(dst + 2) = (lo >> 16) | (hi << 16);
            }
          }
        }
      }
      if (q == 0) reinterpret_cast<float *>(slab + a.norm_off)[off] = nstore;
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
      if constexpr (UMMA) {
        // batch t-2's MMAs done: its residual buffer is this batch's
        if (t >= 2 && !umma_qjl_wait(*U, t - 2, a.err_word)) break;
        // residual hi/lo into this batch's A tiles, row r; the sign-word
        // address (and the zero-vector flag) for the epilogue
        const int r = umma_row(tid >> 5, quad_in_warp);
        const int buf = (int)(t & 1);
        uint8_t *rt = U->r_ptr + 2 * kUmmaTile * buf;
#pragma unroll
        for (int c = 0; c < 4; c++) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int p = 0; p < 4; p++) {
            // split_half of a pair, with paired conversions
            const float x0 = x[8 * c + 2 * p], x1 = x[8 * c + 2 * p + 1];
            const __half2 h = __floats2half2_rn(x0, x1);
            const float2 hf = __half22float2(h);
            const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
            hw[p] = *reinterpret_cast<const uint32_t *>(&h);
            lw[p] = *reinterpret_cast<const uint32_t *>(&l);
          }
          const uint32_t o = umma_tile_off(r, 32 * c + 8 * q);
          *reinterpret_cast<uint4 *>(rt + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4 *>(rt + kUmmaTile + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        if (q == 0) {
          U->info[(t & (kUmmaInfoRing - 1)) * kUmmaRows + r] =
              ok ? ((uint64_t)(uintptr_t)(slab + a.signs_off + off * (kM / 8)) | (zero ? 1u : 0u)) : 0ull;
          if (ok) reinterpret_cast<float *>(slab + a.gamma_off)[off] = gamma;
        }
        // this warp's rows are written: the warp whose arrival completes the
        // batch issues its MMAs (release / acquire through the shared counter;
        // the proxy fence makes the rows visible to the tensor core's reads)
        umma::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          const unsigned before = atomicAdd(U->count + buf, 1u);
          if ((before & (kUmmaThreads / 32 - 1)) == kUmmaThreads / 32 - 1) {
            __threadfence_block();
            umma::fence_after_sync();
            umma_qjl_issue(*U, t);
          }
        }
        __syncwarp();
        if (t >= 2) umma_qjl_signs(*U, t - 2);
      } else {
      // (S e)_l on the tensor cores: rows g / g+8 of the A operand are the fp16
      // hi / lo parts of this quad's residual (vector g of the warp), B is
      // S hi then S lo, so the fp32 sum misses only the lo*lo term (~2^-22).
      // k-indices 2t, 2t+1 | 2t+8, 2t+9 of step ks are the coordinates
      // 32(ks/2) + 8t + 4(ks%2) + {0,1} | +{2,3}: x[4ks .. 4ks+3] of this lane.
      uint32_t A[8][4];
#pragma unroll
      for (int ks = 0; ks < 8; ks++) {
        __half h0, l0, h1, l1, h2, l2, h3, l3;
        split_half(x[4 * ks + 0], h0, l0);
        split_half(x[4 * ks + 1], h1, l1);
        split_half(x[4 * ks + 2], h2, l2);
        split_half(x[4 * ks + 3], h3, l3);
        A[ks][0] = pack_half2_raw(h0, h1);
        A[ks][1] = pack_half2_raw(l0, l1);
        A[ks][2] = pack_half2_raw(h2, h3);
        A[ks][3] = pack_half2_raw(l2, l3);
      }
      uint32_t words[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int nt = 0; nt < 16; nt++) {  // outputs l = 8nt .. 8nt+7; this lane gets 8nt+2q, 8nt+2q+1
        if (parts > 1 && (nt < 16 * part / parts || nt >= 16 * (part + 1) / parts)) continue;  // warp-uniform
        float dh[4] = {0.f, 0.f, 0.f, 0.f}, dl[4] = {0.f, 0.f, 0.f, 0.f};
        const int l = 8 * nt + quad_in_warp;
#pragma unroll
        for (int ks = 0; ks < 8; ks++) {
          const uint4 sv = s_Sq[sq_cell(l, q, ks)];
          mma_16816(dh, A[ks][0], A[ks][1], A[ks][2], A[ks][3], sv.x, sv.y);
          mma_16816(dl, A[ks][0], A[ks][1], A[ks][2], A[ks][3], sv.z, sv.w);
        }
        const float p0 = (dh[0] + dh[2]) + (dl[0] + dl[2]);
        const float p1 = (dh[1] + dh[3]) + (dl[1] + dl[3]);
        const int bit = 8 * (nt & 3) + 2 * q;
        words[nt >> 2] |= ((p0 >= 0.f ? 1u : 0u) << bit) | ((p1 >= 0.f ? 1u : 0u) << (bit + 1));
      }
#pragma unroll
      for (int k = 0; k < 4; k++) {
        words[k] |= __shfl_xor_sync(0xffffffffu, words[k], 1);
        words[k] |= __shfl_xor_sync(0xffffffffu, words[k], 2);
      }
      uint32_t word = q == 0 ? words[0] : q == 1 ? words[1] : q == 2 ? words[2] : words[3];
      if (zero) word = 0u;
      // word q holds n-tiles 4q .. 4q + 3: stored by the warp that computed them
      if (ok && (parts == 1 || (4 * q >= 16 * part / parts && 4 * q < 16 * (part + 1) / parts))) {
        reinterpret_cast<uint32_t *>(slab + a.signs_off + off * (kM / 8))[q] = word;
        if (q == 0) reinterpret_cast<float *>(slab + a.gamma_off)[off] = gamma;
      }
      }  // register path
    }
  }
  if constexpr (UMMA) {
    // the last two batches' sign words
    for (int64_t s = t >= 2 ? t - 2 : 0; s < t; s++)
      if (umma_qjl_wait(*U, s, a.err_word)) umma_qjl_signs(*U, s);
  }
}


// Load, build and loop in one call (kernels that encode one kind without a
// QJL sketch; keys with one run encode_qjl_kernel or the append).
template <int BITS, bool MIXED = false>
__device__ __forceinline__ void encode_body(const EncodeArgs &a, int64_t warp0 = -1, int64_t nwarps_in = 0) {
  __shared__ EncodeTables<MIXED> T;
  if (threadIdx.x < kD) encode_tables_load<BITS, MIXED>(T, a, threadIdx.x);
  __syncthreads();
  encode_tables_build<BITS, MIXED>(T);
  __syncthreads();
  encode_loop<BITS, false, MIXED>(T, a, warp0, nwarps_in);
}

}  // namespace tq
