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
// Per tile (16 tokens of one (b, h)) a warp runs, on the tensor cores
// (mma.sync m16n8k16, fp16 operands, fp32 accumulation):
//   scores[16 x 2G] = Kcodes[16 x 128] * Qrot[128 x 2G]
//     A: the fp16 centroids of each code pair from a shared-memory table (the
//        stored codebook is fp16-exact, so each is an exact operand); rows
//        are the 16 tokens of the tile, one 4-byte table read per register;
//        B: the rotated query, hi/lo split over the 2G columns, so the
//        product is exact to ~2^-22;
//   QJL (keys): + signs[16 x 128] * (S q_rot)[128 x 2G], the +-1 operands are
//        exact in fp16;
//   online softmax in fp32 (log2 domain);
//   acc[128 x G] += Vcodes^T[128 x 16] * W[16 x G], W = p_i * n_i / nu
//        (nu = running max value norm) in fp16.  One MMA takes 8 tokens and
//        32 coordinates, and column 4e + g of B holds head g's weights in
//        the rows of part e and zeros in the others, so the 8 columns carry
//        2 x 4 useful outputs, with no accumulator register for a zero
//        column.  The K index of an MMA is (token slot i, coordinate parity
//        e) for 3-bit values: an A register is one code pair of one token,
//        one table lookup.  For 2- and 4-bit values it is (coordinate half
//        e, token i): an A register pairs two tokens' codes at one
//        coordinate, interleaved in registers and looked up once.
// Thread (r = lane/4, t = lane%4) owns head 4*nt + t of n-tile nt and tokens r
// and r+8 of a tile for the scores; for the values it reads the codes of
// coordinates 16r..16r+15 of tokens 2t, 2t+1, 2t+8, 2t+9 and accumulates
// heads 4nt + 2(t&1) and 4nt + 2(t&1) + 1.
#pragma once

#include "tq_internal.cuh"

namespace tq {

// Key code widths.  KB = 2, 3, 4: every channel at KB bits.  KB = 34 or 23:
// mixed-rate keys ("TurboQuant Family Design Study ...", 'Packed format and
// complete bit accounting': 3.5 and 2.5 bits per channel), KB % 10 bits on
// the channels j with (j mod 16) < 8 and KB / 10 on the others; a token's
// stream holds the high channels' codes, then the low ones'.  Lane t's 32
// channels 32t..32t+31 are 16 of each: high codes 16t..16t+15 and low codes
// 16t..16t+15 of the two streams, used by the k-steps kk with (kk mod 4) < 2
// and >= 2 respectively.
__host__ __device__ constexpr bool kb_mixed(int KB) { return KB > 8; }
__host__ __device__ constexpr int kb_hi(int KB) { return KB > 8 ? KB % 10 : KB; }
__host__ __device__ constexpr int kb_lo(int KB) { return KB > 8 ? KB / 10 : KB; }
__host__ __device__ constexpr int key_words(int KB) { return KB > 8 ? 4 : KB; }  // code registers per slice
__host__ __device__ constexpr int key_token_bytes(int KB) { return KB > 8 ? 8 * (kb_hi(KB) + kb_lo(KB)) : 16 * KB; }

// Registers of one 16-token tile, key half and value half (loaded apart so
// that the keys of the next tile can be in flight while a tile is scored).
template <int KB, bool QJL>
struct KeyRegs {
  // key code slice t (coords 32t..32t+31) of tokens r, r+8; mixed keys: high
  // codes in words 0-1, low codes in words 2-3
  uint32_t k0[key_words(KB)], k1[key_words(KB)];
  float nk0, nk1;           // key norms of tokens r, r+8
  float g0, g1;             // QJL gammas
  uint32_t s0, s1;          // QJL sign word t of tokens r, r+8
  bool ok0, ok1;            // token r / r+8 is a live compressed token
};
template <int VB>
struct ValRegs {
  float nv0, nv1;           // value norms of tokens r, r+8
  // value code bits of coords 16r..16r+15 of tokens 2t, 2t+1, 2t+8, 2t+9: for
  // 3-bit codes word pairs (vlo[i], vhi[i]) of token i's chunk; for 2- and
  // 4-bit codes, (vlo, vhi)[2tp + eo] = the even (eo = 0) or odd coordinate
  // stream of token pair tp (value_pairs_interleaved), vhi unused at 2 bits
  uint32_t vlo[4], vhi[4];
};

// `width` bits at compile-time bit `pos` of the 64-bit (hi:lo), moved to bit
// SH and ORed with `base` (table base and lane slot; the fields never overlap).
template <int SH>
__device__ __forceinline__ uint32_t field_at(uint32_t lo, uint32_t hi, int pos, int width, uint32_t base) {
  const uint32_t mask = ((1u << width) - 1u) << SH;
  uint32_t x;
  if (pos + width <= 32) {
    x = pos >= SH ? (lo >> (pos - SH)) : (lo << (SH - pos));
  } else if (pos >= 32) {
    x = (pos - 32) >= SH ? (hi >> (pos - 32 - SH)) : (hi << (SH - (pos - 32)));
  } else {
    x = __funnelshift_r(lo, hi, pos) << SH;
  }
  return (x & mask) | base;
}

// Shared-memory offset of the key-table entry of code pair p (coordinates
// 32t+2p, 32t+2p+1): table offset | pair code << 8 | lane * 8.
template <int KB>
__device__ __forceinline__ uint32_t key_addr(const uint32_t (&w)[KB], int p, uint32_t laneK) {
  if constexpr (KB == 4) {
    // byte p of the slice into bits 8..15; bytes 0, 2, 3 from laneK
    return __byte_perm(w[p >> 2], laneK, 0x7604 | ((p & 3) << 4));
  } else {
    const int bit = 2 * KB * p, wi = bit >> 5;
    return field_at<8>(w[wi], (wi + 1 < KB) ? w[wi + 1] : 0u, bit & 31, 2 * KB, laneK);
  }
}

// Table offset of code pair p (codes 2p, 2p+1) of a 16-code stream slice of
// BITS-bit codes held in (w1:w0): base | pair code << 8.
template <int BITS>
__device__ __forceinline__ uint32_t mixed_pair_addr(uint32_t w0, uint32_t w1, int p, uint32_t base) {
  if constexpr (BITS == 4) return __byte_perm(p < 4 ? w0 : w1, base, 0x7604 | ((p & 3) << 4));
  else return field_at<8>(w0, w1, 2 * BITS * p, 2 * BITS, base);
}

// +-1 fp16 pair from sign bits p and p+16 of a word (bit set -> +1).
__device__ __forceinline__ uint32_t sign_pair(uint32_t w, int p) {
  return 0xBC00BC00u ^ ((w << (15 - p)) & 0x80008000u);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Ask the TMA engine to stage a page slab in L2 (no registers, no smem).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Read-only streaming loads of the packed cache that do not allocate in L1
// (the tile data is used once; L1 hit rates for it are ~3 %).
__device__ __forceinline__ uint4 ldna(const uint4 *p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldna(const uint2 *p) {
  uint2 v;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldna(const uint32_t *p) {
  uint32_t v;
  asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float ldna(const float *p) {
  float v;
  asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
// 32 bytes in one request (32-byte aligned address): every 32-byte sector a
// warp touches is then read whole by one request, not half by each of two.
__device__ __forceinline__ void ldna32B(const void *p, uint32_t (&w)[8]) {
  asm("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
      : "l"(p));
}
template <int NB>
__device__ __forceinline__ void ldg_words(const uint8_t *p, uint32_t (&w)[NB]) {
  if constexpr (NB == 4) {
    const uint4 v = ldna(reinterpret_cast<const uint4 *>(p));
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (NB == 2) {
    const uint2 v = ldna(reinterpret_cast<const uint2 *>(p));
    w[0] = v.x; w[1] = v.y;
  } else {
#pragma unroll
    for (int k = 0; k < NB; k++) w[k] = ldna(reinterpret_cast<const uint32_t *>(p) + k);
  }
}

// 16 codes of BITS bits starting at byte `off` of a token's key stream (the
// stream starts 8-byte aligned; `off` is a multiple of 8 for 4-bit codes, of
// 4 for 2-bit codes and even for 3-bit codes), as bits 0.. of (w0, w1).
template <int BITS>
__device__ __forceinline__ void load_codes16(const uint8_t *tok, int off, uint32_t &w0, uint32_t &w1) {
  if constexpr (BITS == 4) {
    const uint2 v = ldna(reinterpret_cast<const uint2 *>(tok + off));
    w0 = v.x;
    w1 = v.y;
  } else if constexpr (BITS == 2) {
    w0 = ldna(reinterpret_cast<const uint32_t *>(tok + off));
    w1 = 0u;
  } else {  // 6 bytes at an even offset: the two aligned words around them
    const uint32_t *p = reinterpret_cast<const uint32_t *>(tok + (off & ~3));
    const uint32_t a0 = ldna(p), a1 = ldna(p + 1);
    const int sh = (off & 3) * 8;
    w0 = __funnelshift_r(a0, a1, sh);
    w1 = a1 >> sh;
  }
}

// Lane t's mixed-rate key slice of one token.
template <int KB>
__device__ __forceinline__ void load_mixed_slice(const uint8_t *tok, int t, uint32_t (&w)[4]) {
  constexpr int HB = kb_hi(KB), LB = kb_lo(KB);
  load_codes16<HB>(tok, 2 * HB * t, w[0], w[1]);
  load_codes16<LB>(tok, 8 * HB + 2 * LB * t, w[2], w[3]);
}

// Key registers of the 16-token tile at offset o0 of a page slab; `live` is
// the number of leading tokens of the tile that are compressed tokens (0 for
// a page outside the pool).
template <int KB, bool QJL>
__device__ __forceinline__ void load_keys(const AttnArgs &a, const uint8_t *slab, int o0, int live, int r, int t,
                                          KeyRegs<KB, QJL> &R) {
  constexpr int KCB = key_token_bytes(KB);
  R.ok0 = r < live;
  R.ok1 = r + 8 < live;
  if constexpr (kb_mixed(KB)) {
    const uint8_t *kc = slab + a.k_codes_o;
    load_mixed_slice<KB>(kc + (o0 + r) * KCB, t, R.k0);
    load_mixed_slice<KB>(kc + (o0 + r + 8) * KCB, t, R.k1);
  } else {
    const uint8_t *kc = slab + a.k_codes_o + t * 4 * KB;
    ldg_words<KB>(kc + (o0 + r) * KCB, R.k0);
    ldg_words<KB>(kc + (o0 + r + 8) * KCB, R.k1);
  }
  const float *kn = reinterpret_cast<const float *>(slab + a.k_norm_o) + o0;
  R.nk0 = ldna(kn + r);
  R.nk1 = ldna(kn + r + 8);
  if constexpr (QJL) {
    const float *kg = reinterpret_cast<const float *>(slab + a.k_gamma_o) + o0;
    R.g0 = ldna(kg + r);
    R.g1 = ldna(kg + r + 8);
    const uint32_t *ks = reinterpret_cast<const uint32_t *>(slab + a.k_signs_o) + o0 * (kM / 32) + t;
    R.s0 = ldna(ks + r * (kM / 32));
    R.s1 = ldna(ks + (r + 8) * (kM / 32));
  }
}

// Value registers of the same tile.
template <int VB>
__device__ __forceinline__ void load_values(const AttnArgs &a, const uint8_t *slab, int o0, int r, int t,
                                            ValRegs<VB> &R) {
  constexpr int VCB = 16 * VB;
  const float *vn = reinterpret_cast<const float *>(slab + a.v_norm_o) + o0;
  R.nv0 = ldna(vn + r);
  R.nv1 = ldna(vn + r + 8);
  // chunk r (coordinates 16r..16r+15) of tokens 2t, 2t+1, 2t+8, 2t+9: one
  // contiguous run of 4 * 2VB bytes in the grouped value-code section (two
  // pair-interleaved runs of 4VB bytes for 2- and 4-bit codes)
  const uint8_t *vc = slab + a.v_codes_o + (int64_t)o0 * VCB + r * (16 * 2 * VB) + t * (4 * 2 * VB);
  if constexpr (VB == 4) {
    // 32-byte aligned: sections are multiples of 64 bytes for P % 16 == 0 and
    // the pool is 32-byte aligned
    uint32_t w[8];
    ldna32B(vc, w);
    R.vlo[0] = w[0]; R.vhi[0] = w[1]; R.vlo[1] = w[2]; R.vhi[1] = w[3];
    R.vlo[2] = w[4]; R.vhi[2] = w[5]; R.vlo[3] = w[6]; R.vhi[3] = w[7];
  } else if constexpr (VB == 2) {
    const uint4 x0 = ldna(reinterpret_cast<const uint4 *>(vc));
    R.vlo[0] = x0.x; R.vlo[1] = x0.y; R.vlo[2] = x0.z; R.vlo[3] = x0.w;
#pragma unroll
    for (int i = 0; i < 4; i++) R.vhi[i] = 0u;
  } else {  // four 6-byte chunks in 24 bytes (8-byte aligned)
    const uint2 x0 = ldna(reinterpret_cast<const uint2 *>(vc)), x1 = ldna(reinterpret_cast<const uint2 *>(vc) + 1),
                x2 = ldna(reinterpret_cast<const uint2 *>(vc) + 2);
    R.vlo[0] = x0.x;                                  R.vhi[0] = x0.y & 0xFFFFu;
    R.vlo[1] = __byte_perm(x0.y, x1.x, 0x5432);       R.vhi[1] = x1.x >> 16;
    R.vlo[2] = x1.y;                                  R.vhi[2] = x2.x & 0xFFFFu;
    R.vlo[3] = __byte_perm(x2.x, x2.y, 0x5432);       R.vhi[3] = x2.y >> 16;
  }
}

// Walks the tiles of one segment page by page, without divisions.
struct TileCursor {
  const uint8_t *pool;
  const int32_t *btrow;
  int64_t num_pages, page_bytes, slab_off;  // slab_off = h * slab_bytes
  int P, pidx, o0, tok0, clen;
  const uint8_t *slab;
  bool page_ok;

  __device__ __forceinline__ int live() const { return page_ok ? clen - tok0 : 0; }
  // Block-table entries of the next two pages, loaded a page ahead of use, so
  // that neither the page switch nor the L2 prefetch of the next page waits
  // on a block-table load.
  int last_page;
  int32_t pg_next, pg_ahead;  // entries of pages pidx + 1, pidx + 2 (0 past last_page)
  __device__ __forceinline__ void set_page(int32_t page, int32_t *err_word, bool reporter) {
    page_ok = page >= 0 && (int64_t)page < num_pages;
    if (!page_ok) {
      if (reporter) report(err_word, TQ_DEVERR_PAGE_RANGE);
      page = 0;
    }
    slab = pool + (int64_t)page * page_bytes + slab_off;
  }
  __device__ __forceinline__ const uint8_t *slab_if_valid(int32_t page) const {
    return (page >= 0 && (int64_t)page < num_pages) ? pool + (int64_t)page * page_bytes + slab_off : nullptr;
  }
  // first page of a segment (pidx, last_page set); lane 0 stages it and the
  // next one in L2
  __device__ __forceinline__ void begin(int32_t *err_word, bool lane0, uint32_t slab_bytes) {
    const int32_t page = __ldg(btrow + pidx);
    pg_next = pidx + 1 <= last_page ? __ldg(btrow + pidx + 1) : 0;
    pg_ahead = pidx + 2 <= last_page ? __ldg(btrow + pidx + 2) : 0;
    set_page(page, err_word, lane0);
    if (lane0) {
      if (page_ok) prefetch_l2(slab, slab_bytes);
      const uint8_t *sp = pidx + 1 <= last_page ? slab_if_valid(pg_next) : nullptr;
      if (sp) prefetch_l2(sp, slab_bytes);
    }
  }
  // the next tile; at a page switch lane 0 stages the page after it in L2
  __device__ __forceinline__ void step(int32_t *err_word, bool lane0, uint32_t slab_bytes) {
    if (!advance()) return;
    const int32_t page = pg_next;
    pg_next = pg_ahead;
    pg_ahead = pidx + 2 <= last_page ? __ldg(btrow + pidx + 2) : 0;
    set_page(page, err_word, lane0);
    if (lane0 && pidx + 1 <= last_page) {
      const uint8_t *sp = slab_if_valid(pg_next);
      if (sp) prefetch_l2(sp, slab_bytes);
    }
  }
  __device__ __forceinline__ bool advance() {  // true when a new page starts
    tok0 += 16;
    o0 += 16;
    if (o0 == P) {
      o0 = 0;
      ++pidx;
      return true;
    }
    return false;
  }
};

// Register pipeline over tiles: the next tile's keys in flight while a tile
// is scored, its values loaded as its keys are scored, for uniform key
// widths; mixed widths load a tile, then compute it (measured at the
// Llama-3-8B decode shape, 32K context: K4/V4 141.3 us with keys in flight
// against 146.4 without; K3.5/V3 188.4 against 169.0).
// Value MMA layouts.  Parity pairs (K index = token slot x coordinate
// parity: an A register is one code pair of one token) for 3-bit values,
// where they replace a gather of two tokens' 3-bit fields (measured at the
// Llama-3-8B decode shape, 32K context: K3.5/V3 160.3 us against 170.0);
// coordinate halves (K index = coordinate half x token: an A register pairs
// two tokens' codes of one coordinate, stored so in the pair-interleaved
// layout) for 2- and 4-bit values.
template <int VB>
__host__ __device__ constexpr bool val_parity_pairs() {
  return VB == 3;
}
template <int KB>
__host__ __device__ constexpr bool keys_in_flight() {
  return !kb_mixed(KB);
}
// The whole next tile in flight (values too) for 2-bit keys and values:
// measured at the long-context shape (K2+QJL/V2, 128K) 159.8 against
// 172.2 us per launch; at the Llama-3-8B K4/V4 shape 131.1 against 127.0.
template <int KB, int VB>
__host__ __device__ constexpr bool values_in_flight() {
  return KB == 2 && VB == 2;
}

// Pages of a segment are staged in L2 one page ahead of the page being read
// (no prefetch, and two pages ahead, measured slower at the Llama-3-8B decode
// shape).

// Shared-memory placement of the centroid tables, as offsets from the start
// of dynamic shared memory.  Rows of 256 bytes indexed by a code pair (or a
// code byte); lane l reads its own bank-private entry, so a warp's lookup is
// conflict-free, and an entry offset is (table offset | code << 8 | lane slot),
// one prmt / lop3.
//   - Value table at 0: 4-byte entries (the two fp16 centroids of a code pair)
//     in the first 128 bytes of a row; 2-bit values: 8-byte entries indexed by
//     a byte of interleaved codes (two coordinates), whole rows.
//   - Key table: 4-byte entries (two fp16 centroids; the stored codebook is
//     fp16-exact, so a centroid is an exact tensor-core operand) in the second
//     half of the same rows (offset 128) when both kinds use 4-byte entries;
//     2-bit keys use 8-byte entries indexed by a code byte (two pairs) in rows
//     of their own from 64 KB.  Mixed-rate keys: the low channels' table
//     follows the high channels' rows.
//
// Window-aligned tables (uniform 4-bit keys without QJL): the tables are
// placed, at run time, where their shared-window addresses are multiples of
// 64 KB, so the prmt result is itself the address of an `ld.shared` and no
// lookup adds the base of dynamic shared memory (which is not 0: the window
// starts with reserved bytes).  The launch reserves 64 KB of room for the
// shift.
template <int KB>
__host__ __device__ constexpr bool byte_keys() {
  return KB == 2;
}
template <int VB>
__host__ __device__ constexpr bool byte_values() {
  return VB == 2;
}
template <int KB, int VB>
__host__ __device__ constexpr bool shared_rows() {
  return !byte_keys<KB>() && !byte_values<VB>();
}
template <int KB, bool QJL>
__host__ __device__ constexpr bool aligned_tables() {
  return KB == 4 && !QJL;
}
template <int KB>
__host__ __device__ constexpr uint32_t key_rows() {
  return kb_mixed(KB) ? (uint32_t(1) << (2 * kb_hi(KB))) + (uint32_t(1) << (2 * kb_lo(KB)))
                      : byte_keys<KB>() ? 256u : (uint32_t(1) << (2 * KB));
}
template <int KB, int VB>
__host__ __device__ constexpr uint32_t key_table_off() {
  return shared_rows<KB, VB>() ? 128u : 65536u;
}
// Mixed keys: the low channels' pair table follows the high channels' rows.
template <int KB, int VB>
__host__ __device__ constexpr uint32_t key_lo_table_off() {
  return key_table_off<KB, VB>() + (uint32_t(1) << (2 * kb_hi(KB))) * 256;
}
template <int KB, int VB>
__host__ __device__ constexpr uint32_t attn_tables_end() {
  return shared_rows<KB, VB>() ? 256u * (key_rows<KB>() > (1u << (2 * VB)) ? key_rows<KB>() : (1u << (2 * VB)))
                               : 65536u + 256u * key_rows<KB>();
}
template <int KB, int VB, bool QJL, int NT>
constexpr size_t attn_smem_bytes() {
  return aligned_tables<KB, QJL>()
             ? 65536 + (size_t)attn_tables_end<KB, VB>()  // room to shift the tables to a 64 KB window boundary
             : (size_t)attn_tables_end<KB, VB>();
}

// QOP: the key-score query operands are the prep kernel's ready-made words
// (q_op); otherwise the kernel splits q_rot into them.  The host picks it per
// shape: measured at the Llama-3-8B K4/V4 shape (108 tiles per warp) 118.8 us
// per launch splitting in the kernel against 129.0 with loaded words; at the
// Qwen2.5-3B shape (2 tiles per warp) 15.0 against 12.9.  (A run-time switch
// between the two inside one kernel measured 131.0 at the Llama shape.)
template <int KB, int VB, bool QJL, int NT, bool QOP>
__global__ void __launch_bounds__(attn_threads(NT, QJL), 1) attn_main_kernel(const AttnArgs a) {
  constexpr int EK = 1 << (2 * kb_hi(KB)), EV = 1 << (2 * VB);
  static_assert(byte_values<VB>() || EV * 256 <= 65536, "table sizes");
  static_assert(attn_tables_end<KB, VB>() <= 232448, "tables above the shared-memory limit");
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr bool kAligned = aligned_tables<KB, QJL>();
  constexpr uint32_t kKeyOff = key_table_off<KB, VB>();
  // aligned tables: the shift that puts them on a 64 KB window boundary and
  // that boundary (table offsets below are added to it); otherwise 0, 0
  const uint32_t win_base = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t tshift = kAligned ? (0u - win_base) & 0xFFFFu : 0u;
  const uint32_t tbase = kAligned ? win_base + tshift : 0u;
  uint8_t *const tables = smem + tshift;
  // table reads: at a shared-window address (aligned tables) or at a byte
  // offset from the start of dynamic shared memory
  auto lut64 = [&](uint32_t off) {
    uint2 v;
    if constexpr (kAligned) asm("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(off));
    else v = *reinterpret_cast<const uint2 *>(smem + off);
    return v;
  };
  auto lut32 = [&](uint32_t off) {
    uint32_t v;
    if constexpr (kAligned) asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(off));
    else v = *reinterpret_cast<const uint32_t *>(smem + off);
    return v;
  };

  // Bank-private centroid-pair tables: lane l reads its own copy in bank l
  // (8-byte entries: banks 2l, 2l+1 of its half-warp's wavefront).  The two
  // fp16 centroids (x256) of code pair e of a `bits`-bit codebook cb:
  auto pair_of = [&](const float *cb, int bits, int e) {
    return pack_half2(__ldg(cb + (e & ((1 << bits) - 1))) * kCentScale, __ldg(cb + (e >> bits)) * kCentScale);
  };
  uint32_t *const tab32 = reinterpret_cast<uint32_t *>(tables);
  uint2 *const tab64 = reinterpret_cast<uint2 *>(tables);
  // One thread per entry: its value once, stored to the 32 lane copies with
  // 16-byte stores whose chunk order is rotated by the entry, so the eight
  // stores of a wavefront fall in different banks.  fill32: entry e's copies
  // are words w0 + 64 e .. + 31; fill64: 8-byte slots p0 + 32 e .. + 31.
  auto fill32 = [&](uint32_t w0, int E, auto val) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      const uint32_t v = val(e);
      const uint4 q4 = make_uint4(v, v, v, v);
      uint4 *d = reinterpret_cast<uint4 *>(tab32 + w0 + 64 * e);
#pragma unroll
      for (int k = 0; k < 8; k++) d[(k + e) & 7] = q4;
    }
  };
  auto fill64 = [&](uint32_t p0, int E, auto val) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      const uint2 v = val(e);
      const uint4 q4 = make_uint4(v.x, v.y, v.x, v.y);
      uint4 *d = reinterpret_cast<uint4 *>(tab64 + p0 + 32 * e);
#pragma unroll
      for (int k = 0; k < 16; k++) d[(k + e) & 15] = q4;
    }
  };
  if constexpr (byte_keys<KB>()) {
    // 2-bit keys: indexed by a code byte (pair 2k in the low nibble, 2k + 1 high)
    fill64(kKeyOff / 8, 256, [&](int e) { return make_uint2(pair_of(a.k_cb, 2, e & 15), pair_of(a.k_cb, 2, e >> 4)); });
  } else {
    fill32(kKeyOff / 4, EK, [&](int e) { return pair_of(a.k_cb, kb_hi(KB), e); });
  }
  if constexpr (kb_mixed(KB)) {
    // low channels: the k_bits codebook follows the (k_bits + 1) one
    constexpr int HB = kb_hi(KB), LB = kb_lo(KB), EL = 1 << (2 * LB);
    const float *cb_lo = a.k_cb + (2 << HB) - 1;
    fill32(key_lo_table_off<KB, VB>() / 4, EL, [&](int e) { return pair_of(cb_lo, LB, e); });
  }
  if constexpr (byte_values<VB>()) {
    // 2-bit values: indexed by a byte of the interleaved codes (two coordinates)
    fill64(0, 256, [&](int e) { return make_uint2(pair_of(a.v_cb, VB, e & 15), pair_of(a.v_cb, VB, e >> 4)); });
  } else {
    fill32(0, EV, [&](int e) { return pair_of(a.v_cb, VB, e); });
  }
  __syncthreads();
  // Up to here only the codebooks were read; launched as a dependent of the
  // prep kernel, the table build above overlaps it.  Its outputs (tile
  // counts, rotated queries) are read below.
  griddep_wait();
  griddep_launch_dependents();

  const int lane = threadIdx.x & 31, r = lane >> 2, t = lane & 3;
  const int64_t wg = (int64_t)blockIdx.x * attn_warps(NT, QJL) + (threadIdx.x >> 5);
  // QOP (short tile ranges) with at most 31 sequences: lane i loads pre[i]
  // together with the header, so the first tile is located without a second
  // dependent load (a ballot over the lanes instead of the binary search)
  const bool pre_in_lanes = QOP && a.B <= 31;
  int64_t pre_l = INT64_MAX;
  if (pre_in_lanes && lane <= a.B) pre_l = a.pre[lane];
  const int64_t T = a.hdr->total_tiles;
  const int64_t NW = a.hdr->active_warps;
  if (wg >= NW) return;
  const int64_t ts = T * wg / NW, te = T * (wg + 1) / NW;
  if (ts >= te) return;
  const uint32_t laneK = (tbase + kKeyOff) | ((uint32_t)lane * (byte_keys<KB>() ? 8u : 4u));
  const uint32_t laneKL = (tbase + key_lo_table_off<KB, VB>()) | ((uint32_t)lane * 4u);  // mixed keys: low-channel table
  const uint32_t laneV = tbase | ((uint32_t)lane * (byte_values<VB>() ? 8u : 4u));
  // value-weight operands: the low (tokens 2t, 2t+1) or high (2t+8, 2t+9)
  // half of a weight pair into the half of this lane's parity column r/4
  const uint32_t selW_lo = r < 4 ? 0x4410u : 0x1044u, selW_hi = r < 4 ? 0x4432u : 0x3244u;
  const int H = a.H, G = a.G, Hq = a.Hq;
  const int tpp = a.P >> 4;
  const uint32_t slab_bytes = (uint32_t)a.slab_bytes;

  // locate the first tile: largest b with H * pre[b] <= ts
  int b = 0;
  int64_t pre_b, pre_b1;
  if (pre_in_lanes) {
    // pre is non-decreasing and pre[0] = 0: the lanes b < B with
    // H * pre[b] <= ts are a prefix
    const uint32_t le = __ballot_sync(0xffffffffu, lane < a.B && H * pre_l <= ts);
    b = __popc(le) - 1;
    pre_b = __shfl_sync(0xffffffffu, pre_l, b);
    pre_b1 = __shfl_sync(0xffffffffu, pre_l, b + 1);
  } else {
    int lo = 0, hi = a.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (H * a.pre[mid] <= ts) lo = mid; else hi = mid;
    }
    b = lo;
    pre_b = a.pre[b];
    pre_b1 = a.pre[b + 1];
  }
  int tb = (int)(pre_b1 - pre_b);
  int h = (int)((ts - H * pre_b) / tb);
  int j = (int)((ts - H * pre_b) - (int64_t)h * tb);
  int64_t pos = ts;

  while (pos < te) {
    const int seg_tiles = (int)min(te - pos, (int64_t)(tb - j));

    // ---- the segment's first page: block-table loads issued before the
    // operand loads below, so that both wait on one memory latency
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
    cur.begin(a.err_word, lane == 0, slab_bytes);

    // ---- segment setup: query operands for the G heads of (b, h), as the
    // prep kernel wrote them (hi / lo fp16 words in register order, the
    // score constants): loads only, all issued together
    uint32_t qb[NT][8][2];
    uint32_t sb[NT][QJL ? 8 : 1][2];
    float cK[NT], cQ[NT];
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      const int gcol = 4 * nt + (r >> 1);
      const int part = r & 1;  // hi (even rows) or lo (odd rows) of head gcol
      const bool gval = gcol < G;
      const int64_t qrow = ((int64_t)b * Hq + (int64_t)h * G + (gval ? gcol : 0));
      const uint4 *op = reinterpret_cast<const uint4 *>(a.q_op + qrow * 256 + 16 * t);
      if constexpr (QOP) {  // the prep kernel's operand words
#pragma unroll
        for (int u = 0; u < 4; u++) {
          const uint4 v = gval ? op[16 * part + u] : make_uint4(0u, 0u, 0u, 0u);
          qb[nt][2 * u][0] = v.x;
          qb[nt][2 * u][1] = v.y;
          qb[nt][2 * u + 1][0] = v.z;
          qb[nt][2 * u + 1][1] = v.w;
        }
      } else {  // the hi / lo split of q_rot here
        const int ecol = gval ? a.q_exp[qrow * 2] : 0;
        const float sc = ldexpf(1.0f, ecol);
        const float *qr = a.q_rot + qrow * kD + 32 * t;
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
          const float4 v = gval ? *reinterpret_cast<const float4 *>(qr + 4 * kk) : make_float4(0.f, 0.f, 0.f, 0.f);
          __half hx, lx, hy, ly, hz, lz, hw, lw;
          split_half(v.x * sc, hx, lx);
          split_half(v.y * sc, hy, ly);
          split_half(v.z * sc, hz, lz);
          split_half(v.w * sc, hw, lw);
          qb[nt][kk][0] = part ? pack_half2_raw(lx, ly) : pack_half2_raw(hx, hy);
          qb[nt][kk][1] = part ? pack_half2_raw(lz, lw) : pack_half2_raw(hz, hw);
        }
      }
      if constexpr (QJL) {
#pragma unroll
        for (int u = 0; u < 4; u++) {
          const uint4 v = gval ? op[16 * (2 + part) + u] : make_uint4(0u, 0u, 0u, 0u);
          sb[nt][2 * u][0] = v.x;
          sb[nt][2 * u][1] = v.y;
          sb[nt][2 * u + 1][0] = v.z;
          sb[nt][2 * u + 1][1] = v.w;
        }
      }
      // score constants of this thread's own head g = 4nt + t (log2 domain)
      const int gown = 4 * nt + t;
      const float2 c = a.q_cst[(int64_t)b * Hq + (int64_t)h * G + (gown < G ? gown : 0)];
      cK[nt] = c.x;
      cQ[nt] = QJL ? c.y : 0.f;
    }

    float mu[NT], lsum[NT];
    float acc[4][NT][4];  // value accumulator m-tiles (see the file header)
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      mu[nt] = -INFINITY;
      lsum[nt] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 4; mt++)
#pragma unroll
        for (int i = 0; i < 4; i++) acc[mt][nt][i] = 0.f;
    }
    float nu = 0.f, inv_nu = 0.f;


    auto process = [&](const KeyRegs<KB, QJL> &R, const ValRegs<VB> &V) {
      if (!__any_sync(0xffffffffu, R.ok0)) return;  // token 0 of a tile is live iff any is
      // ---- scores: tokens 0-7, tokens 8-15 and QJL chains run independently.
      // sa rows r / r+8 = token r hi / lo part; sb likewise for token r+8.
      // scr[nt][c]: scores, rows r / r+8 = tokens r / r+8, columns 2t / 2t+1 =
      // head t times the hi / lo part of the query.  One accumulation chain
      // per n-tile for one n-tile, else two (even and odd k-steps): measured
      // at the Llama-3-8B decode shape, 32K context, 127.2 against 129.2 us;
      // at the Qwen2.5-3B shape (two n-tiles) 21.4 against 22.1 us.
      constexpr int kChains = NT == 1 ? 1 : 2;
      float scr[NT][2][4], sq[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int i = 0; i < 4; i++) { scr[nt][0][i] = 0.f; scr[nt][1][i] = 0.f; sq[nt][i] = 0.f; }
#pragma unroll
      for (int kk = 0; kk < 8; kk++) {
        // A operand: the fp16 centroids of code pairs 2kk (k slots 2t, 2t+1)
        // and 2kk + 1 (slots 2t+8, 2t+9) of token r (A0, A2) and r+8 (A1, A3)
        uint32_t A0, A1, A2, A3;
        if constexpr (kb_mixed(KB)) {
          // channels 32t + 4kk .. +3 are the 4-code group g of the lane's
          // high stream when kk mod 4 < 2, of its low stream otherwise
          const int g = (kk & 1) + 2 * (kk >> 2);
          if ((kk & 2) == 0) {
            A0 = lut32(mixed_pair_addr<kb_hi(KB)>(R.k0[0], R.k0[1], 2 * g, laneK));
            A2 = lut32(mixed_pair_addr<kb_hi(KB)>(R.k0[0], R.k0[1], 2 * g + 1, laneK));
            A1 = lut32(mixed_pair_addr<kb_hi(KB)>(R.k1[0], R.k1[1], 2 * g, laneK));
            A3 = lut32(mixed_pair_addr<kb_hi(KB)>(R.k1[0], R.k1[1], 2 * g + 1, laneK));
          } else {
            A0 = lut32(mixed_pair_addr<kb_lo(KB)>(R.k0[2], R.k0[3], 2 * g, laneKL));
            A2 = lut32(mixed_pair_addr<kb_lo(KB)>(R.k0[2], R.k0[3], 2 * g + 1, laneKL));
            A1 = lut32(mixed_pair_addr<kb_lo(KB)>(R.k1[2], R.k1[3], 2 * g, laneKL));
            A3 = lut32(mixed_pair_addr<kb_lo(KB)>(R.k1[2], R.k1[3], 2 * g + 1, laneKL));
          }
        } else if constexpr (byte_keys<KB>()) {  // byte kk = pairs 2kk (low nibble), 2kk+1: one 8-byte entry
          const uint2 L0 = lut64(__byte_perm(R.k0[kk >> 2], laneK, 0x7604 | ((kk & 3) << 4)));
          const uint2 L1 = lut64(__byte_perm(R.k1[kk >> 2], laneK, 0x7604 | ((kk & 3) << 4)));
          A0 = L0.x;
          A2 = L0.y;
          A1 = L1.x;
          A3 = L1.y;
        } else {
          A0 = lut32(key_addr<KB>(R.k0, 2 * kk, laneK));
          A2 = lut32(key_addr<KB>(R.k0, 2 * kk + 1, laneK));
          A1 = lut32(key_addr<KB>(R.k1, 2 * kk, laneK));
          A3 = lut32(key_addr<KB>(R.k1, 2 * kk + 1, laneK));
        }
#pragma unroll
        for (int nt = 0; nt < NT; nt++) mma_16816(scr[nt][kChains == 1 ? 0 : (kk & 1)], A0, A1, A2, A3, qb[nt][kk][0], qb[nt][kk][1]);
        if constexpr (QJL) {
          const uint32_t a0 = sign_pair(R.s0, 2 * kk), a1 = sign_pair(R.s1, 2 * kk);
          const uint32_t a2 = sign_pair(R.s0, 2 * kk + 1), a3 = sign_pair(R.s1, 2 * kk + 1);
#pragma unroll
          for (int nt = 0; nt < NT; nt++) mma_16816(sq[nt], a0, a1, a2, a3, sb[nt][kk][0], sb[nt][kk][1]);
        }
      }
      // ---- online softmax (log2 domain) and value weights, relative to the
      // running (mu, nu).  They are moved (warp reductions, accumulator
      // rescale) only when a live token would exceed the weight bound: a logit
      // above mu + kLazyLog2 or a value norm above kLazyNu * nu.  Weights then
      // stay below 2^kLazyLog2 * kLazyNu, which kWeightScale keeps inside fp16.
      const float vn0 = R.ok0 ? V.nv0 : 0.f, vn1 = R.ok1 ? V.nv1 : 0.f;
      float lg0[NT], lg1[NT];
      bool big = vn0 > kLazyNu * nu || vn1 > kLazyNu * nu;
#pragma unroll
      for (int nt = 0; nt < NT; nt++) {
        float l0 = (scr[nt][0][0] + scr[nt][0][1]) * cK[nt];
        float l1 = (scr[nt][0][2] + scr[nt][0][3]) * cK[nt];
        if constexpr (kChains == 2) {
          l0 = fmaf(scr[nt][1][0] + scr[nt][1][1], cK[nt], l0);
          l1 = fmaf(scr[nt][1][2] + scr[nt][1][3], cK[nt], l1);
        }
        if constexpr (QJL) {
          l0 = fmaf(R.g0 * (sq[nt][0] + sq[nt][1]), cQ[nt], l0);
          l1 = fmaf(R.g1 * (sq[nt][2] + sq[nt][3]), cQ[nt], l1);
        }
        lg0[nt] = R.ok0 ? R.nk0 * l0 : -INFINITY;
        lg1[nt] = R.ok1 ? R.nk1 * l1 : -INFINITY;
        big |= fmaxf(lg0[nt], lg1[nt]) > mu[nt] + kLazyLog2;
      }
      if (__any_sync(0xffffffffu, big)) {
        const float tnu = warp_max_xor(fmaxf(vn0, vn1), 4 | 8 | 16);
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
          mu[nt] = mnew;
          beta[nt] = alpha * nu_ratio;
        }
        // accumulator columns hold heads 4nt + 2(t&1) (i = 0, 2) and
        // 4nt + 2(t&1) + 1 (i = 1, 3): their factors from the lanes owning them
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
      if constexpr (val_parity_pairs<VB>()) {
        // wb[nt][s][0 / 1]: B operand of token group s for the token slots t
        // (token 2t + 8s) and t + 4 (token 2t + 1 + 8s); column r = (coordinate
        // parity r/4, head 4nt + r%4): the token's weight in the half of its
        // parity, 0 in the other half.  The lanes (2t, r%4) and (2t+1, r%4)
        // own the weights.
        uint32_t wb[NT][2][2];
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
          const float p0 = fast_exp2(lg0[nt] - mu[nt]), p1 = fast_exp2(lg1[nt] - mu[nt]);
          lsum[nt] += p0 + p1;
          const float w0 = p0 * vn0 * inv_nu, w1 = p1 * vn1 * inv_nu;
          const uint32_t Wh = pack_half2(w0, w1);  // (token r, token r+8) of head 4nt + t
          const int src0 = 4 * (2 * t) + (r & 3), src1 = src0 + 4;
          const uint32_t h0 = __shfl_sync(0xffffffffu, Wh, src0);  // tokens 2t, 2t+8
          const uint32_t h1 = __shfl_sync(0xffffffffu, Wh, src1);  // tokens 2t+1, 2t+9
          wb[nt][0][0] = __byte_perm(h0, 0u, selW_lo);
          wb[nt][0][1] = __byte_perm(h1, 0u, selW_lo);
          wb[nt][1][0] = __byte_perm(h0, 0u, selW_hi);
          wb[nt][1][1] = __byte_perm(h1, 0u, selW_hi);
        }
        // ---- values.  The K index of an MMA is (token slot i, coordinate
        // parity e): an A register holds two consecutive coordinates of one
        // token, i.e. one code pair of the token's own stream, looked up once.
        // Token group s, m-tile mt: row r is the coordinate pair 2mt of this
        // lane's chunk (coordinates 16r + 4mt, +1), row r+8 the pair 2mt + 1
        // (16r + 4mt + 2, +3); slots t, t+4 are tokens 2t + 8s, 2t + 1 + 8s.
#pragma unroll
        for (int s = 0; s < 2; s++) {
#pragma unroll
          for (int mt = 0; mt < 4; mt++) {
            uint32_t av[4];  // (token 2t+8s | 2t+1+8s) x (pair 2mt | 2mt+1)
#pragma unroll
            for (int q = 0; q < 4; q++) {
              // the 6 bits of code pair 2mt + (q&1) in the token's 48-bit chunk
              const int tok = 2 * s + (q >> 1), pair = 2 * mt + (q & 1);
              av[q] = lut32(field_at<8>(V.vlo[tok], V.vhi[tok], 6 * pair, 6, laneV));
            }
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
              mma_16816(acc[mt][nt], av[0], av[1], av[2], av[3], wb[nt][s][0], wb[nt][s][1]);
          }
        }
      } else {
        // wb[nt][s]: B operand of the value MMAs of token group s
        uint32_t wb[NT][2][2];
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
          const float p0 = fast_exp2(lg0[nt] - mu[nt]), p1 = fast_exp2(lg1[nt] - mu[nt]);
          lsum[nt] += p0 + p1;
          const float w0 = p0 * vn0 * inv_nu, w1 = p1 * vn1 * inv_nu;
          const uint32_t Wh = pack_half2(w0, w1);  // (token r, token r+8) of head 4nt + t
          // column r = (coordinate half r/4, head 4nt + r%4): the weights of
          // tokens 8s + 2t, 8s + 2t + 1 in the rows of half r/4, zeros in the
          // other half's rows; the lanes (2t, r%4), (2t+1, r%4) own them
          const int src0 = 4 * (2 * t) + (r & 3), src1 = src0 + 4;
          const uint32_t h0 = __shfl_sync(0xffffffffu, Wh, src0);
          const uint32_t h1 = __shfl_sync(0xffffffffu, Wh, src1);
          const uint32_t e0 = __byte_perm(h0, h1, 0x5410), e1 = __byte_perm(h0, h1, 0x7632);
          const bool half0 = r < 4;
          wb[nt][0][0] = half0 ? e0 : 0u;
          wb[nt][0][1] = half0 ? 0u : e0;
          wb[nt][1][0] = half0 ? e1 : 0u;
          wb[nt][1][1] = half0 ? 0u : e1;
        }
        // ---- values: the codes of the token pairs (2t, 2t+1) and (2t+8,
        // 2t+9) come interleaved at each coordinate (value_pairs_interleaved);
        // one lookup gives an A register.  Table offset = pair code << 8 | lane slot.
        uint32_t ev[2][2][2];  // [token pair][even/odd coordinate][word]
#pragma unroll
        for (int tp = 0; tp < 2; tp++)
#pragma unroll
          for (int eo = 0; eo < 2; eo++) {
            ev[tp][eo][0] = V.vlo[2 * tp + eo];
            ev[tp][eo][1] = V.vhi[2 * tp + eo];
          }
        // token group s (tokens 8s + 2t, 8s + 2t + 1 in this lane's A
        // registers), m-tile mt: A rows r / r+8 of half h are coordinates
        // 16r + 4mt + 2h / 16r + 4mt + 2h + 1, so av[q] is coordinate 16r + 4mt + q
#pragma unroll
        for (int s = 0; s < 2; s++) {
#pragma unroll
          for (int mt = 0; mt < 4; mt++) {
            uint32_t av[4];
            if constexpr (VB == 2) {
              // byte mt of ev[s][eo]: coordinates 4mt + eo and 4mt + 2 + eo
              const uint2 pe = lut64(__byte_perm(ev[s][0][0], laneV, 0x7604 | (mt << 4)));
              const uint2 po = lut64(__byte_perm(ev[s][1][0], laneV, 0x7604 | (mt << 4)));
              av[0] = pe.x; av[1] = po.x; av[2] = pe.y; av[3] = po.y;
            } else {
#pragma unroll
              for (int q = 0; q < 4; q++) {
                // 4-bit: byte k of ev[s][eo][wi] is coordinate 8wi + 2k + eo
                av[q] = lut32(__byte_perm(ev[s][q & 1][mt >> 1], laneV, 0x7604 | ((2 * (mt & 1) + (q >> 1)) << 4)));
              }
            }
#pragma unroll
            for (int nt = 0; nt < NT; nt++)
              mma_16816(acc[mt][nt], av[0], av[1], av[2], av[3], wb[nt][s][0], wb[nt][s][1]);
          }
        }
      }
    };

    auto step_cursor = [&]() { cur.step(a.err_word, lane == 0, slab_bytes); };

    using KR = KeyRegs<KB, QJL>;
    using VR = ValRegs<VB>;
    auto keys = [&](KR &R) { load_keys<KB, QJL>(a, cur.slab, cur.o0, cur.live(), r, t, R); };
    auto vals = [&](VR &R) { load_values<VB>(a, cur.slab, cur.o0, r, t, R); };
    if constexpr (values_in_flight<KB, VB>()) {
      // the whole next tile one tile ahead, handed over after each tile: one
      // copy of the tile body (measured at the long-context shape 146.9
      // against 149.5 us for a ping-pong over two copies, whose branches cost
      // about 55 register moves per tile)
      KR ka, kb;
      VR va, vb;
      keys(ka);
      vals(va);
      for (int k = 0; k < seg_tiles; k++) {
        if (k + 1 < seg_tiles) {
          step_cursor();
          keys(kb);
          vals(vb);
        }
        process(ka, va);
        ka = kb;
        va = vb;
      }
    } else if constexpr (keys_in_flight<KB>()) {
      // keys one tile ahead (ping-pong ka / kb), values at the tile itself
      KR ka, kb;
      VR v;
      keys(ka);
      for (int k = 0;;) {
        vals(v);
        if (k + 1 < seg_tiles) {
          step_cursor();
          keys(kb);
        }
        process(ka, v);
        if (++k == seg_tiles) break;
        vals(v);
        if (k + 1 < seg_tiles) {
          step_cursor();
          keys(ka);
        }
        process(kb, v);
        if (++k == seg_tiles) break;
      }
    } else {
      for (int k = 0; k < seg_tiles; k++) {
        KR ka;
        VR va;
        keys(ka);
        vals(va);
        process(ka, va);
        if (k + 1 < seg_tiles) step_cursor();
      }
    }

    // ---- segment partial: slot = warp + unit
    const int64_t slot = wg + (int64_t)b * H + h;
    const float vscale = nu / (kWeightScale * kCentScale);
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
      const float ltot = warp_sum_xor(lsum[nt], 4 | 8 | 16);
      const int g = 4 * nt + t;  // this lane's softmax state
      if (g < G && r == 0) {
        a.seg_ml[(slot * G + g) * 2] = mu[nt];
        a.seg_ml[(slot * G + g) * 2 + 1] = ltot;
      }
      // this lane's accumulator: heads gA (i = 0, 2) and gA + 1 (i = 1, 3);
      // parity pairs: coordinates 16r + 4mt + (t>>1) (i = 0, 1) and
      // 16r + 4mt + 2 + (t>>1) (i = 2, 3); coordinate halves: 16r + 4mt +
      // 2(t>>1) + {0, 1}
      const int gA = 4 * nt + 2 * (t & 1);
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        if (gA + hh < G) {
          float *row = a.seg_acc + (slot * G + gA + hh) * kD + 16 * r;
#pragma unroll
          for (int mt = 0; mt < 4; mt++) {
            if constexpr (val_parity_pairs<VB>()) {
              row[4 * mt + (t >> 1)] = acc[mt][nt][hh] * vscale;
              row[4 * mt + 2 + (t >> 1)] = acc[mt][nt][hh + 2] * vscale;
            } else {
              *reinterpret_cast<float2 *>(row + 4 * mt + 2 * (t >> 1)) =
                  make_float2(acc[mt][nt][hh] * vscale, acc[mt][nt][hh + 2] * vscale);
            }
          }
        }
      }
    }

    pos += seg_tiles;
    if (pos < te) {  // next non-empty (b, h)
      j = 0;
      if (++h == H) {
        h = 0;
        do { ++b; } while (a.pre[b + 1] == a.pre[b]);
        tb = (int)(a.pre[b + 1] - a.pre[b]);
      }
    }
  }
}

template <int KB, int VB, bool QJL, int NT, bool QOP>
cudaError_t attn_main_launch_t(const AttnArgs &a, bool query_only, int *blocks_per_sm, int blocks, cudaStream_t st) {
  auto kern = attn_main_kernel<KB, VB, QJL, NT, QOP>;
  constexpr size_t smem_bytes = attn_smem_bytes<KB, VB, QJL, NT>();
  static_assert(smem_bytes <= 232448, "dynamic shared memory above the per-CTA limit");
  static unsigned long long done = 0;
  cudaError_t e = set_smem_once(kern, (int)smem_bytes, done);
  if (e != cudaSuccess) return e;
  if (query_only) return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, kern, attn_threads(NT, QJL), smem_bytes);
  return launch_maybe_dependent(kern, dim3(blocks), dim3(attn_threads(NT, QJL)), smem_bytes, st, a.pdl, a);
}

template <int KB, bool QOP>
cudaError_t attn_main_dispatch(const AttnArgs &a, int v_bits, bool qjl, int nt, bool query_only, int *bps, int blocks,
                               cudaStream_t st) {
#define TQ_CASE(VB, Q, N) \
  if (v_bits == VB && qjl == Q && nt == N) return attn_main_launch_t<KB, VB, Q, N, QOP>(a, query_only, bps, blocks, st);
  TQ_CASE(2, false, 1) TQ_CASE(2, false, 2) TQ_CASE(2, true, 1) TQ_CASE(2, true, 2)
  TQ_CASE(3, false, 1) TQ_CASE(3, false, 2) TQ_CASE(3, true, 1) TQ_CASE(3, true, 2)
  TQ_CASE(4, false, 1) TQ_CASE(4, false, 2) TQ_CASE(4, true, 1) TQ_CASE(4, true, 2)
#undef TQ_CASE
  return cudaErrorInvalidValue;
}

}  // namespace tq
