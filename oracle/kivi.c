/*
 * kivi.c -- plain, slow CPU oracle of the KIVI-style control arm: asymmetric
 * (scale, zero) integer quantization of keys per channel and of values per
 * token, plus decode attention over such a cache with the fp16 recent window.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite and the benchmark's CPU
 * baseline may load this code (it is linked into liboracle.so with oracle.c).
 * The product path (libtq.so) never calls it and shares no code with it.
 *
 * It follows "TurboQuant Family Design Study for CPU and Browser WASM KV
 * Caches", section 'Candidate key and value algorithms', item 1 (Control
 * baseline arm: a KIVI-style per-channel K / per-token V asymmetric baseline
 * with an FP16 recent window), and the same study's summary of KIVI in
 * 'Why keys and values need different treatment' (keys quantized per channel,
 * values per token).  Readings of what the page leaves open:
 *   - Asymmetric quantizer of a group of values x: zero z = min x, scale
 *     s = (max x - min x) / (2^b - 1), code = round((x - z) / s) clamped to
 *     [0, 2^b - 1], reconstruction z + s * code.  z and s are stored as fp16
 *     (the precision of the cache's fp16 data).  The code is decided in fp32:
 *     t = (x - z) / s, code = floor(t + 1/2), with z and s the stored fp16
 *     values; s = fl32(fl32(max - min) / (2^b - 1)) rounded to fp16 (and
 *     held at 65504, the largest fp16, if it would overflow: only a 1-bit
 *     group can); a zero scale gives code 0.  A zero minimum is stored as +0.
 *   - Key groups: one channel over the tokens of one page of one head (P
 *     tokens; the last page of a prefill may hold fewer), so each page-head
 *     stores d (scale, zero) pairs.  Value groups: one token-head over its d
 *     channels.
 *   - Page body (per head-slab, each section 16-byte aligned): K (scale,
 *     zero) fp16 pairs [d], K codes [P][d*b_K/8] LSB-first per token, V
 *     (scale, zero) fp16 pairs [P], V codes [P*d*b_V/8] in the grouped order
 *     of the main format's value section (16-token groups, chunks of 16
 *     coordinates, tokens 0,1,8,9,2,3,10,11,...).
 *   - Attention works in the raw domain (no rotation): l_i = q . k_hat_i /
 *     sqrt(d) over the compressed tokens and the raw fp16 window, exact
 *     softmax, o = sum_i p_i v_hat_i.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KV_OK 0
#define KV_ERR_ARG (-1)
#define KV_ERR_RANGE (-2)

typedef struct {
  int32_t head_dim, k_bits, v_bits, page_size, num_kv_heads;
} kivi_format;

typedef struct {
  int64_t slab_bytes, page_bytes;
  int64_t k_params, k_codes, v_params, v_codes;
  int32_t k_code_bytes, v_code_bytes; /* per token */
} kivi_layout;

double orc_half_to_double(uint16_t h);  /* oracle.c */
double orc_round_to_half(double x);     /* oracle.c */

/* fp16 bit pattern of a value that is exactly representable in fp16. */
static uint16_t half_bits(double v) {
  uint16_t s = signbit(v) ? 0x8000u : 0u;
  double a = fabs(v);
  if (a == 0.0) return s;
  if (isinf(a)) return (uint16_t)(s | 0x7C00u);
  int e;
  double m = frexp(a, &e); /* a = m 2^e, m in [0.5, 1) */
  int ex = e - 1 + 15;     /* biased exponent of 1.f x 2^(e-1) */
  if (ex <= 0)             /* subnormal: a = k 2^-24 */
    return (uint16_t)(s | (uint16_t)llround(ldexp(a, 24)));
  uint16_t frac = (uint16_t)llround((2.0 * m - 1.0) * 1024.0);
  return (uint16_t)(s | (uint16_t)(ex << 10) | frac);
}

static int64_t align16(int64_t x) { return (x + 15) / 16 * 16; }

int orc_kivi_layout(const kivi_format *f, kivi_layout *L) {
  if (!f || !L) return KV_ERR_ARG;
  int d = f->head_dim, P = f->page_size;
  if (d < 16 || d > 256 || d % 16 || P < 16 || P % 16 || f->num_kv_heads < 1) return KV_ERR_ARG;
  if (f->k_bits < 1 || f->k_bits > 8 || f->v_bits < 1 || f->v_bits > 8) return KV_ERR_ARG;
  L->k_code_bytes = d * f->k_bits / 8;
  L->v_code_bytes = d * f->v_bits / 8;
  int64_t c = 0;
  L->k_params = c;
  c = align16(c + 4 * (int64_t)d);
  L->k_codes = c;
  c = align16(c + (int64_t)P * L->k_code_bytes);
  L->v_params = c;
  c = align16(c + 4 * (int64_t)P);
  L->v_codes = c;
  c = align16(c + (int64_t)P * L->v_code_bytes);
  L->slab_bytes = c;
  L->page_bytes = c * f->num_kv_heads;
  return KV_OK;
}

/*
 * Asymmetric b-bit quantization of the n fp16 values x[0], x[stride], ...:
 * stores the fp16 scale and zero and the n codes (see the readings above).
 */
void orc_kivi_quantize_group(int n, const uint16_t *x, int64_t stride, int bits, uint16_t *scale, uint16_t *zero,
                             int32_t *codes) {
  float mn = INFINITY, mx = -INFINITY;
  for (int i = 0; i < n; i++) {
    float v = (float)orc_half_to_double(x[(int64_t)i * stride]);
    if (v < mn) mn = v;
    if (v > mx) mx = v;
  }
  if (n == 0) mn = mx = 0.0f;
  const int top = (1 << bits) - 1;
  float diff = mx - mn;                           /* fp32 */
  float s32 = diff / (float)top;                  /* fp32 */
  double sh = orc_round_to_half((double)s32);     /* the stored scale */
  if (sh > 65504.0) sh = 65504.0;                 /* only 1-bit groups of range > 65504 */
  double zh = (double)(mn + 0.0f);                /* an fp16 value already; -0 becomes +0 */
  *scale = half_bits(sh);
  *zero = half_bits(zh);
  float sf = (float)sh, zf = (float)zh;
  for (int i = 0; i < n; i++) {
    float v = (float)orc_half_to_double(x[(int64_t)i * stride]);
    int code = 0;
    if (sf > 0.0f) {
      float t = (v - zf) / sf; /* fp32 */
      float r = floorf(t + 0.5f);
      code = r >= 0.0f ? (r > (float)top ? top : (int)r) : 0; /* NaN: 0 */
    }
    codes[i] = code;
  }
}

/* LSB-first bitstream of `count` codes of b bits. */
static void pack(int count, int b, const int32_t *vals, uint8_t *out) {
  memset(out, 0, (size_t)(count * b + 7) / 8);
  for (int j = 0; j < count; j++)
    for (int k = 0; k < b; k++)
      if ((vals[j] >> k) & 1) out[(j * b + k) >> 3] |= (uint8_t)(1u << ((j * b + k) & 7));
}
static void unpack(int count, int b, const uint8_t *in, int32_t *vals) {
  for (int j = 0; j < count; j++) {
    int32_t v = 0;
    for (int k = 0; k < b; k++) v |= ((in[(j * b + k) >> 3] >> ((j * b + k) & 7)) & 1) << k;
    vals[j] = v;
  }
}

/* Grouped value-code order of the main format: chunk r (coordinates
 * 16r..16r+15, 2*vb bytes of the token's stream) of the token at page offset
 * off, inside 16-token groups stored chunk by chunk. */
static int64_t v_chunk(int64_t off, int r, int d, int vb) {
  int64_t g = off / 16;
  int i = (int)(off % 16);
  int slot = 4 * ((i % 8) / 2) + 2 * (i / 8) + (i % 2);
  return g * 16 * (d * vb / 8) + (int64_t)r * 16 * (2 * vb) + slot * (2 * vb);
}

static void put16(uint8_t *p, uint16_t v) { memcpy(p, &v, 2); }
static uint16_t get16(const uint8_t *p) {
  uint16_t v;
  memcpy(&v, p, 2);
  return v;
}

/*
 * Keys: x[N][H][d] fp16 bits, tokens in order; token n goes to page
 * page_ids[n / P], offset n % P.  Each page's group (the P tokens, or the
 * N mod P of a last, partial page) is quantized per channel.  A page id
 * outside [0, num_pages) skips its group and returns KV_ERR_RANGE.
 */
int orc_kivi_encode_keys(const kivi_format *f, const uint16_t *x, int64_t N, const int32_t *page_ids,
                         uint8_t *pool, int64_t num_pages) {
  kivi_layout L;
  if (orc_kivi_layout(f, &L) != KV_OK || N < 0) return KV_ERR_ARG;
  const int d = f->head_dim, H = f->num_kv_heads, P = f->page_size, b = f->k_bits;
  int32_t *codes = (int32_t *)malloc(sizeof(int32_t) * (size_t)P * d);
  int32_t *tok = (int32_t *)malloc(sizeof(int32_t) * d);
  int32_t *col = (int32_t *)malloc(sizeof(int32_t) * P);
  int rc = KV_OK;
  for (int64_t g = 0; g * P < N; g++) {
    const int n = (int)((N - g * P) < P ? (N - g * P) : P);
    const int32_t pg = page_ids[g];
    if (pg < 0 || pg >= num_pages) {
      rc = KV_ERR_RANGE;
      continue;
    }
    for (int h = 0; h < H; h++) {
      uint8_t *slab = pool + (int64_t)pg * L.page_bytes + (int64_t)h * L.slab_bytes;
      for (int j = 0; j < d; j++) {
        uint16_t s, z;
        const uint16_t *x0 = x + ((g * P) * H + h) * (int64_t)d + j;
        orc_kivi_quantize_group(n, x0, (int64_t)H * d, b, &s, &z, col);
        put16(slab + L.k_params + 4 * j, s);
        put16(slab + L.k_params + 4 * j + 2, z);
        for (int i = 0; i < n; i++) codes[i * d + j] = col[i];
      }
      for (int i = 0; i < n; i++) {
        for (int j = 0; j < d; j++) tok[j] = codes[i * d + j];
        pack(d, b, tok, slab + L.k_codes + (int64_t)i * L.k_code_bytes);
      }
    }
  }
  free(codes);
  free(tok);
  free(col);
  return rc;
}

/*
 * Values: x[N][H][d] fp16 bits; token n goes to slot slot_mapping[n] =
 * page * P + offset (negative: skipped; beyond the pool: KV_ERR_RANGE).
 * Each token-head is quantized over its d channels.
 */
int orc_kivi_encode_values(const kivi_format *f, const uint16_t *x, int64_t N, const int32_t *slot_mapping,
                           uint8_t *pool, int64_t num_pages) {
  kivi_layout L;
  if (orc_kivi_layout(f, &L) != KV_OK || N < 0) return KV_ERR_ARG;
  const int d = f->head_dim, H = f->num_kv_heads, P = f->page_size, b = f->v_bits;
  int32_t *codes = (int32_t *)malloc(sizeof(int32_t) * d);
  uint8_t *stream = (uint8_t *)malloc((size_t)d);
  int rc = KV_OK;
  for (int64_t n = 0; n < N; n++) {
    const int32_t slot = slot_mapping[n];
    if (slot < 0) continue;
    if ((int64_t)slot >= num_pages * P) {
      rc = KV_ERR_RANGE;
      continue;
    }
    const int64_t pg = slot / P, off = slot % P;
    for (int h = 0; h < H; h++) {
      uint8_t *slab = pool + pg * L.page_bytes + (int64_t)h * L.slab_bytes;
      uint16_t s, z;
      orc_kivi_quantize_group(d, x + (n * H + h) * (int64_t)d, 1, b, &s, &z, codes);
      put16(slab + L.v_params + 4 * off, s);
      put16(slab + L.v_params + 4 * off + 2, z);
      pack(d, b, codes, stream);
      for (int r = 0; r < d / 16; r++)
        memcpy(slab + L.v_codes + v_chunk(off, r, d, b), stream + 2 * b * r, (size_t)(2 * b));
    }
  }
  free(codes);
  free(stream);
  return rc;
}

/* Reconstruction of the token at `slot`, head h, of one kind into out[d]. */
static void decode_slot(const kivi_format *f, const kivi_layout *L, int kind, const uint8_t *pool, int64_t slot,
                        int h, int32_t *codes, double *out) {
  const int d = f->head_dim, P = f->page_size;
  const int64_t pg = slot / P, off = slot % P;
  const uint8_t *slab = pool + pg * L->page_bytes + (int64_t)h * L->slab_bytes;
  if (kind == 0) {
    unpack(d, f->k_bits, slab + L->k_codes + off * L->k_code_bytes, codes);
    for (int j = 0; j < d; j++) {
      double s = orc_half_to_double(get16(slab + L->k_params + 4 * j));
      double z = orc_half_to_double(get16(slab + L->k_params + 4 * j + 2));
      out[j] = z + s * codes[j];
    }
  } else {
    uint8_t stream[256]; /* d * b_V / 8 <= 256: the layout rejects d > 256 */
    for (int r = 0; r < d / 16; r++)
      memcpy(stream + 2 * f->v_bits * r, slab + L->v_codes + v_chunk(off, r, d, f->v_bits), (size_t)(2 * f->v_bits));
    unpack(d, f->v_bits, stream, codes);
    double s = orc_half_to_double(get16(slab + L->v_params + 4 * off));
    double z = orc_half_to_double(get16(slab + L->v_params + 4 * off + 2));
    for (int j = 0; j < d; j++) out[j] = z + s * codes[j];
  }
}

/* Decode N slots of one kind into out[N][H][d] (fp64); negative slot: zeros. */
int orc_kivi_decode(const kivi_format *f, int kind, const uint8_t *pool, int64_t num_pages,
                    const int32_t *slot_mapping, int64_t N, double *out) {
  kivi_layout L;
  if (orc_kivi_layout(f, &L) != KV_OK) return KV_ERR_ARG;
  const int d = f->head_dim, H = f->num_kv_heads, P = f->page_size;
  int32_t *codes = (int32_t *)malloc(sizeof(int32_t) * d);
  int rc = KV_OK;
  for (int64_t n = 0; n < N; n++)
    for (int h = 0; h < H; h++) {
      double *o = out + (n * H + h) * (int64_t)d;
      const int32_t slot = slot_mapping[n];
      if (slot < 0 || (int64_t)slot >= num_pages * P) {
        if (slot >= 0) rc = KV_ERR_RANGE;
        for (int j = 0; j < d; j++) o[j] = 0.0;
        continue;
      }
      decode_slot(f, &L, kind, pool, slot, h, codes, o);
    }
  free(codes);
  return rc;
}

/*
 * Decode-step attention over [KIVI pages U fp16 window], materialized and
 * exact: l_i = q . k_hat_i / sqrt(d) (window: raw fp16 k_i), o = sum_i
 * softmax(l)_i v_hat_i.  Arguments and error rules as orc_attention's.
 */
int orc_kivi_attention(const kivi_format *f, int B, int Hq, const uint16_t *q, const uint8_t *pool,
                       int64_t num_pages, const int32_t *block_tables, int max_pages, const int32_t *comp_lens,
                       const uint16_t *k_win, const uint16_t *v_win, const int32_t *win_lens, int W,
                       const int32_t *heads, int n_heads, double *out) {
  kivi_layout L;
  if (orc_kivi_layout(f, &L) != KV_OK) return KV_ERR_ARG;
  const int d = f->head_dim, H = f->num_kv_heads, P = f->page_size;
  if (B < 1 || Hq < 1 || Hq % H) return KV_ERR_ARG;
  const int G = Hq / H, total = heads ? n_heads : B * Hq;
  int32_t *codes = (int32_t *)malloc(sizeof(int32_t) * d);
  double *qv = (double *)malloc(sizeof(double) * d);
  double *kh = (double *)malloc(sizeof(double) * d);
  double *vh = (double *)malloc(sizeof(double) * d);
  int rc = KV_OK;
  for (int t = 0; t < total; t++) {
    const int bq = heads ? heads[t] : t;
    const int b = bq / Hq, qh = bq % Hq, h = qh / G;
    double *o = out + (int64_t)t * d;
    for (int j = 0; j < d; j++) {
      o[j] = 0.0;
      qv[j] = orc_half_to_double(q[((int64_t)b * Hq + qh) * d + j]);
    }
    const int comp = comp_lens[b], win = (W > 0 && win_lens) ? win_lens[b] : 0, ntok = comp + win;
    if (ntok <= 0) continue;
    double *logit = (double *)malloc(sizeof(double) * ntok);
    char *valid = (char *)malloc((size_t)ntok);
    double mx = -INFINITY;
    for (int i = 0; i < ntok; i++) {
      valid[i] = 1;
      if (i < comp) {
        const int32_t pg = block_tables[(int64_t)b * max_pages + i / P];
        if (pg < 0 || pg >= num_pages) {
          valid[i] = 0;
          rc = KV_ERR_RANGE;
          continue;
        }
        decode_slot(f, &L, 0, pool, (int64_t)pg * P + i % P, h, codes, kh);
      } else {
        const uint16_t *kw = k_win + (((int64_t)b * H + h) * W + (i - comp)) * d;
        for (int j = 0; j < d; j++) kh[j] = orc_half_to_double(kw[j]);
      }
      double s = 0.0;
      for (int j = 0; j < d; j++) s += qv[j] * kh[j];
      logit[i] = s / sqrt((double)d);
      if (logit[i] > mx) mx = logit[i];
    }
    double denom = 0.0;
    for (int i = 0; i < ntok; i++) {
      if (!valid[i]) continue;
      const double p = exp(logit[i] - mx);
      denom += p;
      if (i < comp) {
        const int32_t pg = block_tables[(int64_t)b * max_pages + i / P];
        decode_slot(f, &L, 1, pool, (int64_t)pg * P + i % P, h, codes, vh);
      } else {
        const uint16_t *vw = v_win + (((int64_t)b * H + h) * W + (i - comp)) * d;
        for (int j = 0; j < d; j++) vh[j] = orc_half_to_double(vw[j]);
      }
      for (int j = 0; j < d; j++) o[j] += p * vh[j];
    }
    if (denom > 0.0)
      for (int j = 0; j < d; j++) o[j] /= denom;
    free(logit);
    free(valid);
  }
  free(codes);
  free(qv);
  free(kh);
  free(vh);
  return rc;
}
