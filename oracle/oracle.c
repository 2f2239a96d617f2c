/*
 * oracle.c -- plain, slow, fp64 CPU oracle for TurboQuant-style KV-cache
 * compression (encode, decode, and attention over a compressed paged cache).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline / reference arm may load this library.  The
 * product path (libtq.so and its Python binding) never calls it, and it shares
 * no code, header, table or constant generator with the CUDA path.
 *
 * Every step follows the pages, in their order, one vector at a time:
 *
 *   "TurboQuant Family Design Study for CPU and Browser WASM KV Caches"
 *     - Capacity model (bytes per token 2*L*Hkv*d*s, M(T) with a W-token fp16
 *       window)                                           -> orc_page_layout
 *     - Why keys and values need different treatment (logit
 *       l_i = q.k_i/sqrt(d), p = softmax(l), o = sum p_i v_i) -> orc_attention
 *     - Placement relative to RoPE and attention (q.k = (Tq).(Tk) for an
 *       orthogonal T)                                     -> attention algebra
 *     - Dense and structured transform comparison (Rademacher signs then an
 *       FWHT, per head, from a seed)                      -> fwht, rotate
 *     - Packed format and complete bit accounting (section order inside a
 *       fixed-token page, 16-byte alignment)              -> orc_page_layout
 *   "From 0% to 100%: Debugging a KV Cache Compression Algorithm ..."
 *     - Why this caught my eye (random rotation, then a precomputed Lloyd-Max
 *       scalar quantizer per coordinate)                  -> orc_make_codebook
 *     - The QJL detective story (Gaussian S, dequant scale sqrt(pi/2)/d,
 *       unbiased inner products)                          -> qjl parts
 *     - Round 2, Bug 4 (an all-zero block encodes to a true zero block)
 *   aither-kvcache 2.4.0 README
 *     - Algorithm (normalize, rotate, quantize, pack, store packed bytes plus
 *       an fp32 norm; decoding reverses the steps)        -> encode/decode
 *     - Zero-buffer fused attention (rotate q once, score in the rotated
 *       domain, rotate back once)                         -> what the GPU does;
 *       the oracle instead materializes every token and takes the exact
 *       softmax, which is algebraically the same computation.
 *
 * Readings of points the pages leave open:
 *   - Codebook: Lloyd-Max for N(0,1), fp64 fixed-point iteration from a
 *     symmetric start, symmetrized, then stored at fp16 (each centroid
 *     rounded to the nearest fp16 value); the thresholds are the exact
 *     midpoints of neighbouring stored centroids.
 *   - u-domain: u = H (D . x) / ||x||, H the unnormalized Sylvester Hadamard
 *     matrix, so ||u||^2 = d and each u_j is close to N(0,1).
 *   - Quantizer: idx_j = #{k : t_k <= u_j} (ties go to the upper code).
 *   - QJL: residual in the unit-sphere rotated domain, e = (u - c[idx])/sqrt(d),
 *     gamma = ||e||, z_l = [(S e)_l >= 0]; dequant adds
 *     sqrt(pi/2)/m * gamma * S^T (2z - 1).
 *   - A zero vector stores n = 0, gamma = 0 and all codes / bits 0.
 *   - Bitstreams are LSB-first: code j occupies bits [j*b, j*b+b), sign l is
 *     bit l; byte k of the stream holds stream bits [8k, 8k+8).
 *   - Page body: the passage's section order, each section 16-byte aligned,
 *     pages of a multiple of 16 tokens and d a multiple of 16.  The value
 *     code section stores a group of 16 tokens chunk by chunk (16
 *     coordinates, 2*b bytes of each token), tokens in the order 0,1,8,9,
 *     2,3,10,11, 4,5,12,13, 6,7,14,15 (v_chunk_pos); for b = 2 and 4 the two
 *     tokens of an offset pair interleave their codes coordinate by
 *     coordinate inside their 4*b bytes (v_code_bit).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared oracle.c -lm   (no fast-math)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_RANGE (-2)

#define ORC_PI 3.14159265358979323846

typedef struct {
  int32_t head_dim, k_bits, v_bits, k_qjl, qjl_m, page_size, num_kv_heads;
  int32_t norm_correct; /* store n / ||y_hat|| (Bug 3 of the debugging post) */
  float qjl_scale;      /* factor of gamma S^T (2z - 1); 0: sqrt(pi/2) / m   */
  int32_t k_mixed;      /* keys at a fractional rate: b+1 bits on half the channels */
} orc_format;

/* Mixed-channel rates ("TurboQuant Family Design Study ...", 'Packed format
 * and complete bit accounting': 3.5 bits per channel = 64 channels at 4 bits
 * and 64 at 3; 2.5 = 64 at 3 and 64 at 2).  Which half carries the extra bit
 * is not fixed by the page; here channel j is a high channel when
 * (j mod 16) < 8.  A mixed code stream holds the high channels' codes first,
 * then the low channels', each in channel order and LSB-first. */
static int is_high_channel(int j) { return (j & 15) < 8; }

/* The QJL dequantization factor: the paper's sqrt(pi/2)/m for a Gaussian S
 * ("The QJL detective story"), or the format's own (an orthogonal S takes
 * sqrt(pi/2)/sqrt(d), times a shrinkage as in 'Testing it with an
 * ablation'). */
static double orc_qjl_coef(const orc_format *f) {
  return f->qjl_scale > 0.0f ? (double)f->qjl_scale : sqrt(ORC_PI / 2.0) / (double)f->qjl_m;
}

typedef struct {
  int64_t slab_bytes, page_bytes;
  int64_t k_norm, k_gamma, k_codes, k_signs, v_norm, v_codes;
  int32_t k_code_bytes, k_sign_bytes, v_code_bytes;
} orc_layout;

/* ------------------------------------------------------------------ fp16 -- */

/* IEEE binary16 bit pattern -> exact double. */
double orc_half_to_double(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x400), e - 25);
  return s ? -v : v;
}

/* ---------------------------------------------------------- Lloyd-Max ---- */

static double std_normal_pdf(double x) { return exp(-0.5 * x * x) / sqrt(2.0 * ORC_PI); }
/* Upper tail Q(x) = P(X > x), accurate in the far tail. */
static double upper_tail(double x) { return 0.5 * erfc(x / sqrt(2.0)); }
/* P(a < X < b) for X ~ N(0,1), written to avoid cancellation. */
static double cell_probability(double a, double b) {
  if (a >= 0.0) return upper_tail(a) - upper_tail(b);
  if (b <= 0.0) return upper_tail(-b) - upper_tail(-a);
  return 1.0 - upper_tail(b) - upper_tail(-a);
}

/*
 * Lloyd-Max scalar quantizer for N(0,1) with 2^bits levels, in fp64.
 * Fixed point: t_k = (c_k + c_{k+1})/2 and c_k = E[X | t_{k-1} < X < t_k]
 *            = (phi(t_{k-1}) - phi(t_k)) / (Phi(t_k) - Phi(t_{k-1})).
 * Returns the number of iterations used, or a negative error.
 */
int orc_lloyd_max_f64(int bits, double *c, double *t) {
  if (bits < 1 || bits > 8) return ORC_ERR_ARG;
  int L = 1 << bits;
  for (int k = 0; k < L; k++) c[k] = (k - 0.5 * (L - 1)) * (6.0 / L);
  int it;
  for (it = 1; it <= 200000; it++) {
    for (int k = 0; k + 1 < L; k++) t[k] = 0.5 * (c[k] + c[k + 1]);
    double delta = 0.0;
    for (int k = 0; k < L; k++) {
      double a = (k == 0) ? -INFINITY : t[k - 1];
      double b = (k == L - 1) ? INFINITY : t[k];
      double pa = (k == 0) ? 0.0 : std_normal_pdf(a);
      double pb = (k == L - 1) ? 0.0 : std_normal_pdf(b);
      double ck = (pa - pb) / cell_probability(a, b);
      double dd = fabs(ck - c[k]);
      if (dd > delta) delta = dd;
      c[k] = ck;
    }
    if (delta < 1e-15) break;
  }
  /* The start is symmetric, so the fixed point is too; remove rounding noise. */
  for (int k = 0; k < L / 2; k++) {
    double m = 0.5 * (c[L - 1 - k] - c[k]);
    c[k] = -m;
    c[L - 1 - k] = m;
  }
  for (int k = 0; k + 1 < L; k++) t[k] = 0.5 * (c[k] + c[k + 1]);
  return it;
}

/* The nearest IEEE binary16 value to x (ties to even), as a double; out of
 * range gives an infinity.  11 significant bits for normal values, a fixed
 * quantum of 2^-24 below 2^-14. */
double orc_round_to_half(double x) {
  if (x == 0.0 || !isfinite(x)) return x;
  int e;
  frexp(x, &e); /* |x| = m 2^e, m in [0.5, 1) */
  int q = e - 11;
  if (q < -24) q = -24;
  double r = ldexp(nearbyint(ldexp(x, -q)), q);
  if (fabs(r) > 65504.0) r = copysign(INFINITY, x);
  return r;
}

/*
 * The stored codebook: centroids [2^b] and decision thresholds [2^b - 1],
 * held as fp32 arrays.  The pages fix no storage precision for the
 * precomputed codebook; it is stored at fp16, the precision of the cache's
 * own dense data (the fp16 K/V and window): each centroid is the fp64
 * Lloyd-Max fixed point rounded to the nearest fp16 value, and each
 * threshold is the exact midpoint of two stored neighbours (representable in
 * fp32), so the quantizer stays the nearest-centroid rule of the table it
 * stores.  The fp16 rounding moves a centroid by at most 2^-12 of itself,
 * which changes the quantizer's MSE by about 1e-5 relative.
 */
int orc_make_codebook(int bits, float *centroids, float *midpoints) {
  double c[256], t[256];
  int it = orc_lloyd_max_f64(bits, c, t);
  if (it < 0) return it;
  int L = 1 << bits;
  for (int k = 0; k < L; k++) c[k] = orc_round_to_half(c[k]);
  for (int k = 0; k < L; k++) centroids[k] = (float)c[k];
  for (int k = 0; k + 1 < L; k++) midpoints[k] = (float)(0.5 * (c[k] + c[k + 1]));
  return it;
}

/* idx = #{k : t_k <= u}, t ascending (2^bits - 1 values). */
int orc_quantize_scalar(int bits, const float *midpoints, double u) {
  int L = 1 << bits, idx = 0;
  for (int k = 0; k + 1 < L; k++)
    if ((double)midpoints[k] <= u) idx++;
  return idx;
}

/* ------------------------------------------------------------- rotation -- */

static int is_pow2(int d) { return d >= 2 && (d & (d - 1)) == 0; }

/* In-place unnormalized Walsh-Hadamard transform, Sylvester (natural) order:
 * butterflies on pairs (i, i+h) for h = 1, 2, 4, ..., d/2. */
void orc_fwht(double *x, int d) {
  for (int h = 1; h < d; h <<= 1)
    for (int i = 0; i < d; i += 2 * h)
      for (int j = i; j < i + h; j++) {
        double a = x[j], b = x[j + h];
        x[j] = a + b;
        x[j + h] = a - b;
      }
}

/* sign_bit 1 means the coordinate is negated. */
static double rademacher(const uint8_t *signs, int j) { return signs[j] ? -1.0 : 1.0; }

/* Orthonormal structured rotation T x = H (D . x) / sqrt(d). */
void orc_rotate(int d, const uint8_t *signs, const double *x, double *y) {
  for (int j = 0; j < d; j++) y[j] = rademacher(signs, j) * x[j];
  orc_fwht(y, d);
  for (int j = 0; j < d; j++) y[j] /= sqrt((double)d);
}

/* Inverse: T^-1 y = D . (H y) / sqrt(d). */
void orc_unrotate(int d, const uint8_t *signs, const double *y, double *x) {
  for (int j = 0; j < d; j++) x[j] = y[j];
  orc_fwht(x, d);
  for (int j = 0; j < d; j++) x[j] = rademacher(signs, j) * x[j] / sqrt((double)d);
}

/* --------------------------------------------------------- one vector ---- */

int orc_decode_vector(int d, int bits, int qjl, int m, double norm, double gamma, const int32_t *idx,
                      const uint8_t *z, const uint8_t *signs, const float *centroids, const float *S,
                      double *out, double qjl_coef, int mixed, const float *lo_centroids);

/*
 * Encode one head vector x[d] (fp64 values of the fp16 input).
 * Outputs: *norm = ||x||, *gamma = ||e|| (QJL only), idx[d], z[m] (QJL only).
 * With norm_correct, *norm = ||x|| / ||y_hat|| instead, y_hat being the
 * unit-domain reconstruction of orc_decode_vector with factor qjl_coef, so
 * that the decoded vector has norm ||x|| ("From 0% to 100% ...", section
 * 'Round 2: the llama.cpp bug hunt', Bug 3: store original_norm /
 * reconstruction_norm).
 * Optional diagnostics (may be NULL): u[d] (u-domain coordinates),
 * code_margin[d] = min_k |u_j - t_k|, sign_margin[m] = |(S e)_l| / gamma.
 */
int orc_encode_vector(int d, int bits, int qjl, int m, const double *x, const uint8_t *signs,
                      const float *centroids, const float *midpoints, const float *S,
                      double *norm, double *gamma, int32_t *idx, uint8_t *z, double *u_out,
                      double *code_margin, double *sign_margin, int norm_correct, double qjl_coef,
                      int mixed, const float *lo_centroids, const float *lo_midpoints) {
  if (!is_pow2(d) || bits < 1 || bits > 8 || (qjl && m < 1) || (mixed && bits < 2)) return ORC_ERR_ARG;
  double *w = (double *)malloc(sizeof(double) * d);
  double *e = (double *)malloc(sizeof(double) * d);
  double ss = 0.0;
  for (int j = 0; j < d; j++) ss += x[j] * x[j];
  double n = sqrt(ss);
  *norm = n;
  if (qjl) *gamma = 0.0;
  if (n == 0.0) { /* true zero block */
    for (int j = 0; j < d; j++) {
      idx[j] = 0;
      if (u_out) u_out[j] = 0.0;
      if (code_margin) code_margin[j] = 0.0;
    }
    if (qjl)
      for (int l = 0; l < m; l++) {
        z[l] = 0;
        if (sign_margin) sign_margin[l] = 0.0;
      }
    free(w);
    free(e);
    return ORC_OK;
  }
  for (int j = 0; j < d; j++) w[j] = rademacher(signs, j) * x[j];
  orc_fwht(w, d);
  for (int j = 0; j < d; j++) {
    /* this channel's width and codebook: `bits` on high channels of a mixed
       kind (and on every channel otherwise), bits - 1 on its low channels */
    const int lo = mixed && !is_high_channel(j);
    const int bj = lo ? bits - 1 : bits, Lj = 1 << bj;
    const float *cj = lo ? lo_centroids : centroids, *tj = lo ? lo_midpoints : midpoints;
    double u = w[j] / n;
    idx[j] = orc_quantize_scalar(bj, tj, u);
    if (u_out) u_out[j] = u;
    if (code_margin) {
      double mg = INFINITY;
      for (int k = 0; k + 1 < Lj; k++) {
        double dd = fabs(u - (double)tj[k]);
        if (dd < mg) mg = dd;
      }
      code_margin[j] = mg;
    }
    e[j] = (u - (double)cj[idx[j]]) / sqrt((double)d);
  }
  if (qjl) {
    double g2 = 0.0;
    for (int j = 0; j < d; j++) g2 += e[j] * e[j];
    double g = sqrt(g2);
    *gamma = g;
    for (int l = 0; l < m; l++) {
      double p = 0.0;
      for (int j = 0; j < d; j++) p += (double)S[(int64_t)l * d + j] * e[j];
      z[l] = (p >= 0.0) ? 1 : 0;
      if (sign_margin) sign_margin[l] = (g > 0.0) ? fabs(p) / g : 0.0;
    }
  }
  if (norm_correct) {
    /* ||decode(norm = 1)|| = ||y_hat|| (H / sqrt(d) and the signs are orthogonal) */
    double *r = w;
    orc_decode_vector(d, bits, qjl, m, 1.0, qjl ? *gamma : 0.0, idx, z, signs, centroids, S, r, qjl_coef, mixed,
                      lo_centroids);
    double r2 = 0.0;
    for (int j = 0; j < d; j++) r2 += r[j] * r[j];
    if (r2 > 0.0) *norm = n / sqrt(r2);
  }
  free(w);
  free(e);
  return ORC_OK;
}

/*
 * Decode one head vector:
 *   y_hat = c[idx]/sqrt(d) + qjl_coef * gamma * S^T (2z - 1)   (QJL term optional;
 *           qjl_coef = sqrt(pi/2)/m in the paper's estimator)
 *   x_hat = norm * D . (H y_hat) / sqrt(d)
 */
int orc_decode_vector(int d, int bits, int qjl, int m, double norm, double gamma, const int32_t *idx,
                      const uint8_t *z, const uint8_t *signs, const float *centroids, const float *S,
                      double *out, double qjl_coef, int mixed, const float *lo_centroids) {
  if (!is_pow2(d) || bits < 1 || bits > 8 || (qjl && m < 1)) return ORC_ERR_ARG;
  double *y = (double *)malloc(sizeof(double) * d);
  for (int j = 0; j < d; j++)
    y[j] = (double)((mixed && !is_high_channel(j)) ? lo_centroids : centroids)[idx[j]] / sqrt((double)d);
  if (qjl) {
    double scale = qjl_coef * gamma;
    for (int j = 0; j < d; j++) {
      double acc = 0.0;
      for (int l = 0; l < m; l++) acc += (double)S[(int64_t)l * d + j] * (z[l] ? 1.0 : -1.0);
      y[j] += scale * acc;
    }
  }
  orc_fwht(y, d);
  for (int j = 0; j < d; j++) out[j] = norm * rademacher(signs, j) * y[j] / sqrt((double)d);
  free(y);
  return ORC_OK;
}

/* ------------------------------------------------------------ bitstreams -- */

/* LSB-first: value j occupies stream bits [j*b, j*b + b). */
void orc_pack_bits(int count, int b, const int32_t *vals, uint8_t *out) {
  int nbytes = (count * b + 7) / 8;
  memset(out, 0, (size_t)nbytes);
  for (int j = 0; j < count; j++)
    for (int i = 0; i < b; i++) {
      int bit = j * b + i;
      if ((vals[j] >> i) & 1) out[bit / 8] |= (uint8_t)(1u << (bit % 8));
    }
}

void orc_unpack_bits(int count, int b, const uint8_t *in, int32_t *vals) {
  for (int j = 0; j < count; j++) {
    int v = 0;
    for (int i = 0; i < b; i++) {
      int bit = j * b + i;
      v |= ((in[bit / 8] >> (bit % 8)) & 1) << i;
    }
    vals[j] = v;
  }
}

/* ---------------------------------------------------------- page layout -- */

/* One vector's code stream: LSB-first codes of every channel at `bits` bits,
 * or for a mixed kind the high channels' codes at `bits` bits followed by the
 * low channels' at bits - 1 (see is_high_channel). */
static void pack_codes(int d, int bits, int mixed, const int32_t *idx, uint8_t *out) {
  if (!mixed) {
    orc_pack_bits(d, bits, idx, out);
    return;
  }
  int32_t hi[d / 2], lo[d / 2];
  int nh = 0, nl = 0;
  for (int j = 0; j < d; j++) {
    if (is_high_channel(j)) hi[nh++] = idx[j];
    else lo[nl++] = idx[j];
  }
  orc_pack_bits(nh, bits, hi, out);
  orc_pack_bits(nl, bits - 1, lo, out + nh * bits / 8);
}

static void unpack_codes(int d, int bits, int mixed, const uint8_t *in, int32_t *idx) {
  if (!mixed) {
    orc_unpack_bits(d, bits, in, idx);
    return;
  }
  int32_t hi[d / 2], lo[d / 2];
  orc_unpack_bits(d / 2, bits, in, hi);
  orc_unpack_bits(d / 2, bits - 1, in + (d / 2) * bits / 8, lo);
  int nh = 0, nl = 0;
  for (int j = 0; j < d; j++) idx[j] = is_high_channel(j) ? hi[nh++] : lo[nl++];
}

static int64_t align16(int64_t x) { return (x + 15) / 16 * 16; }

/*
 * Byte position, inside the value-code section, of chunk r (coordinates
 * 16r .. 16r+15, i.e. bytes 2*vb*r .. 2*vb*r + 2*vb - 1 of the token's
 * bitstream) of the token at page offset `off`: groups of 16 tokens, inside a
 * group chunk-major, token i at slot 4*((i mod 8) div 2) + 2*(i div 8) + (i mod 2).
 */
static int64_t v_chunk_pos(int64_t off, int r, int d, int vb) {
  int64_t grp = off / 16;
  int i = (int)(off % 16);
  int slot = 4 * ((i % 8) / 2) + 2 * (i / 8) + (i % 2);
  int64_t token_bytes = (int64_t)d * vb / 8, chunk_bytes = 2 * vb;
  return grp * 16 * token_bytes + (int64_t)r * 16 * chunk_bytes + (int64_t)slot * chunk_bytes;
}

/*
 * Bit position, inside the value-code section, of bit k of the code of
 * coordinate j of the token at page offset `off`.  For 2- and 4-bit codes the
 * tokens of an offset pair (2p, 2p+1) share the 4*vb bytes of their two chunk
 * slots, as two bitstreams of vb-bit fields: the even coordinates first, then
 * the odd ones, and in each the two tokens' codes of one coordinate side by
 * side (even offset first).  Other widths keep each token's chunk whole.
 */
static int64_t v_code_bit(int64_t off, int j, int k, int d, int vb) {
  int r = j / 16, c = j % 16;
  if (vb == 2 || vb == 4) {
    int64_t pair = v_chunk_pos(off - off % 2, r, d, vb);
    return 8 * pair + (int64_t)(c % 2) * 16 * vb + (int64_t)(c / 2) * 2 * vb + (off % 2) * vb + k;
  }
  return 8 * v_chunk_pos(off, r, d, vb) + (int64_t)c * vb + k;
}

/* Writes the token's d codes (bits of nothing else change). */
static void put_v_codes(uint8_t *section, int64_t off, int d, int vb, const int32_t *idx) {
  for (int j = 0; j < d; j++)
    for (int k = 0; k < vb; k++) {
      int64_t bit = v_code_bit(off, j, k, d, vb);
      uint8_t m = (uint8_t)(1u << (bit % 8));
      if ((idx[j] >> k) & 1) section[bit / 8] |= m;
      else section[bit / 8] &= (uint8_t)~m;
    }
}

static void get_v_codes(const uint8_t *section, int64_t off, int d, int vb, int32_t *idx) {
  for (int j = 0; j < d; j++) {
    idx[j] = 0;
    for (int k = 0; k < vb; k++) {
      int64_t bit = v_code_bit(off, j, k, d, vb);
      idx[j] |= ((section[bit / 8] >> (bit % 8)) & 1) << k;
    }
  }
}

/*
 * One pool per layer: [num_pages][num_kv_heads] head-slabs.  Inside a slab,
 * the section order of the packed-format passage: K norms (fp32 [P]),
 * K QJL gammas (fp32 [P], QJL only), K codes ([P][d*kb/8]), K sign bits
 * ([P][m/8], QJL only), V norms (fp32 [P]), V codes (P*d*vb/8 bytes in
 * 16-token groups, see v_code_bit); every section starts on a 16-byte
 * boundary and the slab is padded to 16 bytes.  P and d are multiples of 16.
 */
int orc_page_layout(const orc_format *f, orc_layout *L) {
  if (!f || !L) return ORC_ERR_ARG;
  if (!is_pow2(f->head_dim) || f->head_dim % 16 || f->k_bits < 1 || f->k_bits > 8 || f->v_bits < 1 ||
      f->v_bits > 8 || f->page_size < 16 || f->page_size % 16 || f->num_kv_heads < 1)
    return ORC_ERR_ARG;
  if ((f->head_dim * f->k_bits) % 8 || (f->head_dim * f->v_bits) % 8) return ORC_ERR_ARG;
  if (f->k_qjl && (f->qjl_m < 8 || f->qjl_m % 8)) return ORC_ERR_ARG;
  if (f->k_mixed != 0 && f->k_mixed != 1) return ORC_ERR_ARG;
  if (f->k_mixed && f->k_bits + 1 > 8) return ORC_ERR_ARG;
  int64_t P = f->page_size, off = 0;
  /* mixed keys: d/2 channels at k_bits + 1 and d/2 at k_bits */
  L->k_code_bytes = f->k_mixed ? (f->head_dim / 2) * (2 * f->k_bits + 1) / 8 : f->head_dim * f->k_bits / 8;
  L->v_code_bytes = f->head_dim * f->v_bits / 8;
  L->k_sign_bytes = f->k_qjl ? f->qjl_m / 8 : 0;
  L->k_norm = off;
  off = align16(off + 4 * P);
  L->k_gamma = off;
  if (f->k_qjl) off = align16(off + 4 * P);
  L->k_codes = off;
  off = align16(off + P * L->k_code_bytes);
  L->k_signs = off;
  if (f->k_qjl) off = align16(off + P * L->k_sign_bytes);
  L->v_norm = off;
  off = align16(off + 4 * P);
  L->v_codes = off;
  off = align16(off + P * L->v_code_bytes);
  L->slab_bytes = off;
  L->page_bytes = off * f->num_kv_heads;
  return ORC_OK;
}

/* ------------------------------------------------------------ paged cache -- */

static void put_f32(uint8_t *p, float v) { memcpy(p, &v, 4); }
static float get_f32(const uint8_t *p) {
  float v;
  memcpy(&v, p, 4);
  return v;
}

/*
 * Encode N tokens x[N][H][d] (fp16 bits) of one kind (0 = K, 1 = V) into the
 * pool at slots slot_mapping[n] = page * P + offset (negative slot: skipped).
 * Diagnostics (nullable): u_out / code_margin [N][H][d], sign_margin [N][H][m].
 */
int orc_encode(const orc_format *f, int kind, const uint16_t *x, int64_t N, const int32_t *slot_mapping,
               uint8_t *pool, int64_t num_pages, const uint8_t *signs, const float *centroids,
               const float *midpoints, const float *S, double *u_out, double *code_margin,
               double *sign_margin) {
  orc_layout L;
  if (orc_page_layout(f, &L) != ORC_OK) return ORC_ERR_ARG;
  int d = f->head_dim, H = f->num_kv_heads, P = f->page_size;
  /* mixed keys: `centroids` / `midpoints` hold the k_bits + 1 codebook, then
     the k_bits one (the layout of the device codebooks) */
  int mixed = kind == 0 && f->k_mixed;
  int bits = kind == 0 ? f->k_bits + mixed : f->v_bits;
  const float *lo_c = mixed ? centroids + (1 << bits) : NULL;
  const float *lo_t = mixed ? midpoints + (1 << bits) - 1 : NULL;
  int qjl = (kind == 0) && f->k_qjl;
  int m = qjl ? f->qjl_m : 0;
  int code_bytes = L.k_code_bytes;
  double *xv = (double *)malloc(sizeof(double) * d);
  int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * d);
  uint8_t *z = (uint8_t *)malloc((size_t)(m > 0 ? m : 1));
  int32_t *zi = (int32_t *)malloc(sizeof(int32_t) * (m > 0 ? m : 1));
  int rc = ORC_OK;
  for (int64_t n = 0; n < N; n++) {
    int64_t slot = slot_mapping[n];
    if (slot < 0) continue;
    if (slot >= num_pages * P) {
      rc = ORC_ERR_RANGE;
      continue;
    }
    int64_t page = slot / P, off = slot % P;
    for (int h = 0; h < H; h++) {
      const uint16_t *src = x + (n * H + h) * d;
      for (int j = 0; j < d; j++) xv[j] = orc_half_to_double(src[j]);
      double norm = 0.0, gamma = 0.0;
      int64_t vh = n * H + h;
      orc_encode_vector(d, bits, qjl, m, xv, signs, centroids, midpoints, S, &norm, &gamma, idx, z,
                        u_out ? u_out + vh * d : NULL, code_margin ? code_margin + vh * d : NULL,
                        sign_margin ? sign_margin + vh * m : NULL, f->norm_correct, orc_qjl_coef(f), mixed, lo_c,
                        lo_t);
      uint8_t *slab = pool + page * L.page_bytes + (int64_t)h * L.slab_bytes;
      if (kind == 0) {
        put_f32(slab + L.k_norm + 4 * off, (float)norm);
        pack_codes(d, bits, mixed, idx, slab + L.k_codes + off * code_bytes);
        if (qjl) {
          put_f32(slab + L.k_gamma + 4 * off, (float)gamma);
          for (int l = 0; l < m; l++) zi[l] = z[l];
          orc_pack_bits(m, 1, zi, slab + L.k_signs + off * L.k_sign_bytes);
        }
      } else {
        put_f32(slab + L.v_norm + 4 * off, (float)norm);
        put_v_codes(slab + L.v_codes, off, d, bits, idx);
      }
    }
  }
  free(xv);
  free(idx);
  free(z);
  free(zi);
  return rc;
}

/* Decode the token stored at `slot`, head h, of one kind, into out[d]. */
static void decode_slot(const orc_format *f, const orc_layout *L, int kind, const uint8_t *pool,
                        int64_t slot, int h, const uint8_t *signs, const float *centroids, const float *S,
                        int32_t *idx, uint8_t *z, int32_t *zi, double *out) {
  int d = f->head_dim, P = f->page_size;
  int64_t page = slot / P, off = slot % P;
  const uint8_t *slab = pool + page * L->page_bytes + (int64_t)h * L->slab_bytes;
  if (kind == 0) {
    int qjl = f->k_qjl, m = qjl ? f->qjl_m : 0;
    int mixed = f->k_mixed, bits = f->k_bits + mixed;
    double norm = get_f32(slab + L->k_norm + 4 * off);
    unpack_codes(d, bits, mixed, slab + L->k_codes + off * L->k_code_bytes, idx);
    double gamma = 0.0;
    if (qjl) {
      gamma = get_f32(slab + L->k_gamma + 4 * off);
      orc_unpack_bits(m, 1, slab + L->k_signs + off * L->k_sign_bytes, zi);
      for (int l = 0; l < m; l++) z[l] = (uint8_t)zi[l];
    }
    orc_decode_vector(d, bits, qjl, m, norm, gamma, idx, z, signs, centroids, S, out, orc_qjl_coef(f), mixed,
                      mixed ? centroids + (1 << bits) : NULL);
  } else {
    double norm = get_f32(slab + L->v_norm + 4 * off);
    get_v_codes(slab + L->v_codes, off, d, f->v_bits, idx);
    orc_decode_vector(d, f->v_bits, 0, 0, norm, 0.0, idx, NULL, signs, centroids, NULL, out, 0.0, 0, NULL);
  }
}

/* Decode N slots of one kind into out[N][H][d] (fp64).  Negative slot: zeros. */
int orc_decode(const orc_format *f, int kind, const uint8_t *pool, int64_t num_pages, const int32_t *slot_mapping,
               int64_t N, const uint8_t *signs, const float *centroids, const float *S, double *out) {
  orc_layout L;
  if (orc_page_layout(f, &L) != ORC_OK) return ORC_ERR_ARG;
  int d = f->head_dim, H = f->num_kv_heads, m = f->k_qjl ? f->qjl_m : 1;
  int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * d);
  uint8_t *z = (uint8_t *)malloc((size_t)m);
  int32_t *zi = (int32_t *)malloc(sizeof(int32_t) * m);
  int rc = ORC_OK;
  for (int64_t n = 0; n < N; n++) {
    int64_t slot = slot_mapping[n];
    for (int h = 0; h < H; h++) {
      double *o = out + (n * H + h) * d;
      if (slot < 0 || slot >= num_pages * f->page_size) {
        if (slot >= 0) rc = ORC_ERR_RANGE;
        for (int j = 0; j < d; j++) o[j] = 0.0;
        continue;
      }
      decode_slot(f, &L, kind, pool, slot, h, signs, centroids, S, idx, z, zi, o);
    }
  }
  free(idx);
  free(z);
  free(zi);
  return rc;
}

/*
 * Decode-step attention over [compressed pages U fp16 window], exact softmax,
 * in the "materialize every token, then attend" form:
 *   l_i = q . k_hat_i / sqrt(d)      (window tokens use the raw fp16 k_i)
 *   o   = sum_i softmax(l)_i v_hat_i (window tokens use the raw fp16 v_i)
 * q: [B][Hq][d] fp16 bits; block_tables: [B][max_pages]; comp_lens[B] =
 * compressed tokens (positions [0, comp_len)); k_win/v_win: [B][Hkv][W][d]
 * fp16 bits with win_lens[B] valid tokens (may be NULL when W == 0).
 * heads (nullable): list of b*Hq + qh to compute; out is [n_heads][d] then,
 * else [B][Hq][d].  A block-table entry outside [0, num_pages) skips its page
 * and makes the call return ORC_ERR_RANGE.  No token at all gives o = 0.
 */
int orc_attention(const orc_format *f, int B, int Hq, const uint16_t *q, const uint8_t *pool, int64_t num_pages,
                  const int32_t *block_tables, int max_pages, const int32_t *comp_lens, const uint16_t *k_win,
                  const uint16_t *v_win, const int32_t *win_lens, int W, const uint8_t *k_signs,
                  const uint8_t *v_signs, const float *k_centroids, const float *v_centroids, const float *S,
                  const int32_t *heads, int n_heads, double *out) {
  orc_layout L;
  if (orc_page_layout(f, &L) != ORC_OK) return ORC_ERR_ARG;
  int d = f->head_dim, H = f->num_kv_heads, P = f->page_size;
  if (B < 1 || Hq < 1 || Hq % H) return ORC_ERR_ARG;
  int G = Hq / H, m = f->k_qjl ? f->qjl_m : 1;
  int total = heads ? n_heads : B * Hq;
  int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * d);
  uint8_t *z = (uint8_t *)malloc((size_t)m);
  int32_t *zi = (int32_t *)malloc(sizeof(int32_t) * m);
  double *qv = (double *)malloc(sizeof(double) * d);
  double *kh = (double *)malloc(sizeof(double) * d);
  double *vh = (double *)malloc(sizeof(double) * d);
  int rc = ORC_OK;
  for (int t = 0; t < total; t++) {
    int bq = heads ? heads[t] : t;
    int b = bq / Hq, qh = bq % Hq, h = qh / G;
    double *o = out + (int64_t)t * d;
    for (int j = 0; j < d; j++) {
      o[j] = 0.0;
      qv[j] = orc_half_to_double(q[((int64_t)b * Hq + qh) * d + j]);
    }
    int comp = comp_lens[b], win = (W > 0 && win_lens) ? win_lens[b] : 0;
    int ntok = comp + win;
    if (ntok <= 0) continue;
    /* pass 1: logits */
    double *logit = (double *)malloc(sizeof(double) * ntok);
    char *valid = (char *)malloc((size_t)ntok);
    double mx = -INFINITY;
    for (int i = 0; i < ntok; i++) {
      valid[i] = 1;
      if (i < comp) {
        int32_t pg = block_tables[(int64_t)b * max_pages + i / P];
        if (pg < 0 || pg >= num_pages) {
          valid[i] = 0;
          rc = ORC_ERR_RANGE;
          continue;
        }
        decode_slot(f, &L, 0, pool, (int64_t)pg * P + i % P, h, k_signs, k_centroids, S, idx, z, zi, kh);
      } else {
        const uint16_t *kw = k_win + (((int64_t)b * H + h) * W + (i - comp)) * d;
        for (int j = 0; j < d; j++) kh[j] = orc_half_to_double(kw[j]);
      }
      double s = 0.0;
      for (int j = 0; j < d; j++) s += qv[j] * kh[j];
      logit[i] = s / sqrt((double)d);
      if (logit[i] > mx) mx = logit[i];
    }
    /* pass 2: softmax-weighted values */
    double denom = 0.0;
    for (int i = 0; i < ntok; i++) {
      if (!valid[i]) continue;
      double p = exp(logit[i] - mx);
      denom += p;
      if (i < comp) {
        int32_t pg = block_tables[(int64_t)b * max_pages + i / P];
        decode_slot(f, &L, 1, pool, (int64_t)pg * P + i % P, h, v_signs, v_centroids, NULL, idx, z, zi, vh);
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
  free(idx);
  free(z);
  free(zi);
  free(qv);
  free(kh);
  free(vh);
  return rc;
}
