// tq_api.cu -- the C ABI of libtq.so: argument checks, layout, codebook,
// decode-attention planning and kernel launches.
#include <math.h>
#include <string.h>

#include <mutex>

#include "tq_internal.cuh"

using namespace tq;

namespace {

// ------------------------------------------------------------------ format --
bool format_valid(const tq_format *f) {
  if (!f) return false;
  const int d = f->head_dim;
  if (d < 16 || (d & (d - 1))) return false;
  if (f->k_bits < 1 || f->k_bits > 8 || f->v_bits < 1 || f->v_bits > 8) return false;
  if ((d * f->k_bits) % 8 || (d * f->v_bits) % 8) return false;
  if (f->k_qjl != 0 && f->k_qjl != 1) return false;
  if (f->k_qjl && (f->qjl_m < 8 || f->qjl_m % 8)) return false;
  if (f->page_size < 16 || f->page_size % 16 || f->num_kv_heads < 1) return false;
  if (f->norm_correct != 0 && f->norm_correct != 1) return false;
  if (f->k_mixed != 0 && f->k_mixed != 1) return false;
  if (f->k_mixed && f->k_bits + 1 > 8) return false;
  if (!(f->qjl_scale >= 0.0f) || !isfinite(f->qjl_scale)) return false;
  return true;
}

// Factor of gamma * S^T (2z - 1) in y_hat: the format's, else sqrt(pi/2)/m.
float qjl_coef(const tq_format *f) {
  return f->qjl_scale > 0.0f ? f->qjl_scale : (float)(1.2533141373155003 / (double)f->qjl_m);
}

bool bits_supported(int b) { return b >= 2 && b <= 4; }

bool format_gpu_supported(const tq_format *f) {
  return f->head_dim == kD && bits_supported(f->k_bits) && bits_supported(f->k_bits + f->k_mixed) &&
         bits_supported(f->v_bits) &&
         (!f->k_qjl || f->qjl_m == kM) && f->page_size % kTile == 0;
}

int64_t round16(int64_t x) { return (x + 15) & ~int64_t(15); }

void compute_layout(const tq_format *f, tq_layout *L) {
  const int64_t P = f->page_size;
  // mixed keys: d/2 channels at k_bits + 1 and d/2 at k_bits
  L->k_code_bytes = f->k_mixed ? (f->head_dim / 2) * (2 * f->k_bits + 1) / 8 : f->head_dim * f->k_bits / 8;
  L->v_code_bytes = f->head_dim * f->v_bits / 8;
  L->k_sign_bytes = f->k_qjl ? f->qjl_m / 8 : 0;
  int64_t cursor = 0;
  L->k_norm = cursor;
  cursor = round16(cursor + 4 * P);
  L->k_gamma = cursor;
  if (f->k_qjl) cursor = round16(cursor + 4 * P);
  L->k_codes = cursor;
  cursor = round16(cursor + P * L->k_code_bytes);
  L->k_signs = cursor;
  if (f->k_qjl) cursor = round16(cursor + P * L->k_sign_bytes);
  L->v_norm = cursor;
  cursor = round16(cursor + 4 * P);
  L->v_codes = cursor;
  cursor = round16(cursor + P * L->v_code_bytes);
  L->slab_bytes = cursor;
  L->page_bytes = cursor * f->num_kv_heads;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

tq_status sm_count(int *sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TQ_ERR_CUDA;
  return TQ_OK;
}

// ---------------------------------------------------------------- codebook --
// Gaussian Lloyd-Max by iterating the decision thresholds: each threshold
// moves to the midpoint of the conditional means of its two neighbouring cells.
double gauss_pdf(double x) { return exp(-0.5 * x * x) * 0.39894228040143267794; }
double gauss_sf(double x) { return 0.5 * erfc(x * 0.70710678118654752440); }  // P(X > x)
double cell_mean(double lo, double hi) {
  const double flo = isinf(lo) ? 0.0 : gauss_pdf(lo), fhi = isinf(hi) ? 0.0 : gauss_pdf(hi);
  double mass;
  if (lo >= 0.0)
    mass = gauss_sf(lo) - gauss_sf(hi);
  else if (hi <= 0.0)
    mass = gauss_sf(-hi) - gauss_sf(-lo);
  else
    mass = 1.0 - gauss_sf(hi) - gauss_sf(-lo);
  return (flo - fhi) / mass;
}

void lloyd_max_thresholds(int bits, double *cent, double *thr) {
  const int levels = 1 << bits;
  for (int k = 0; k + 1 < levels; k++) thr[k] = 5.0 * ((k + 1.0) / levels - 0.5);
  for (int iter = 0; iter < 400000; iter++) {
    for (int k = 0; k < levels; k++) {
      const double lo = k == 0 ? -INFINITY : thr[k - 1];
      const double hi = k == levels - 1 ? INFINITY : thr[k];
      cent[k] = cell_mean(lo, hi);
    }
    double moved = 0.0;
    for (int k = 0; k + 1 < levels; k++) {
      const double nt = 0.5 * (cent[k] + cent[k + 1]);
      moved = fmax(moved, fabs(nt - thr[k]));
      thr[k] = nt;
    }
    if (moved < 1e-15) break;
  }
  for (int k = 0; k < levels; k++) {
    const double lo = k == 0 ? -INFINITY : thr[k - 1];
    const double hi = k == levels - 1 ? INFINITY : thr[k];
    cent[k] = cell_mean(lo, hi);
  }
  for (int k = 0; k < levels / 2; k++) {  // exact antisymmetry of a symmetric density
    const double m = 0.5 * (cent[levels - 1 - k] - cent[k]);
    cent[k] = -m;
    cent[levels - 1 - k] = m;
  }
  for (int k = 0; k + 1 < levels; k++) thr[k] = 0.5 * (cent[k] + cent[k + 1]);
}

// ---------------------------------------------------------- attention plan --
struct AttnPlan {
  int G, NT, nw_launch, blocks, slices;
  bool qop_keys, win_apart;
  size_t off_hdr, off_pre, off_clen, off_wlen, off_qrot, off_qop, off_qcst, off_qexp, off_segml, off_segacc, off_winml, off_winacc,
      off_mpart, off_mcnt, total;
};

// Fewest tiles per warp of the main kernel: one (a latency-bound shape gets
// as many warps as the machine holds; the wide merge's slices absorb the
// extra partials).
constexpr int kMinTilesPerWarp = 1;
// Up to this many tiles per warp (at the longest lengths the shape allows)
// the main kernel takes its key-score query operands ready-made from the
// prep kernel (the QOP instances); beyond it, it splits q_rot itself.
constexpr int64_t kQopMaxTilesPerWarp = 8;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

cudaError_t main_kernel_call(const tq_format *f, const AttnArgs &a, int nt, bool query, int *bps, int blocks,
                             cudaStream_t st) {
  const bool q = f->k_qjl != 0, o = a.qop_keys;
  if (f->k_mixed) {
    switch (f->k_bits) {
      case 2: return (o ? attn_main_k23_qop : attn_main_k23)(a, f->v_bits, q, nt, query, bps, blocks, st);
      case 3: return (o ? attn_main_k34_qop : attn_main_k34)(a, f->v_bits, q, nt, query, bps, blocks, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (f->k_bits) {
    case 2: return (o ? attn_main_k2_qop : attn_main_k2)(a, f->v_bits, q, nt, query, bps, blocks, st);
    case 3: return (o ? attn_main_k3_qop : attn_main_k3)(a, f->v_bits, q, nt, query, bps, blocks, st);
    case 4: return (o ? attn_main_k4_qop : attn_main_k4)(a, f->v_bits, q, nt, query, bps, blocks, st);
    default: return cudaErrorInvalidValue;
  }
}

// Occupancy of each main-kernel instance, per device (queried once).
std::mutex g_occ_mu;
int g_occ[64][5][3][2][2];  // [device][key widths][vb-2][qjl][nt-1]; 0 = unknown
int g_occ_kivi[64][5][3][2];  // KIVI main kernel: [device][kb-2][vb-2][nt-1]

tq_status plan_attention(const tq_format *f, int B, int Hq, int max_pages, int window, AttnPlan *p,
                         bool kivi = false) {
  const int H = f->num_kv_heads;
  p->G = Hq / H;
  p->NT = p->G <= 4 ? 1 : 2;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
  if (sm_count(&sms) != TQ_OK) return TQ_ERR_CUDA;
  int bps = 0;
  {
    std::lock_guard<std::mutex> lk(g_occ_mu);
    // key kinds 2, 3, 4, then 2.5, 3.5; KIVI keys in the QJL slot of kinds 2 and 4
    const int kw = f->k_mixed ? 3 + (f->k_bits - 2) : f->k_bits - 2;
    int *slot = dev < 64 ? &g_occ[dev][kw][f->v_bits - 2][kivi ? 1 : f->k_qjl][p->NT - 1] : nullptr;
    if (kivi && slot) slot = &g_occ_kivi[dev][kw][f->v_bits - 2][p->NT - 1];
    if (slot && *slot > 0) {
      bps = *slot;
    } else {
      AttnArgs dummy;
      memset(&dummy, 0, sizeof(dummy));
      const cudaError_t e = kivi ? kivi_main(dummy, f->k_bits, f->v_bits, p->NT, true, &bps, 0, 0)
                                 : main_kernel_call(f, dummy, p->NT, true, &bps, 0, 0);
      if (e != cudaSuccess) return TQ_ERR_CUDA;
      if (bps < 1) bps = 1;
      if (slot) *slot = bps;
    }
  }
  const int64_t tiles_max = (int64_t)B * H * max_pages * (f->page_size / kTile);
  int64_t warps = (tiles_max + kMinTilesPerWarp - 1) / kMinTilesPerWarp;
  const int wpb = kivi ? kivi_threads(p->NT) / 32 : attn_warps(p->NT, f->k_qjl != 0);
  const int64_t cap = (int64_t)sms * bps * wpb;
  if (warps > cap) warps = cap;
  if (warps < 1) warps = 1;
  p->blocks = (int)((warps + wpb - 1) / wpb);
  p->nw_launch = p->blocks * wpb;
  p->qop_keys = tiles_max <= kQopMaxTilesPerWarp * p->nw_launch;
  if (!kivi && p->qop_keys && bps == 1) {
    // Latency-bound shape: the main kernel is launched while the prep kernel
    // runs, and a CTA of one per SM cannot start on an SM that holds a prep
    // block until it completes; those CTAs would start late and set the
    // kernel's end.  Leave the prep kernel's SMs to it.
    const int64_t prep_blocks = (f->k_qjl ? (int64_t)B * Hq : ((int64_t)B * Hq + 3) / 4) +
                                (window > 0 ? (int64_t)B * H * ((window + kWinChunk - 1) / kWinChunk) : 0);
    const int64_t free_sms = sms - prep_blocks;
    if (p->blocks > free_sms && free_sms >= sms / 2) {
      p->blocks = (int)free_sms;
      p->nw_launch = p->blocks * wpb;
    }
  }
  // The window partials by their own kernel beside the main one when the
  // main grid leaves SMs to run it (latency-bound shapes): the prep kernel,
  // which the main kernel waits for, then only prepares the queries.
  p->win_apart = !kivi && p->qop_keys && window > 0 && bps == 1 && p->blocks < sms;

  const int64_t rows = (int64_t)B * Hq;
  const int64_t slots = (int64_t)p->nw_launch + (int64_t)B * H;
  size_t off = 0;
  p->off_hdr = off;    off = align256(off + sizeof(AttnHeader));
  p->off_pre = off;    off = align256(off + sizeof(int64_t) * (B + 1));
  p->off_clen = off;   off = align256(off + sizeof(int32_t) * B);
  p->off_wlen = off;   off = align256(off + sizeof(int32_t) * B);
  p->off_qrot = off;   off = align256(off + sizeof(float) * rows * kD);
  p->off_qop = off;    off = align256(off + sizeof(uint32_t) * rows * 4 * 64);
  p->off_qcst = off;   off = align256(off + sizeof(float2) * rows);
  p->off_qexp = off;   off = align256(off + sizeof(int32_t) * rows * 2);
  p->off_segml = off;  off = align256(off + sizeof(float) * slots * p->G * 2);
  p->off_segacc = off; off = align256(off + sizeof(float) * slots * p->G * kD);
  const int64_t nch = (window + kWinChunk - 1) / kWinChunk;
  p->off_winml = off;  off = align256(off + sizeof(float) * rows * nch * 2);
  p->off_winacc = off; off = align256(off + sizeof(float) * rows * nch * kD);
  p->slices = merge_slices(p->nw_launch, (int64_t)B * H);
  p->off_mpart = off;  off = align256(off + (p->slices > 1 ? sizeof(float) * rows * p->slices * kMergePartStride : 0));
  p->off_mcnt = off;   off = align256(off + sizeof(int32_t) * rows);
  p->total = off;
  return TQ_OK;
}

tq_status check_attn_shape(const tq_format *fmt, int B, int Hq, int max_pages, int window) {
  if (!format_valid(fmt) || B < 1 || Hq < 1 || max_pages < 1 || window < 0) return TQ_ERR_INVALID_ARG;
  if (Hq % fmt->num_kv_heads) return TQ_ERR_INVALID_ARG;
  if (!format_gpu_supported(fmt) || Hq / fmt->num_kv_heads > 8) return TQ_ERR_UNSUPPORTED;
  return TQ_OK;
}

}  // namespace

// ================================================================== ABI ====
extern "C" {

const char *tq_status_string(tq_status s) {
  switch (s) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARG: return "invalid argument";
    case TQ_ERR_UNSUPPORTED: return "unsupported format for the GPU kernels (need d=128, bits 2..4, m=128, page_size%16==0, G<=8)";
    case TQ_ERR_CUDA: return "CUDA runtime error";
    case TQ_ERR_DEVICE_FAULT: return "device-side data error (see err_word)";
    case TQ_ERR_TIMEOUT: return "timeout";
    case TQ_ERR_WORKSPACE: return "workspace too small";
    case TQ_ERR_SCRATCH_LIMIT: return "shape needs more scratch than the static buffer of tq_decode_attn_static holds";
  }
  return "unknown status";
}

tq_status tq_make_codebook(int bits, float *centroids, float *midpoints) {
  if (bits < 1 || bits > 8 || !centroids || (bits > 0 && !midpoints)) return TQ_ERR_INVALID_ARG;
  double c[256], t[256];
  lloyd_max_thresholds(bits, c, t);
  const int levels = 1 << bits;
  // stored at fp16: the nearest fp16 value of each centroid (ties to even);
  // the thresholds are then the exact midpoints of the stored neighbours
  for (int k = 0; k < levels; k++) {
    const double x = c[k];
    if (x != 0.0) {
      const int e = ilogb(x) < -14 ? -14 : ilogb(x);  // fp16 binade (subnormals share -14)
      const double quantum = ldexp(1.0, e - 10);      // 10 fraction bits
      c[k] = rint(x / quantum) * quantum;
    }
  }
  for (int k = 0; k < levels; k++) centroids[k] = (float)c[k];
  for (int k = 0; k + 1 < levels; k++) midpoints[k] = (float)(0.5 * (c[k] + c[k + 1]));
  return TQ_OK;
}

tq_status tq_page_layout(const tq_format *fmt, tq_layout *out) {
  if (!format_valid(fmt) || !out) return TQ_ERR_INVALID_ARG;
  compute_layout(fmt, out);
  return TQ_OK;
}

static tq_status encode_args(const tq_format *fmt, int kind, const void *x_f16, int64_t n_tokens,
                             const int32_t *slot_mapping, void *page_pool, int64_t num_pages, const uint8_t *signs,
                             const float *codebook, const float *S, int32_t *err_word, EncodeArgs *a) {
  if (!format_valid(fmt) || (kind != TQ_KIND_K && kind != TQ_KIND_V) || n_tokens < 0 || num_pages < 1)
    return TQ_ERR_INVALID_ARG;
  if (!format_gpu_supported(fmt)) return TQ_ERR_UNSUPPORTED;
  const bool qjl = kind == TQ_KIND_K && fmt->k_qjl;
  if (qjl && fmt->norm_correct) return TQ_ERR_UNSUPPORTED;  // would need S^T z per key in the encode
  if (!x_f16 || !slot_mapping || !page_pool || !signs || !codebook || (qjl && !S)) return TQ_ERR_INVALID_ARG;
  if (!aligned(x_f16, 16) || !aligned(page_pool, 16) || !aligned(slot_mapping, 4) || !aligned(codebook, 4) ||
      (qjl && !aligned(S, 16)))
    return TQ_ERR_INVALID_ARG;
  tq_layout L;
  compute_layout(fmt, &L);
  a->x = static_cast<const __half *>(x_f16);
  a->n_tokens = n_tokens;
  a->H = fmt->num_kv_heads;
  a->P = fmt->page_size;
  a->slot_mapping = slot_mapping;
  a->pool = static_cast<uint8_t *>(page_pool);
  a->num_pages = num_pages;
  a->page_bytes = L.page_bytes;
  a->slab_bytes = L.slab_bytes;
  a->norm_off = kind == TQ_KIND_K ? L.k_norm : L.v_norm;
  a->codes_off = kind == TQ_KIND_K ? L.k_codes : L.v_codes;
  a->gamma_off = L.k_gamma;
  a->signs_off = L.k_signs;
  a->code_bytes = kind == TQ_KIND_K ? L.k_code_bytes : L.v_code_bytes;
  a->grouped = kind == TQ_KIND_V;
  a->norm_correct = fmt->norm_correct != 0;
  a->signs = signs;
  a->codebook = codebook;
  a->S = S;
  a->err_word = err_word;
  return TQ_OK;
}

tq_status tq_encode(const tq_format *fmt, int kind, const void *x_f16, int64_t n_tokens, const int32_t *slot_mapping,
                    void *page_pool, int64_t num_pages, const uint8_t *signs, const float *codebook, const float *S,
                    int32_t *err_word, void *stream) {
  EncodeArgs a;
  tq_status s = encode_args(fmt, kind, x_f16, n_tokens, slot_mapping, page_pool, num_pages, signs, codebook, S, err_word, &a);
  if (s != TQ_OK) return s;
  if (n_tokens == 0) return TQ_OK;
  int sms = 0;
  if (sm_count(&sms) != TQ_OK) return TQ_ERR_CUDA;
  const bool mixed = kind == TQ_KIND_K && fmt->k_mixed;  // width below: the high channels'
  const int bits = kind == TQ_KIND_K ? fmt->k_bits + (mixed ? 1 : 0) : fmt->v_bits;
  const bool qjl = kind == TQ_KIND_K && fmt->k_qjl;
  return launch_encode(a, bits, qjl, mixed, sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TQ_OK
                                                                                                    : TQ_ERR_CUDA;
}

// K then V of one append: one launch when both kinds share a uniform bit
// width and keys carry no QJL sketch, else two.
static tq_status launch_kv(const tq_format *fmt, const EncodeArgs &ka, const EncodeArgs &va, void *stream) {
  int sms = 0;
  if (sm_count(&sms) != TQ_OK) return TQ_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (fmt->k_bits == fmt->v_bits && !fmt->k_qjl && !fmt->k_mixed)
    return launch_encode_kv(ka, va, fmt->k_bits, sms, st) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
  if (launch_encode(ka, fmt->k_bits + fmt->k_mixed, fmt->k_qjl != 0, fmt->k_mixed != 0, sms, st) != cudaSuccess)
    return TQ_ERR_CUDA;
  return launch_encode(va, fmt->v_bits, false, false, sms, st) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status tq_encode_kv(const tq_format *fmt, const void *k_f16, const void *v_f16, int64_t n_tokens,
                       const int32_t *slot_mapping, void *page_pool, int64_t num_pages, const uint8_t *k_signs,
                       const uint8_t *v_signs, const float *k_codebook, const float *v_codebook, const float *S,
                       int32_t *err_word, void *stream) {
  EncodeArgs ka, va;
  tq_status s = encode_args(fmt, TQ_KIND_K, k_f16, n_tokens, slot_mapping, page_pool, num_pages, k_signs, k_codebook, S,
                            err_word, &ka);
  if (s != TQ_OK) return s;
  s = encode_args(fmt, TQ_KIND_V, v_f16, n_tokens, slot_mapping, page_pool, num_pages, v_signs, v_codebook, nullptr,
                  err_word, &va);
  if (s != TQ_OK) return s;
  if (n_tokens == 0) return TQ_OK;
  return launch_kv(fmt, ka, va, stream);
}



tq_status tq_append_window_workspace_size(const tq_format *fmt, int batch, size_t *bytes) {
  if (!bytes || !format_valid(fmt) || batch < 0) return TQ_ERR_INVALID_ARG;
  *bytes = 0;  // the append stages its tokens in shared memory
  return TQ_OK;
}

tq_status tq_append_window(const tq_format *fmt, int batch, const void *k_new_f16, const void *v_new_f16,
                           void *k_win_f16, void *v_win_f16, int window, int32_t *win_lens, int32_t *win_head,
                           int32_t *comp_lens, const int32_t *block_tables, int max_pages, void *page_pool,
                           int64_t num_pages, const uint8_t *k_signs, const uint8_t *v_signs, const float *k_codebook,
                           const float *v_codebook, const float *S, void *workspace, size_t workspace_bytes,
                           int32_t *err_word, void *stream) {
  if (!format_valid(fmt) || batch < 0 || window < 0 || max_pages < 1 || num_pages < 1) return TQ_ERR_INVALID_ARG;
  if (!format_gpu_supported(fmt)) return TQ_ERR_UNSUPPORTED;
  if (num_pages > INT32_MAX / fmt->page_size) return TQ_ERR_UNSUPPORTED;  // page slots are int32
  if (fmt->num_kv_heads > 128) return TQ_ERR_UNSUPPORTED;                 // a sequence's tokens in one block
  if (!k_new_f16 || !v_new_f16 || !comp_lens || !block_tables) return TQ_ERR_INVALID_ARG;
  if (window > 0 && (!k_win_f16 || !v_win_f16 || !win_lens || !win_head)) return TQ_ERR_INVALID_ARG;
  if (!aligned(k_new_f16, 16) || !aligned(v_new_f16, 16) || !aligned(comp_lens, 4) ||
      !aligned(block_tables, 4) || (window > 0 && (!aligned(k_win_f16, 16) || !aligned(v_win_f16, 16) ||
                                                   !aligned(win_lens, 4) || !aligned(win_head, 4))))
    return TQ_ERR_INVALID_ARG;
  (void)workspace;  // no device workspace (tq_append_window_workspace_size is 0)
  (void)workspace_bytes;
  if (batch == 0) return TQ_OK;

  RollArgs r;
  r.k_new = static_cast<const __half *>(k_new_f16);
  r.v_new = static_cast<const __half *>(v_new_f16);
  r.k_win = static_cast<__half *>(k_win_f16);
  r.v_win = static_cast<__half *>(v_win_f16);
  r.B = batch;
  r.H = fmt->num_kv_heads;
  r.W = window;
  r.P = fmt->page_size;
  r.max_pages = max_pages;
  r.num_pages = num_pages;
  r.win_lens = win_lens;
  r.win_head = win_head;
  r.comp_lens = comp_lens;
  r.block_tables = block_tables;
  r.err_word = err_word;
  // the encodes of the tokens that leave the windows (their inputs and page
  // slots are set by the kernel, in shared memory); the arguments are checked
  // before anything is launched
  EncodeArgs ka, va;
  tq_status s = encode_args(fmt, TQ_KIND_K, r.k_new, batch, comp_lens, page_pool, num_pages, k_signs, k_codebook, S,
                            err_word, &ka);
  if (s != TQ_OK) return s;
  s = encode_args(fmt, TQ_KIND_V, r.v_new, batch, comp_lens, page_pool, num_pages, v_signs, v_codebook, nullptr,
                  err_word, &va);
  if (s != TQ_OK) return s;
  int sms = 0;
  if (sm_count(&sms) != TQ_OK) return TQ_ERR_CUDA;
  return launch_append(r, ka, va, fmt->k_bits + fmt->k_mixed, fmt->k_qjl != 0, fmt->k_mixed != 0, fmt->v_bits, sms,
                       static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? TQ_OK
             : TQ_ERR_CUDA;
}

tq_status tq_decode(const tq_format *fmt, int kind, const void *page_pool, int64_t num_pages,
                    const int32_t *slot_mapping, int64_t n_tokens, const uint8_t *signs, const float *codebook,
                    const float *S, float *out, int32_t *err_word, void *stream) {
  if (!format_valid(fmt) || (kind != TQ_KIND_K && kind != TQ_KIND_V) || n_tokens < 0 || num_pages < 1)
    return TQ_ERR_INVALID_ARG;
  if (!format_gpu_supported(fmt)) return TQ_ERR_UNSUPPORTED;
  const bool qjl = kind == TQ_KIND_K && fmt->k_qjl;
  if (!page_pool || !slot_mapping || !signs || !codebook || !out || (qjl && !S)) return TQ_ERR_INVALID_ARG;
  if (!aligned(page_pool, 16) || !aligned(out, 16) || (qjl && !aligned(S, 16))) return TQ_ERR_INVALID_ARG;
  if (n_tokens == 0) return TQ_OK;
  tq_layout L;
  compute_layout(fmt, &L);
  DecodeArgs a;
  a.pool = static_cast<const uint8_t *>(page_pool);
  a.n_tokens = n_tokens;
  a.H = fmt->num_kv_heads;
  a.P = fmt->page_size;
  a.slot_mapping = slot_mapping;
  a.num_pages = num_pages;
  a.page_bytes = L.page_bytes;
  a.slab_bytes = L.slab_bytes;
  a.norm_off = kind == TQ_KIND_K ? L.k_norm : L.v_norm;
  a.codes_off = kind == TQ_KIND_K ? L.k_codes : L.v_codes;
  a.gamma_off = L.k_gamma;
  a.signs_off = L.k_signs;
  a.code_bytes = kind == TQ_KIND_K ? L.k_code_bytes : L.v_code_bytes;
  a.grouped = kind == TQ_KIND_V;
  a.signs = signs;
  a.codebook = codebook;
  a.S = S;
  a.qjl_coef = qjl_coef(fmt);
  a.out = out;
  a.err_word = err_word;
  int sms = 0;
  if (sm_count(&sms) != TQ_OK) return TQ_ERR_CUDA;
  const bool mixed = kind == TQ_KIND_K && fmt->k_mixed;
  const int bits = kind == TQ_KIND_K ? fmt->k_bits + (mixed ? 1 : 0) : fmt->v_bits;
  return launch_decode(a, bits, qjl, mixed, sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TQ_OK
                                                                                                    : TQ_ERR_CUDA;
}

tq_status tq_decode_attn_workspace_size(const tq_format *fmt, int batch, int num_q_heads, int max_pages, int window,
                                        size_t *bytes) {
  if (!bytes) return TQ_ERR_INVALID_ARG;
  tq_status s = check_attn_shape(fmt, batch, num_q_heads, max_pages, window);
  if (s != TQ_OK) return s;
  AttnPlan p;
  s = plan_attention(fmt, batch, num_q_heads, max_pages, window, &p);
  if (s != TQ_OK) return s;
  *bytes = p.total;
  return TQ_OK;
}

static tq_status decode_attn_impl(const tq_format *fmt, int batch, int num_q_heads, const void *q_f16,
                                  const void *page_pool, int64_t num_pages, const int32_t *block_tables, int max_pages,
                                  const int32_t *comp_lens, const void *k_win_f16, const void *v_win_f16,
                                  const int32_t *win_lens, int window, const uint8_t *k_signs, const uint8_t *v_signs,
                                  const float *k_codebook, const float *v_codebook, const float *S, float *out,
                                  void *workspace, size_t workspace_bytes, int32_t *err_word, cudaEvent_t ev_begin,
                                  cudaEvent_t ev_end, void *stream) {
  tq_status s = check_attn_shape(fmt, batch, num_q_heads, max_pages, window);
  if (s != TQ_OK) return s;
  if (num_pages < 1 || !q_f16 || !page_pool || !block_tables || !comp_lens || !k_signs || !v_signs || !k_codebook ||
      !v_codebook || !out || !workspace || (fmt->k_qjl && !S))
    return TQ_ERR_INVALID_ARG;
  if (window > 0 && (!k_win_f16 || !v_win_f16 || !win_lens)) return TQ_ERR_INVALID_ARG;
  if (!aligned(q_f16, 8) || !aligned(page_pool, 32) || !aligned(workspace, 256) || !aligned(out, 4) ||
      (fmt->k_qjl && !aligned(S, 16)) || (window > 0 && (!aligned(k_win_f16, 16) || !aligned(v_win_f16, 16))))
    return TQ_ERR_INVALID_ARG;
  AttnPlan p;
  s = plan_attention(fmt, batch, num_q_heads, max_pages, window, &p);
  if (s != TQ_OK) return s;
  if (workspace_bytes < p.total) return TQ_ERR_WORKSPACE;

  tq_layout L;
  compute_layout(fmt, &L);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.pool = static_cast<const uint8_t *>(page_pool);
  a.num_pages = num_pages;
  a.page_bytes = L.page_bytes;
  a.slab_bytes = L.slab_bytes;
  a.k_norm_o = L.k_norm;
  a.k_gamma_o = L.k_gamma;
  a.k_codes_o = L.k_codes;
  a.k_signs_o = L.k_signs;
  a.v_norm_o = L.v_norm;
  a.v_codes_o = L.v_codes;
  a.k_code_bytes = L.k_code_bytes;
  a.v_code_bytes = L.v_code_bytes;
  a.B = batch;
  a.Hq = num_q_heads;
  a.H = fmt->num_kv_heads;
  a.G = p.G;
  a.P = fmt->page_size;
  a.max_pages = max_pages;
  a.window = window;
  a.block_tables = block_tables;
  a.comp_lens = comp_lens;
  a.q = static_cast<const __half *>(q_f16);
  a.k_win = static_cast<const __half *>(k_win_f16);
  a.v_win = static_cast<const __half *>(v_win_f16);
  a.win_lens = win_lens;
  a.k_signs = k_signs;
  a.v_signs = v_signs;
  a.k_cb = k_codebook;
  a.v_cb = v_codebook;
  a.S = S;
  a.qjl_coef = qjl_coef(fmt);
  a.out = out;
  a.err_word = err_word;
  a.hdr = reinterpret_cast<AttnHeader *>(ws + p.off_hdr);
  a.pre = reinterpret_cast<int64_t *>(ws + p.off_pre);
  a.clen = reinterpret_cast<int32_t *>(ws + p.off_clen);
  a.wlen = reinterpret_cast<int32_t *>(ws + p.off_wlen);
  a.q_rot = reinterpret_cast<float *>(ws + p.off_qrot);
  a.q_op = reinterpret_cast<uint32_t *>(ws + p.off_qop);
  a.q_cst = reinterpret_cast<float2 *>(ws + p.off_qcst);
  a.q_exp = reinterpret_cast<int32_t *>(ws + p.off_qexp);
  a.seg_ml = reinterpret_cast<float *>(ws + p.off_segml);
  a.seg_acc = reinterpret_cast<float *>(ws + p.off_segacc);
  a.win_ml = reinterpret_cast<float *>(ws + p.off_winml);
  a.win_acc = reinterpret_cast<float *>(ws + p.off_winacc);
  a.nw_launch = p.nw_launch;
  a.min_tiles = kMinTilesPerWarp;
  a.merge_slices = p.slices;
  a.qop_keys = p.qop_keys;
  a.win_apart = p.win_apart;
  a.merge_part = reinterpret_cast<float *>(ws + p.off_mpart);
  a.merge_cnt = reinterpret_cast<int32_t *>(ws + p.off_mcnt);
  // prep, main and merge start as programmatic dependents (their launches and
  // prologues overlap the previous kernel; prep waits before it reads
  // anything), except when the caller times the main kernel
  a.pdl = ev_begin == nullptr && ev_end == nullptr;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_attn_prep(a, fmt->k_qjl != 0, st) != cudaSuccess) return TQ_ERR_CUDA;
  if (ev_begin && cudaEventRecord(ev_begin, st) != cudaSuccess) return TQ_ERR_CUDA;
  if (main_kernel_call(fmt, a, p.NT, false, nullptr, p.blocks, st) != cudaSuccess) return TQ_ERR_CUDA;
  if (ev_end && cudaEventRecord(ev_end, st) != cudaSuccess) return TQ_ERR_CUDA;
  if (launch_attn_window(a, st) != cudaSuccess) return TQ_ERR_CUDA;
  if (launch_attn_merge(a, st) != cudaSuccess) return TQ_ERR_CUDA;
  return TQ_OK;
}

tq_status tq_decode_attn(const tq_format *fmt, int batch, int num_q_heads, const void *q_f16, const void *page_pool,
                         int64_t num_pages, const int32_t *block_tables, int max_pages, const int32_t *comp_lens,
                         const void *k_win_f16, const void *v_win_f16, const int32_t *win_lens, int window,
                         const uint8_t *k_signs, const uint8_t *v_signs, const float *k_codebook,
                         const float *v_codebook, const float *S, float *out, void *workspace, size_t workspace_bytes,
                         int32_t *err_word, void *stream) {
  return decode_attn_impl(fmt, batch, num_q_heads, q_f16, page_pool, num_pages, block_tables, max_pages, comp_lens,
                          k_win_f16, v_win_f16, win_lens, window, k_signs, v_signs, k_codebook, v_codebook, S, out,
                          workspace, workspace_bytes, err_word, nullptr, nullptr, stream);
}

tq_status tq_decode_attn_timed(const tq_format *fmt, int batch, int num_q_heads, const void *q_f16,
                               const void *page_pool, int64_t num_pages, const int32_t *block_tables, int max_pages,
                               const int32_t *comp_lens, const void *k_win_f16, const void *v_win_f16,
                               const int32_t *win_lens, int window, const uint8_t *k_signs, const uint8_t *v_signs,
                               const float *k_codebook, const float *v_codebook, const float *S, float *out,
                               void *workspace, size_t workspace_bytes, int32_t *err_word, void *main_begin_event,
                               void *main_end_event, void *stream) {
  return decode_attn_impl(fmt, batch, num_q_heads, q_f16, page_pool, num_pages, block_tables, max_pages, comp_lens,
                          k_win_f16, v_win_f16, win_lens, window, k_signs, v_signs, k_codebook, v_codebook, S, out,
                          workspace, workspace_bytes, err_word, static_cast<cudaEvent_t>(main_begin_event),
                          static_cast<cudaEvent_t>(main_end_event), stream);
}

}  // extern "C"

// ------------------------------------------------------------------ KIVI --
static bool kivi_format_valid(const tq_kivi_format *f) {
  if (!f) return false;
  const int d = f->head_dim;
  if (d < 16 || d > 256 || d % 16 || f->page_size < 16 || f->page_size % 16 || f->num_kv_heads < 1) return false;
  if (f->k_bits < 1 || f->k_bits > 8 || f->v_bits < 1 || f->v_bits > 8) return false;
  return true;
}
static bool kivi_gpu_supported(const tq_kivi_format *f) {
  return f->head_dim == kD && (f->k_bits == 2 || f->k_bits == 4) && (f->v_bits == 2 || f->v_bits == 4);
}
static void kivi_layout(const tq_kivi_format *f, tq_kivi_layout *L) {
  const int64_t d = f->head_dim, P = f->page_size;
  L->k_code_bytes = (int32_t)(d * f->k_bits / 8);
  L->v_code_bytes = (int32_t)(d * f->v_bits / 8);
  int64_t c = 0;
  L->k_params = c;
  c = round16(c + 4 * d);  // (scale, zero) fp16 pairs per channel
  L->k_codes = c;
  c = round16(c + P * L->k_code_bytes);
  L->v_params = c;
  c = round16(c + 4 * P);  // (scale, zero) fp16 pairs per token
  L->v_codes = c;
  c = round16(c + P * L->v_code_bytes);
  L->slab_bytes = c;
  L->page_bytes = c * f->num_kv_heads;
}
// The planner's view of a KIVI format (no QJL, no mixed rates).
static tq_format kivi_as_format(const tq_kivi_format *f) {
  tq_format g;
  memset(&g, 0, sizeof(g));
  g.head_dim = f->head_dim;
  g.k_bits = f->k_bits;
  g.v_bits = f->v_bits;
  g.page_size = f->page_size;
  g.num_kv_heads = f->num_kv_heads;
  return g;
}

static tq_status kivi_attn_impl(const tq_kivi_format *fmt, int batch, int num_q_heads, const void *q_f16,
                                const void *page_pool, int64_t num_pages, const int32_t *block_tables, int max_pages,
                                const int32_t *comp_lens, const void *k_win_f16, const void *v_win_f16,
                                const int32_t *win_lens, int window, float *out, void *workspace,
                                size_t workspace_bytes, int32_t *err_word, cudaEvent_t ev_begin, cudaEvent_t ev_end,
                                void *stream) {
  if (!kivi_format_valid(fmt) || batch < 1 || num_q_heads < 1 || max_pages < 1 || window < 0 ||
      num_q_heads % fmt->num_kv_heads)
    return TQ_ERR_INVALID_ARG;
  if (!kivi_gpu_supported(fmt) || num_q_heads / fmt->num_kv_heads > 8) return TQ_ERR_UNSUPPORTED;
  if (num_pages < 1 || !q_f16 || !page_pool || !block_tables || !comp_lens || !out || !workspace)
    return TQ_ERR_INVALID_ARG;
  if (window > 0 && (!k_win_f16 || !v_win_f16 || !win_lens)) return TQ_ERR_INVALID_ARG;
  if (!aligned(q_f16, 8) || !aligned(page_pool, 32) || !aligned(workspace, 256) || !aligned(out, 4) ||
      (window > 0 && (!aligned(k_win_f16, 16) || !aligned(v_win_f16, 16))))
    return TQ_ERR_INVALID_ARG;
  const tq_format pf = kivi_as_format(fmt);
  AttnPlan p;
  tq_status s = plan_attention(&pf, batch, num_q_heads, max_pages, window, &p, true);
  if (s != TQ_OK) return s;
  if (workspace_bytes < p.total) return TQ_ERR_WORKSPACE;
  tq_kivi_layout L;
  kivi_layout(fmt, &L);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.pool = static_cast<const uint8_t *>(page_pool);
  a.num_pages = num_pages;
  a.page_bytes = L.page_bytes;
  a.slab_bytes = L.slab_bytes;
  a.k_norm_o = L.k_params;  // (scale, zero) sections in the norm slots
  a.k_codes_o = L.k_codes;
  a.v_norm_o = L.v_params;
  a.v_codes_o = L.v_codes;
  a.k_code_bytes = L.k_code_bytes;
  a.v_code_bytes = L.v_code_bytes;
  a.B = batch;
  a.Hq = num_q_heads;
  a.H = fmt->num_kv_heads;
  a.G = p.G;
  a.P = fmt->page_size;
  a.max_pages = max_pages;
  a.window = window;
  a.block_tables = block_tables;
  a.comp_lens = comp_lens;
  a.q = static_cast<const __half *>(q_f16);
  a.k_win = static_cast<const __half *>(k_win_f16);
  a.v_win = static_cast<const __half *>(v_win_f16);
  a.win_lens = win_lens;
  a.out = out;
  a.err_word = err_word;
  a.hdr = reinterpret_cast<AttnHeader *>(ws + p.off_hdr);
  a.pre = reinterpret_cast<int64_t *>(ws + p.off_pre);
  a.clen = reinterpret_cast<int32_t *>(ws + p.off_clen);
  a.wlen = reinterpret_cast<int32_t *>(ws + p.off_wlen);
  a.q_rot = reinterpret_cast<float *>(ws + p.off_qrot);
  a.q_op = reinterpret_cast<uint32_t *>(ws + p.off_qop);
  a.q_cst = reinterpret_cast<float2 *>(ws + p.off_qcst);
  a.q_exp = reinterpret_cast<int32_t *>(ws + p.off_qexp);
  a.seg_ml = reinterpret_cast<float *>(ws + p.off_segml);
  a.seg_acc = reinterpret_cast<float *>(ws + p.off_segacc);
  a.win_ml = reinterpret_cast<float *>(ws + p.off_winml);
  a.win_acc = reinterpret_cast<float *>(ws + p.off_winacc);
  a.nw_launch = p.nw_launch;
  a.min_tiles = kMinTilesPerWarp;
  a.merge_slices = p.slices;
  a.qop_keys = p.qop_keys;
  a.win_apart = false;
  a.merge_part = reinterpret_cast<float *>(ws + p.off_mpart);
  a.merge_cnt = reinterpret_cast<int32_t *>(ws + p.off_mcnt);
  a.pdl = ev_begin == nullptr && ev_end == nullptr;
  a.raw = true;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_attn_prep(a, false, st) != cudaSuccess) return TQ_ERR_CUDA;
  if (ev_begin && cudaEventRecord(ev_begin, st) != cudaSuccess) return TQ_ERR_CUDA;
  if (kivi_main(a, fmt->k_bits, fmt->v_bits, p.NT, false, nullptr, p.blocks, st) != cudaSuccess) return TQ_ERR_CUDA;
  if (ev_end && cudaEventRecord(ev_end, st) != cudaSuccess) return TQ_ERR_CUDA;
  if (launch_attn_merge(a, st) != cudaSuccess) return TQ_ERR_CUDA;
  return TQ_OK;
}

extern "C" {

tq_status tq_kivi_page_layout(const tq_kivi_format *fmt, tq_kivi_layout *out) {
  if (!kivi_format_valid(fmt) || !out) return TQ_ERR_INVALID_ARG;
  kivi_layout(fmt, out);
  return TQ_OK;
}

static tq_status kivi_encode(const tq_kivi_format *fmt, int kind, const void *x_f16, int64_t n_tokens,
                             const int32_t *map, void *page_pool, int64_t num_pages, int32_t *err_word,
                             void *stream) {
  if (!kivi_format_valid(fmt) || n_tokens < 0 || num_pages < 1) return TQ_ERR_INVALID_ARG;
  if (!kivi_gpu_supported(fmt)) return TQ_ERR_UNSUPPORTED;
  if (!x_f16 || !map || !page_pool) return TQ_ERR_INVALID_ARG;
  if (!aligned(x_f16, 16) || !aligned(page_pool, 16) || !aligned(map, 4)) return TQ_ERR_INVALID_ARG;
  if (n_tokens == 0) return TQ_OK;
  tq_kivi_layout L;
  kivi_layout(fmt, &L);
  KiviEncodeArgs a;
  memset(&a, 0, sizeof(a));
  a.x = static_cast<const __half *>(x_f16);
  a.n_tokens = n_tokens;
  a.H = fmt->num_kv_heads;
  a.P = fmt->page_size;
  a.page_ids = kind == TQ_KIND_K ? map : nullptr;
  a.slot_mapping = kind == TQ_KIND_V ? map : nullptr;
  a.pool = static_cast<uint8_t *>(page_pool);
  a.num_pages = num_pages;
  a.page_bytes = L.page_bytes;
  a.slab_bytes = L.slab_bytes;
  a.params_off = kind == TQ_KIND_K ? L.k_params : L.v_params;
  a.codes_off = kind == TQ_KIND_K ? L.k_codes : L.v_codes;
  a.err_word = err_word;
  return launch_kivi_encode(a, kind, kind == TQ_KIND_K ? fmt->k_bits : fmt->v_bits, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? TQ_OK
             : TQ_ERR_CUDA;
}

tq_status tq_kivi_encode_keys(const tq_kivi_format *fmt, const void *k_f16, int64_t n_tokens, const int32_t *page_ids,
                              void *page_pool, int64_t num_pages, int32_t *err_word, void *stream) {
  return kivi_encode(fmt, TQ_KIND_K, k_f16, n_tokens, page_ids, page_pool, num_pages, err_word, stream);
}

tq_status tq_kivi_encode_values(const tq_kivi_format *fmt, const void *v_f16, int64_t n_tokens,
                                const int32_t *slot_mapping, void *page_pool, int64_t num_pages, int32_t *err_word,
                                void *stream) {
  return kivi_encode(fmt, TQ_KIND_V, v_f16, n_tokens, slot_mapping, page_pool, num_pages, err_word, stream);
}

tq_status tq_kivi_decode(const tq_kivi_format *fmt, int kind, const void *page_pool, int64_t num_pages,
                         const int32_t *slot_mapping, int64_t n_tokens, float *out, int32_t *err_word, void *stream) {
  if (!kivi_format_valid(fmt) || (kind != TQ_KIND_K && kind != TQ_KIND_V) || n_tokens < 0 || num_pages < 1)
    return TQ_ERR_INVALID_ARG;
  if (!kivi_gpu_supported(fmt)) return TQ_ERR_UNSUPPORTED;
  if (!page_pool || !slot_mapping || !out) return TQ_ERR_INVALID_ARG;
  if (!aligned(page_pool, 16) || !aligned(out, 16)) return TQ_ERR_INVALID_ARG;
  if (n_tokens == 0) return TQ_OK;
  tq_kivi_layout L;
  kivi_layout(fmt, &L);
  KiviDecodeArgs a;
  memset(&a, 0, sizeof(a));
  a.pool = static_cast<const uint8_t *>(page_pool);
  a.n_tokens = n_tokens;
  a.H = fmt->num_kv_heads;
  a.P = fmt->page_size;
  a.kind = kind;
  a.slot_mapping = slot_mapping;
  a.num_pages = num_pages;
  a.page_bytes = L.page_bytes;
  a.slab_bytes = L.slab_bytes;
  a.params_off = kind == TQ_KIND_K ? L.k_params : L.v_params;
  a.codes_off = kind == TQ_KIND_K ? L.k_codes : L.v_codes;
  a.out = out;
  a.err_word = err_word;
  return launch_kivi_decode(a, kind == TQ_KIND_K ? fmt->k_bits : fmt->v_bits, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? TQ_OK
             : TQ_ERR_CUDA;
}

tq_status tq_kivi_decode_attn_workspace_size(const tq_kivi_format *fmt, int batch, int num_q_heads, int max_pages,
                                             int window, size_t *bytes) {
  if (!bytes || !kivi_format_valid(fmt) || batch < 1 || num_q_heads < 1 || max_pages < 1 || window < 0 ||
      num_q_heads % fmt->num_kv_heads)
    return TQ_ERR_INVALID_ARG;
  if (!kivi_gpu_supported(fmt) || num_q_heads / fmt->num_kv_heads > 8) return TQ_ERR_UNSUPPORTED;
  const tq_format pf = kivi_as_format(fmt);
  AttnPlan p;
  const tq_status s = plan_attention(&pf, batch, num_q_heads, max_pages, window, &p, true);
  if (s != TQ_OK) return s;
  *bytes = p.total;
  return TQ_OK;
}

tq_status tq_kivi_decode_attn(const tq_kivi_format *fmt, int batch, int num_q_heads, const void *q_f16,
                              const void *page_pool, int64_t num_pages, const int32_t *block_tables, int max_pages,
                              const int32_t *comp_lens, const void *k_win_f16, const void *v_win_f16,
                              const int32_t *win_lens, int window, float *out, void *workspace, size_t workspace_bytes,
                              int32_t *err_word, void *stream) {
  return kivi_attn_impl(fmt, batch, num_q_heads, q_f16, page_pool, num_pages, block_tables, max_pages, comp_lens,
                        k_win_f16, v_win_f16, win_lens, window, out, workspace, workspace_bytes, err_word, nullptr,
                        nullptr, stream);
}

tq_status tq_kivi_decode_attn_timed(const tq_kivi_format *fmt, int batch, int num_q_heads, const void *q_f16,
                                    const void *page_pool, int64_t num_pages, const int32_t *block_tables,
                                    int max_pages, const int32_t *comp_lens, const void *k_win_f16,
                                    const void *v_win_f16, const int32_t *win_lens, int window, float *out,
                                    void *workspace, size_t workspace_bytes, int32_t *err_word,
                                    void *main_begin_event, void *main_end_event, void *stream) {
  return kivi_attn_impl(fmt, batch, num_q_heads, q_f16, page_pool, num_pages, block_tables, max_pages, comp_lens,
                        k_win_f16, v_win_f16, win_lens, window, out, workspace, workspace_bytes, err_word,
                        static_cast<cudaEvent_t>(main_begin_event), static_cast<cudaEvent_t>(main_end_event), stream);
}

}  // extern "C"
