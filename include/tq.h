/*
 * tq.h -- C ABI of libtq.so: TurboQuant-style compressed KV cache on one
 * NVIDIA GB300 (sm_103a).  Encode (append) head vectors into a paged cache and
 * run fused decode attention directly on the packed pages.
 *
 * Conventions for every entry point
 *   - All device memory is allocated by the caller; the library allocates
 *     nothing and keeps no state between calls.
 *   - Device pointers must be valid on the CUDA device that is current on the
 *     calling thread.  Work is enqueued asynchronously on `stream` (a
 *     cudaStream_t; NULL means the legacy default stream).  Host pointers are
 *     read before the call returns.
 *   - No exception crosses the ABI.  Each call returns a tq_status.  Argument
 *     errors are detected on the host before anything is launched, and then
 *     nothing is launched.  TQ_ERR_CUDA reports a failed launch
 *     (cudaGetLastError after the launch).
 *   - Data errors that only the device can see (a slot or a block-table entry
 *     outside the pool, a length larger than its buffer) never trap: the
 *     kernel skips the offending token/page and ORs a TQ_DEVERR_* bit into
 *     the caller's optional int32 *err_word (device memory, may be NULL).
 *   - No kernel spins on another kernel or on a flag another block sets.  The
 *     one polled wait is inside the QJL key encode: a block waits, with a
 *     one-second limit, for its own tensor-core products (TQ_DEVERR_TIMEOUT).
 *
 * Format (tq_format): d = head_dim, b_K / b_V = bits per coordinate of the
 * Lloyd-Max codes, optional 1-bit QJL residual sketch of length m on keys,
 * P = page_size tokens per page, H = num_kv_heads.  A valid format has d a
 * power of two and a multiple of 16 and P a multiple of 16 (pages hold whole
 * 16-token groups).  The GPU kernels support d = 128, b in {2, 3, 4} (mixed
 * keys: k_bits in {2, 3}, i.e. 2.5 and 3.5 bits), m = 128, and no norm
 * correction on QJL keys; other valid shapes return TQ_ERR_UNSUPPORTED.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,   /* a null pointer, a negative size, inconsistent shapes */
  TQ_ERR_UNSUPPORTED = 2,   /* a valid format the GPU kernels do not implement    */
  TQ_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed               */
  TQ_ERR_DEVICE_FAULT = 4,  /* reserved: reported through err_word instead         */
  TQ_ERR_TIMEOUT = 5,       /* reserved: no kernel waits on another               */
  TQ_ERR_WORKSPACE = 6,     /* the workspace passed is smaller than required       */
  TQ_ERR_SCRATCH_LIMIT = 7  /* tq_decode_attn_static: the shape needs more scratch
                               than its fixed buffer (TQ_STATIC_SCRATCH_BYTES)    */
} tq_status;

/* Which stream of the cache a call works on. */
enum { TQ_KIND_K = 0, TQ_KIND_V = 1 };

/* Bits ORed into *err_word by the kernels. */
#define TQ_DEVERR_SLOT_RANGE 0x1   /* slot_mapping[n] >= num_pages * page_size          */
#define TQ_DEVERR_PAGE_RANGE 0x2   /* block_tables entry outside [0, num_pages)         */
#define TQ_DEVERR_LENGTH 0x4       /* comp_lens[b] > max_pages*P, win_lens[b] > window, or a negative length */
#define TQ_DEVERR_TIMEOUT 0x8      /* a bounded wait inside a kernel ran out (the tensor-core
                                      completion of the QJL key encode); that launch's sign
                                      words are incomplete                                 */

typedef struct {
  int32_t head_dim;     /* d                                                   */
  int32_t k_bits;       /* b_K, Lloyd-Max bits per key coordinate              */
  int32_t v_bits;       /* b_V, Lloyd-Max bits per value coordinate            */
  int32_t k_qjl;        /* 1: keys also store the QJL sign sketch and gamma    */
  int32_t qjl_m;        /* m, number of QJL sign bits per key                  */
  int32_t page_size;    /* P, tokens per page                                  */
  int32_t num_kv_heads; /* H, KV heads per layer                               */
  /* Variants of "From 0% to 100%: Debugging a KV Cache Compression
   * Algorithm ...", sections 'The QJL detective story', 'Testing it with an
   * ablation' and 'Round 2: the llama.cpp bug hunt' (Bug 3).  A zeroed
   * field keeps the paper's estimator. */
  int32_t norm_correct; /* 1: store n / ||y_hat|| instead of n, so that the
                           reconstruction keeps the input's norm (on the GPU:
                           not for keys with QJL)                           */
  float qjl_scale;      /* factor of gamma * S^T (2z - 1) in y_hat; 0 means
                           sqrt(pi/2)/m (Gaussian S).  An orthogonal S takes
                           sqrt(pi/2)/sqrt(d); a shrinkage a in (0, 1]
                           multiplies either (2/pi is the MMSE choice)      */
  int32_t k_mixed;      /* 1: keys at the fractional rate k_bits + 1/2: the
                           channels j with (j mod 16) < 8 take k_bits + 1
                           bits, the others k_bits ("TurboQuant Family Design
                           Study ...", 'Packed format and complete bit
                           accounting': 3.5 = 64 x 4 + 64 x 3 bits, 2.5 =
                           64 x 3 + 64 x 2).  A key's code stream holds the
                           high channels' codes first, then the low ones',
                           each LSB-first in channel order; the key codebook
                           argument is then the device codebook of k_bits + 1
                           followed by that of k_bits                        */
} tq_format;

/* Byte layout of one page (one pool per layer = [num_pages][H] head-slabs).
 * Section offsets are relative to the start of a head-slab; each section
 * starts on a 16-byte boundary.  Section order follows the page format of
 * "TurboQuant Family Design Study for CPU and Browser WASM KV Caches",
 * section 'Packed format and complete bit accounting': K norms fp32 [P],
 * K QJL gammas fp32 [P] (QJL only), K codes [P][d*b_K/8], K sign bits
 * [P][m/8] (QJL only), V norms fp32 [P], V codes (P*d*b_V/8 bytes, grouped
 * as below).  Codes are an LSB-first bitstream per token (code j at bits
 * [j*b, j*b+b)); sign bit l is bit l.  Token t of a page is at offset t of
 * every per-token section, except in the V codes section: there each token's
 * bitstream is cut into d/16 chunks of 16 coordinates (2*b_V bytes), and a
 * group of 16 tokens (offsets 16g .. 16g+15) is stored chunk by chunk: chunk r
 * of the token at offset 16g+i sits at byte
 *   g*16*(d*b_V/8) + r*16*(2*b_V) + s(i)*(2*b_V),
 *   s(i) = 4*((i mod 8) div 2) + 2*(i div 8) + (i mod 2)
 * (tokens in the order 0,1,8,9,2,3,10,11,4,5,12,13,6,7,14,15), so that the
 * attention kernel reads chunk r of the four tokens one thread multiplies in
 * one contiguous load.  For b_V = 2 and 4 the two tokens of an offset pair
 * (2p, 2p+1) share their two chunk slots (4*b_V bytes from the slot of 2p):
 * bit (c mod 2)*16*b_V + (c div 2)*2*b_V + (offset mod 2)*b_V + k holds bit k
 * of the code of chunk coordinate c, i.e. the even coordinates first, then
 * the odd ones, the pair's two codes of one coordinate side by side; the
 * attention kernel takes one 32-bit word of that as a tensor-core operand
 * register of both tokens.  Other widths keep each chunk as the token's own
 * stream.  An encode of one token of a pair leaves the partner's bits as they
 * were (the bits are set atomically unless both tokens come in one call in
 * order). */
typedef struct {
  int64_t slab_bytes, page_bytes;
  int64_t k_norm, k_gamma, k_codes, k_signs, v_norm, v_codes;
  int32_t k_code_bytes, k_sign_bytes, v_code_bytes; /* per token */
} tq_layout;

/* Human-readable text for a status (static storage). */
const char *tq_status_string(tq_status s);

/*
 * Lloyd-Max scalar quantizer for N(0, 1) with 2^bits levels (host only).
 * The precomputed Gaussian codebook of "From 0% to 100%: Debugging a KV Cache
 * Compression Algorithm on a 16GB MacBook", section 'Why this caught my eye',
 * applied to the unit-variance rotated coordinates.  fp64 fixed-point
 * iteration, rounded to fp32.  centroids: host float[2^bits], ascending;
 * midpoints: host float[2^bits - 1], ascending (decision thresholds).
 * bits in [1, 8].  The device codebook the other calls take is the
 * concatenation centroids || midpoints (2^(b+1) - 1 floats).  There is no
 * head_dim argument (build choice, no passage): the table quantizes the
 * unit-variance coordinates u = H(D x)/||x||, whose N(0, 1) law is the same
 * for every d, so one table serves every head size.
 */
tq_status tq_make_codebook(int bits, float *centroids, float *midpoints);

/* Page layout of a format (host only); see tq_layout. */
tq_status tq_page_layout(const tq_format *fmt, tq_layout *out);

/*
 * Encode (append) N tokens of one kind into the paged cache: for each head
 * vector x, n = ||x||, u = H (D . x) / n (signs D, unnormalized Sylvester
 * Hadamard H), code_j = #{k : t_k <= u_j}, then for keys with QJL:
 * e = (u - c[code]) / sqrt(d), gamma = ||e||, bit_l = [(S e)_l >= 0].
 * Follows the aither-kvcache README, section 'Algorithm', with the
 * structured rotation of the design study's 'Dense and structured transform
 * comparison' and the QJL sketch of the debugging post's 'The QJL detective
 * story'.  An all-zero vector stores n = 0, gamma = 0, all codes/bits 0.
 * Keys with QJL compute S e on the tensor cores in batches of 128 vectors
 * and wait for each batch's products with a time limit (one second); a wait
 * that runs out sets TQ_DEVERR_TIMEOUT and leaves the later sign words of
 * that launch unwritten.
 *   x_f16        device fp16 [N][H][d]
 *   slot_mapping device int32 [N]; token n goes to page slot/P, offset slot%P;
 *                a negative slot skips the token; two tokens with one slot
 *                in one call race (which one is stored is not defined).
 *                2- and 4-bit values are written fastest when tokens 2k and
 *                2k+1 go to offsets 2p and 2p+1 of one page (their shared
 *                words in one store, see tq_layout)
 *   page_pool    device bytes [num_pages * page_bytes], 16-byte aligned
 *   signs        device uint8 [d], 1 = negate coordinate (the kind's D)
 *   codebook     device fp32 [2^b + 2^b - 1] for this kind's b
 *   S            device fp32 [m][d] row-major (keys with QJL), else NULL
 *   err_word     device int32 or NULL (TQ_DEVERR_SLOT_RANGE; TQ_DEVERR_TIMEOUT
 *                for keys with QJL, see above)
 */
tq_status tq_encode(const tq_format *fmt, int kind, const void *x_f16, int64_t n_tokens,
                    const int32_t *slot_mapping, void *page_pool, int64_t num_pages,
                    const uint8_t *signs, const float *codebook, const float *S, int32_t *err_word,
                    void *stream);

/*
 * Append N tokens' keys and values in one call: the same result as
 * tq_encode(K, k_f16, ...) followed by tq_encode(V, v_f16, ...) with the same
 * slot_mapping (byte-identical pages).  A decode step appends both kinds of
 * the new token at once (aither-kvcache README, section 'Algorithm': keys and
 * values are compressed alike, each with its own rotation and codebook).
 * When k_bits == v_bits, keys carry no QJL sketch and are not mixed-rate,
 * this is one kernel launch; otherwise it is two launches, in this order, on
 * `stream`.
 *   k_f16, v_f16          device fp16 [N][H][d]
 *   k_signs, v_signs      device uint8 [d] (the kinds' D)
 *   k_codebook/v_codebook device fp32 codebooks for k_bits / v_bits
 *   S                     device fp32 [m][d] when fmt->k_qjl, else NULL
 * Argument rules and errors are those of tq_encode for each kind.
 */
tq_status tq_encode_kv(const tq_format *fmt, const void *k_f16, const void *v_f16, int64_t n_tokens,
                       const int32_t *slot_mapping, void *page_pool, int64_t num_pages, const uint8_t *k_signs,
                       const uint8_t *v_signs, const float *k_codebook, const float *v_codebook, const float *S,
                       int32_t *err_word, void *stream);

/*
 * Bytes of device workspace tq_append_window needs for `batch` sequences:
 * 0 (the tokens that leave the window are staged in shared memory).  Kept so
 * that callers size the workspace the same way as for tq_decode_attn.  Host
 * only.
 */
tq_status tq_append_window_workspace_size(const tq_format *fmt, int batch, size_t *bytes);

/*
 * One decode step's append for `batch` sequences, for a cache of compressed
 * pages plus an fp16 recent window of `window` tokens kept as a ring per
 * sequence.  Follows "TurboQuant Family Design Study for CPU and Browser WASM
 * KV Caches": 'Packed format and complete bit accounting' (the last W tokens
 * stay fp16 for K and V), 'Append cost and memory-bandwidth tradeoffs' (the
 * append runs once per generated token) and 'Paging, lifecycle, and cache
 * identity' (fixed pages filled in order).  Per sequence b:
 *   window == 0: the new token is encoded at compressed position comp_lens[b];
 *   win_lens[b] < window: the new token goes to ring slot win_lens[b], which
 *     then grows by one (win_head[b] stays 0 until the ring is full);
 *   otherwise: the token in ring slot win_head[b] (the oldest) is encoded at
 *     compressed position comp_lens[b], the new token takes that ring slot and
 *     win_head[b] advances by one modulo the window.
 * Compressed position c goes to physical page block_tables[b][c / P], offset
 * c % P: the caller allocates the page before the append that needs it.
 * Afterwards tq_decode_attn with the updated counters sees the new token
 * (attention does not depend on the order of the window's tokens).
 *   k_new_f16, v_new_f16  device fp16 [batch][H][d], the new token
 *   k_win_f16, v_win_f16  device fp16 [batch][H][window][d], updated in place
 *                         (NULL when window == 0)
 *   win_lens, win_head    device int32 [batch], updated in place (NULL when
 *                         window == 0)
 *   comp_lens             device int32 [batch], updated in place
 *   block_tables          device int32 [batch][max_pages]
 *   signs, codebooks, S   as for tq_encode_kv
 *   workspace             device, tq_append_window_workspace_size bytes (0:
 *                         may be NULL)
 * All counters are read and written on the device, so a step can be replayed
 * from a CUDA graph.  One kernel launch on `stream`: each block rolls the
 * windows of a group of sequences, encodes the keys and values that left
 * them and then advances their counters.  Host argument errors return before
 * any launch; more than 128 kv heads return TQ_ERR_UNSUPPORTED (a block holds
 * one sequence's tokens in shared memory).  A negative or out-of-range
 * counter (TQ_DEVERR_LENGTH), or a block table entry outside [0, num_pages)
 * (TQ_DEVERR_PAGE_RANGE), leaves that sequence untouched and sets the bit in
 * err_word.
 */
tq_status tq_append_window(const tq_format *fmt, int batch, const void *k_new_f16, const void *v_new_f16,
                           void *k_win_f16, void *v_win_f16, int window, int32_t *win_lens, int32_t *win_head,
                           int32_t *comp_lens, const int32_t *block_tables, int max_pages, void *page_pool,
                           int64_t num_pages, const uint8_t *k_signs, const uint8_t *v_signs, const float *k_codebook,
                           const float *v_codebook, const float *S, void *workspace, size_t workspace_bytes,
                           int32_t *err_word, void *stream);

/*
 * Decode N slots of one kind back to vectors (tests and offline use; never on
 * the attention path, which reads the packed pages directly).  Follows the
 * aither-kvcache README, section 'Algorithm' (decoding runs the encode's
 * steps backwards: centroid look-up, inverse rotation, rescale by the norm),
 * with the QJL reconstruction of "From 0% to 100%: Debugging a KV Cache
 * Compression Algorithm ...", section 'The QJL detective story':
 *   x_hat = n * D . (H y) / sqrt(d),
 *   y = c[code] / sqrt(d) + a * gamma * S^T (2 bits - 1)   (QJL keys),
 *   a = fmt->qjl_scale, or sqrt(pi/2)/m when qjl_scale is 0.
 *   page_pool    as for tq_encode; slot_mapping device int32 [N] (slot as in
 *                tq_encode); signs, codebook, S as for tq_encode
 *   out          device fp32 [N][H][d].  A negative slot gives zeros.
 *   err_word     device int32 or NULL (TQ_DEVERR_SLOT_RANGE: that slot gives
 *                zeros)
 */
tq_status tq_decode(const tq_format *fmt, int kind, const void *page_pool, int64_t num_pages,
                    const int32_t *slot_mapping, int64_t n_tokens, const uint8_t *signs,
                    const float *codebook, const float *S, float *out, int32_t *err_word, void *stream);

/*
 * Bytes of device workspace tq_decode_attn needs for these sizes on the
 * current device (depends on its SM count).  Host only.  Build choice, no
 * passage: the size is given by max_pages (block-table columns: the largest
 * compressed context is max_pages * P) and window (its fp16 partials) rather
 * than one max_ctx, because the two parts of the context have separate
 * scratch sections and the caller sizes both anyway.
 */
tq_status tq_decode_attn_workspace_size(const tq_format *fmt, int batch, int num_q_heads, int max_pages,
                                        int window, size_t *bytes);

/*
 * One decode step of attention over [compressed pages U fp16 recent window]:
 *   l_i = q . k_i / sqrt(d),  o = sum_i softmax(l)_i v_i
 * ("TurboQuant Family Design Study ...", section 'Why keys and values need
 * different treatment'), computed as in the aither-kvcache README section
 * 'Zero-buffer fused attention': q is rotated once into the key basis
 * (q.k = (Tq).(Tk), design study 'Placement relative to RoPE and attention'),
 * each compressed key is scored from its codes through the centroids plus the
 * QJL correction, values are accumulated in the rotated domain and rotated
 * back once per head.  No decoded copy of the cache is ever written.
 *   q_f16        device fp16 [B][Hq][d]; Hq = G * H (GQA, G <= 8)
 *   page_pool    as for tq_encode, but 32-byte aligned (the kernel reads
 *                32-byte runs of value codes in single requests)
 *   block_tables device int32 [B][max_pages]: logical page -> pool page
 *   comp_lens    device int32 [B]: compressed tokens (positions [0, comp_len))
 *   k_win_f16, v_win_f16  device fp16 [B][H][window][d] raw recent tokens,
 *                win_lens device int32 [B] valid window tokens (order free);
 *                all three may be NULL when window == 0
 *   k_signs, v_signs      device uint8 [d]; k_codebook, v_codebook as in
 *                tq_encode; S device fp32 [m][d] when fmt->k_qjl, else NULL
 *   out          device fp32 [B][Hq][d]; a head with no token at all gives 0
 *   workspace    device scratch of at least tq_decode_attn_workspace_size()
 *                bytes, 256-byte aligned; overwritten by every call, so calls
 *                that overlap on the GPU need separate workspaces
 *   err_word     device int32 or NULL (TQ_DEVERR_PAGE_RANGE / _LENGTH)
 * Stream order: the call's kernels are launched as programmatic dependents
 * of the kernel before them.  The first one reads q_f16, S and k_signs
 * before that kernel has completed when that kernel lets its dependents
 * launch early (as tq_append_window does once the work before it has
 * completed); everything else waits for it.  A kernel of the caller that
 * lets dependents launch early must have written those three by then.
 */
tq_status tq_decode_attn(const tq_format *fmt, int batch, int num_q_heads, const void *q_f16,
                         const void *page_pool, int64_t num_pages, const int32_t *block_tables,
                         int max_pages, const int32_t *comp_lens, const void *k_win_f16,
                         const void *v_win_f16, const int32_t *win_lens, int window,
                         const uint8_t *k_signs, const uint8_t *v_signs, const float *k_codebook,
                         const float *v_codebook, const float *S, float *out, void *workspace,
                         size_t workspace_bytes, int32_t *err_word, void *stream);

/*
 * tq_decode_attn, and additionally records two caller-created CUDA events
 * (cudaEvent_t, may be NULL) on `stream` immediately before and after the
 * split-KV main kernel, so a caller can time the dominant kernel in place
 * with cudaEventElapsedTime.  Same arguments, results and errors otherwise.
 */
tq_status tq_decode_attn_timed(const tq_format *fmt, int batch, int num_q_heads, const void *q_f16,
                               const void *page_pool, int64_t num_pages, const int32_t *block_tables,
                               int max_pages, const int32_t *comp_lens, const void *k_win_f16,
                               const void *v_win_f16, const int32_t *win_lens, int window,
                               const uint8_t *k_signs, const uint8_t *v_signs, const float *k_codebook,
                               const float *v_codebook, const float *S, float *out, void *workspace,
                               size_t workspace_bytes, int32_t *err_word, void *main_begin_event,
                               void *main_end_event, void *stream);

/*
 * tq_decode_attn without a workspace argument: the library's own scratch is
 * one fixed device buffer of TQ_STATIC_SCRATCH_BYTES per device, a static
 * array in the library image, so this call allocates nothing at all.  The
 * pages have no counterpart; it exists for callers that cannot hand over a
 * workspace: a plug-in that only receives tensor pointers from its host
 * framework and has no handle on that framework's allocator, or a loop that
 * must not call into any allocator.
 *   - Arguments, layouts, results and device-side errors are those of
 *     tq_decode_attn, minus workspace / workspace_bytes.
 *   - Every call looks up the buffer's address in the current context with
 *     cudaGetSymbolAddress (a host-side lookup once the library's module is
 *     loaded in that context, so a context created anew after
 *     cudaDeviceReset is found too).  The first call on a device, that
 *     device current, may load the module: make it before any stream
 *     capture.  A failed look-up returns TQ_ERR_CUDA.
 *   - The buffer is part of the library's device image: every device
 *     context that loads the module holds its 16 MiB until the process
 *     exits.  With lazy module loading (the CUDA default) that is a device
 *     on which a libtq kernel has run; with CUDA_MODULE_LOADING=EAGER it is
 *     every device the process touches after loading libtq.so, even if
 *     tq_decode_attn_static is never called.
 *   - The tensors must live on the device that is current on the calling
 *     thread: the buffer used is that device's.
 *   - A shape whose tq_decode_attn_workspace_size exceeds
 *     TQ_STATIC_SCRATCH_BYTES returns TQ_ERR_SCRATCH_LIMIT before anything
 *     is launched (16 MiB covers, e.g., B 16 x 32/8 heads at 32K context).
 *   - Nothing in the buffer has to start at zero: every call writes each
 *     scratch word it later reads.
 *   - All calls on one device share the buffer: two calls whose work
 *     overlaps in time (different streams, or threads without ordering)
 *     race and corrupt each other's results.  Order them on one stream.
 */
#define TQ_STATIC_SCRATCH_BYTES (16u << 20)
tq_status tq_decode_attn_static(const tq_format *fmt, int batch, int num_q_heads, const void *q_f16,
                                const void *page_pool, int64_t num_pages, const int32_t *block_tables,
                                int max_pages, const int32_t *comp_lens, const void *k_win_f16,
                                const void *v_win_f16, const int32_t *win_lens, int window,
                                const uint8_t *k_signs, const uint8_t *v_signs, const float *k_codebook,
                                const float *v_codebook, const float *S, float *out, int32_t *err_word,
                                void *stream);

/* ----------------------------------------------------------------------
 * KIVI-style control arm: asymmetric integer quantization of keys per
 * channel and of values per token, with the same fp16 recent window.
 * "TurboQuant Family Design Study for CPU and Browser WASM KV Caches",
 * section 'Candidate key and value algorithms', item 1 (Control baseline
 * arm), and its summary of KIVI in 'Why keys and values need different
 * treatment' (keys per channel, values per token).  No rotation: the cache
 * holds the raw-domain vectors.
 *
 * Quantizer of a group of fp16 values x (the same on every path): zero
 * z = min x, scale s = (max x - min x) / (2^b - 1), both stored as fp16 (s
 * rounded to nearest); the code of x is floor((x - z) / s + 1/2), clamped to
 * [0, 2^b - 1], decided in fp32 with the stored z and s; a zero scale gives
 * code 0.  Reconstruction z + s * code.  Key groups: one channel of one head
 * over the tokens of one page; value groups: one token-head over its d
 * channels.  Non-finite inputs give unspecified (but in-range) codes.
 * ---------------------------------------------------------------------- */
typedef struct {
  int32_t head_dim;     /* d                                     */
  int32_t k_bits;       /* b_K, bits per key code                */
  int32_t v_bits;       /* b_V, bits per value code              */
  int32_t page_size;    /* P, tokens per page (a multiple of 16) */
  int32_t num_kv_heads; /* H                                     */
} tq_kivi_format;

/* One pool per layer = [num_pages][H] head-slabs; per slab, each section
 * 16-byte aligned: K (scale, zero) fp16 pairs [d] (this page's per-channel
 * groups), K codes [P][d*b_K/8] (LSB-first per token), V (scale, zero) fp16
 * pairs [P], V codes (P*d*b_V/8 bytes in the grouped chunk order of
 * tq_layout's value section, each chunk the token's own LSB-first stream at
 * every width). */
typedef struct {
  int64_t slab_bytes, page_bytes;
  int64_t k_params, k_codes, v_params, v_codes;
  int32_t k_code_bytes, v_code_bytes; /* per token */
} tq_kivi_layout;

/* Layout of a KIVI format (host only).  The GPU kernels support d = 128 and
 * b_K, b_V in {2, 4}; other valid formats return TQ_ERR_UNSUPPORTED from the
 * device calls. */
tq_status tq_kivi_page_layout(const tq_kivi_format *fmt, tq_kivi_layout *out);

/*
 * Prefill keys into whole pages: x_f16 device fp16 [N][H][d] in token order;
 * token n goes to page page_ids[n / P], offset n % P (page_ids: device int32
 * [ceil(N / P)]).  Each page's tokens (the last page may hold N mod P) form
 * the per-channel groups.  A page id outside [0, num_pages) skips its group
 * and sets TQ_DEVERR_PAGE_RANGE in err_word (device int32 or NULL).
 */
tq_status tq_kivi_encode_keys(const tq_kivi_format *fmt, const void *k_f16, int64_t n_tokens, const int32_t *page_ids,
                              void *page_pool, int64_t num_pages, int32_t *err_word, void *stream);

/* Values, per token: v_f16 device fp16 [N][H][d], token n to slot
 * slot_mapping[n] (as tq_encode: negative skips, beyond the pool sets
 * TQ_DEVERR_SLOT_RANGE). */
tq_status tq_kivi_encode_values(const tq_kivi_format *fmt, const void *v_f16, int64_t n_tokens,
                                const int32_t *slot_mapping, void *page_pool, int64_t num_pages, int32_t *err_word,
                                void *stream);

/* Reconstruction z + s * code of N slots of one kind into out device fp32
 * [N][H][d] (tests and offline use; a negative slot gives zeros). */
tq_status tq_kivi_decode(const tq_kivi_format *fmt, int kind, const void *page_pool, int64_t num_pages,
                         const int32_t *slot_mapping, int64_t n_tokens, float *out, int32_t *err_word, void *stream);

/* Workspace bytes of tq_kivi_decode_attn (host only; depends on the current
 * device's SM count). */
tq_status tq_kivi_decode_attn_workspace_size(const tq_kivi_format *fmt, int batch, int num_q_heads, int max_pages,
                                             int window, size_t *bytes);

/*
 * One decode step of attention over [KIVI pages U fp16 recent window]:
 * l_i = q . k_hat_i / sqrt(d), o = sum_i softmax(l)_i v_hat_i, computed from
 * the codes on the tensor cores (keys: q scaled per page by the channel
 * scales against the integer codes, plus q . z; values: weights p * s against
 * the integer codes, plus sum p * z), split-KV with a log-sum-exp merge.  No
 * decoded copy of the cache is written.  Arguments, layouts and errors as
 * for tq_decode_attn, without signs, codebooks or S; the page pool must be
 * 32-byte aligned.
 */
tq_status tq_kivi_decode_attn(const tq_kivi_format *fmt, int batch, int num_q_heads, const void *q_f16,
                              const void *page_pool, int64_t num_pages, const int32_t *block_tables, int max_pages,
                              const int32_t *comp_lens, const void *k_win_f16, const void *v_win_f16,
                              const int32_t *win_lens, int window, float *out, void *workspace, size_t workspace_bytes,
                              int32_t *err_word, void *stream);

/* tq_kivi_decode_attn that also records two caller events (cudaEvent_t, may
 * be NULL) around its main kernel on `stream`, as tq_decode_attn_timed. */
tq_status tq_kivi_decode_attn_timed(const tq_kivi_format *fmt, int batch, int num_q_heads, const void *q_f16,
                                    const void *page_pool, int64_t num_pages, const int32_t *block_tables,
                                    int max_pages, const int32_t *comp_lens, const void *k_win_f16,
                                    const void *v_win_f16, const int32_t *win_lens, int window, float *out,
                                    void *workspace, size_t workspace_bytes, int32_t *err_word,
                                    void *main_begin_event, void *main_end_event, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
