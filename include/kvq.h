/*
 * kvq.h -- C ABI of the quantized KV-cache decode-attention library.
 *
 * The library implements the decode hot path of a transformer whose KV cache
 * is stored as group-wise asymmetric INT4/INT8 codes:
 *
 *   kvq_append       quantize new K/V vectors into the cache
 *                    ("What actually happens when you quantize a KV cache",
 *                    section 3 steps 2-5 and section 4: per group s =
 *                    (max-min)/(2^b-1), z = round(-min/s), q = clamp(round(x/s)
 *                    + z, 0, 2^b-1); two INT4 codes per byte, even channel in
 *                    the low nibble; fp16 scale and zero kept in their own
 *                    contiguous arrays);
 *   kvq_decode_attn  one decode row per query head over every cached token of
 *                    its sequence, the token just appended included
 *                    ("Quantization & inference optimisation", "Prefill, then
 *                    decode": append, then attend without a mask; "Serving
 *                    many users at once", batched decode_step with per-user
 *                    lengths and grouped-query heads), reading the codes and
 *                    dequantizing x_hat = (q - z) * s in registers
 *                    ("What actually happens ...", section 6).
 *
 * Conventions shared by every entry point:
 *   - Pointers marked "device" are CUDA device memory owned by the caller; the
 *     library never allocates, frees or retains them.  Arrays must be
 *     16-byte aligned.  fp16 data is passed as uint16_t (IEEE binary16 bits).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; nothing synchronizes.
 *   - Errors that the host can see (bad sizes, null pointers, unsupported
 *     shapes, too small a workspace) are returned synchronously and nothing
 *     is launched.  A failed launch returns KVQ_ERR_CUDA (with KVQ_VERBOSE
 *     set in the environment, the CUDA error's name also goes to stderr).
 *   - Errors that only the data reveals (a length beyond the cache, a bad
 *     block-table entry, a group the format cannot store) are OR-ed as
 *     KVQ_FLAG_* bits into *dev_status (a device uint32_t, may be NULL) and
 *     the offending unit is skipped as documented per call; read the word
 *     after the stream has synchronized.  No kernel traps or waits.
 *
 * Cache layouts (one instance for K, one for V; the same shapes for both):
 *   row_bytes = head_dim * bits / 8;  groups = head_dim / group_size
 *   codes: INT8 one per byte; INT4 two per byte, even channel in the low
 *   nibble; INT2 four per byte, channel 4m + k in bits 2k and 2k + 1.
 *   DENSE  codes  [batch][num_kv_heads][capacity][row_bytes]       uint8
 *          scale  [batch][num_kv_heads][capacity][groups]          fp16
 *          zero   same shape as scale
 *          token p of sequence b lives in slot p (0 <= p < capacity).
 *   PAGED  codes  [num_pages][num_kv_heads][page_size][row_bytes]   uint8
 *          scale, zero  [num_pages][num_kv_heads][page_size][groups]
 *          block_table [batch][max_blocks_per_seq] int32 (device);
 *          token p of sequence b lives in page block_table[b][p / page_size]
 *          at offset p % page_size.  Pages may be shared by sequences.
 *   bits == 16 stores the fp16 vectors themselves in the codes arrays
 *   (row_bytes = 2 * head_dim) and uses no scale/zero arrays.
 *   symmetric == 1 and nf4 == 1 use no zero arrays (k_zero, v_zero ignored).
 *
 * Axis-aware caches (k_per_channel == 1; "What actually happens when you
 * quantize a KV cache", section 3 step 7 and section 7: K grouped per
 * channel, V per token, the first tokens and the newest ones kept in fp16).
 * With S = sink_tokens, g = group_size, and L tokens cached:
 *   positions [0, min(S, L))          fp16 sinks, window slot p;
 *   block j covers [S + j g, S + (j+1) g), quantized once all g of its
 *     tokens have arrived: K codes in row p of k_codes with one scale and
 *     zero per channel for the block, V codes in row p of v_codes with
 *     per-token groups of g channels as in the default layout;
 *   the newest L - S - floor((L - S) / g) g tokens (fewer than g) form the
 *     fp16 residual window, slot S + (p - S) mod g.
 *   DENSE: capacity must be a multiple of g and larger than S.
 *          k_codes, v_codes  [batch][num_kv_heads][capacity][row_bytes]
 *          k_scale, k_zero   [batch][num_kv_heads][capacity / g][head_dim]
 *          v_scale, v_zero   [batch][num_kv_heads][capacity][head_dim / g]
 *          k_window, v_window [batch][num_kv_heads][S + g][head_dim] fp16
 *   PAGED: only the positions after the sinks are paged, by u = p - S:
 *     position p >= S lives in page block_table[b][u / capacity] at row
 *     u mod capacity, and block j's K headers in that page's row
 *     j mod (capacity / g).  capacity (tokens per page) must be a multiple
 *     of g, so that no block straddles two pages.  A sequence holds at most
 *     S + capacity * max_blocks_per_seq positions.  The window stays per
 *     sequence.
 *          k_codes, v_codes  [num_pages][num_kv_heads][capacity][row_bytes]
 *          k_scale, k_zero   [num_pages][num_kv_heads][capacity / g][head_dim]
 *          v_scale, v_zero   [num_pages][num_kv_heads][capacity][head_dim / g]
 *          k_window, v_window [batch][num_kv_heads][S + g][head_dim] fp16
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

/* Every entry point below is exported from the shared library; the library
 * is built with hidden default visibility, so nothing else is. */
#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned array      */
  KVQ_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head_dim 512) */
  KVQ_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required    */
  KVQ_ERR_CUDA = 4          /* a CUDA runtime call or launch failed          */
} kvq_status;

/* Largest batch of one decode call (and of one append on an axis-aware
 * cache): the kernels take the sequence from a grid dimension. */
#define KVQ_MAX_BATCH 65535

/* Bits OR-ed into the caller's device status word. */
#define KVQ_FLAG_SEQ_LEN      0x1u /* position/length outside the cache        */
#define KVQ_FLAG_BLOCK_TABLE  0x2u /* block-table entry outside [0,num_pages)  */
#define KVQ_FLAG_ZERO_CLAMPED 0x4u /* zero-point outside +-2048, clamped       */
#define KVQ_FLAG_NONFINITE    0x8u /* group held inf/NaN, stored as zeros      */
#define KVQ_FLAG_OOB          0x10u /* debug builds: an access outside its array
                                       was skipped (see kvq_debug_checks)      */

typedef enum { KVQ_DENSE = 0, KVQ_PAGED = 1 } kvq_layout;

typedef struct {
  int32_t bits;               /* 2, 4 or 8 (quantized), 16 (fp16 cache)       */
  int32_t group_size;         /* channels per group, multiple of 8, divides
                                 head_dim; ignored when bits == 16            */
  int32_t num_kv_heads;       /* >= 1                                          */
  int32_t head_dim;           /* 64, 128 or 256                                */
  int32_t layout;             /* kvq_layout                                    */
  int32_t capacity;           /* DENSE: token slots per sequence;
                                 PAGED: tokens per page (multiple of 8)        */
  int32_t num_pages;          /* PAGED only: pages in the pool                 */
  int32_t max_blocks_per_seq; /* PAGED only: row length of block_table         */
  int32_t symmetric;          /* 0: asymmetric, fp16 scale + zero per group;
                                 1: symmetric, fp16 scale only, codes offset
                                 by 2^(bits-1); must be 0 when bits == 16     */
  int32_t k_per_channel;      /* 1: axis-aware cache (bits 4/8,
                                 asymmetric): K grouped per channel over
                                 group_size consecutive tokens, V per token,
                                 fp16 sinks and residual window (see below)   */
  int32_t sink_tokens;        /* k_per_channel only: leading tokens kept fp16 */
  int32_t nf4;                /* 1: bits 4 coded as 16 normal-quantile levels
                                 with one fp16 absmax scale per group and no
                                 zero arrays (see kvq_append)                 */
} kvq_cache_desc;

typedef struct {              /* all device pointers, caller-owned             */
  void* k_codes;
  void* v_codes;
  uint16_t* k_scale;
  uint16_t* k_zero;
  uint16_t* v_scale;
  uint16_t* v_zero;
  const int32_t* block_table; /* PAGED only                                    */
  uint16_t* k_window;         /* k_per_channel only: fp16 sinks + residual     */
  uint16_t* v_window;
} kvq_cache;

/*
 * Bytes of K+V cache that `tokens` positions of ONE sequence occupy in one
 * layer: 2 * num_kv_heads * tokens * (row_bytes + 4 * groups), i.e. codes
 * plus a 4-byte fp16 scale+zero header per group ("What actually happens
 * when you quantize a KV cache", section 5; a symmetric or NF4 cache keeps
 * only the 2-byte scale; for bits == 16 the header is absent and this is
 * 2 * kv_heads * head_dim * 2 bytes per token, the formula of
 * "Quantization & inference optimisation", "What the cache costs").  Host
 * arithmetic only.  Returns 0 for an invalid descriptor.
 */
KVQ_API size_t kvq_cache_bytes(const kvq_cache_desc* desc, int64_t tokens);

/*
 * Bytes of each of k_window and v_window for `batch` sequences of an
 * axis-aware cache (batch * num_kv_heads * (sink_tokens + group_size) *
 * head_dim * 2); 0 for other caches or an invalid descriptor.
 */
KVQ_API size_t kvq_cache_window_bytes(const kvq_cache_desc* desc, int32_t batch);

/*
 * Allocation sizes for one layer's cache: *codes_bytes for each of k_codes
 * and v_codes, *header_bytes for each of k_scale, k_zero, v_scale, v_zero
 * (0 when bits == 16; a symmetric cache needs no zero arrays).  DENSE sizes
 * cover `batch` sequences of `capacity` slots; PAGED sizes cover num_pages
 * pages (`batch` is ignored).
 */
KVQ_API kvq_status kvq_cache_array_bytes(const kvq_cache_desc* desc, int32_t batch,
                                 size_t* codes_bytes, size_t* header_bytes);

/*
 * Quantize num_new new K and V vectors per sequence into the cache.
 *
 *   k_new, v_new     device fp16 [batch][num_new][num_kv_heads][head_dim]
 *   seq_lens_before  device int32 [batch]: tokens already cached; token t of
 *                    sequence b is written at position seq_lens_before[b]+t.
 *   dev_status       device uint32 (may be NULL)
 *
 * Per group of group_size consecutive channels of one vector: min and max;
 * s = fp16 rounded up from (max-min)/(2^bits-1) computed in fp64; z =
 * round-half-even(-min/s) in fp32, stored as an fp16 integer; codes
 * clamp(round-half-even(x/s) + z, 0, 2^bits-1) in fp32.  A constant group
 * stores s = |min| (1 if min == 0) so that it decodes exactly.  A zero-point
 * beyond +-2048 is clamped and flags KVQ_FLAG_ZERO_CLAMPED; a group with
 * inf/NaN is stored as s = z = 0, codes 0, and flags KVQ_FLAG_NONFINITE.
 * A position outside the cache (or an unmapped page) flags SEQ_LEN /
 * BLOCK_TABLE and that vector is not written.  Lengths are not modified:
 * the caller passes seq_lens_before + num_new to kvq_decode_attn.
 *
 * Symmetric caches (the zero-centred grid that "What actually happens when
 * you quantize a KV cache", section 3, compares against; the absmax
 * quantizer of "Serving many users at once", "Quantization: rounding the
 * weights"): per group a = max |x|; s = fp16 rounded up from
 * a/(2^(bits-1)-1) (s = 1 when a == 0); q = clamp(round-half-even(x/s),
 * -2^(bits-1), 2^(bits-1)-1) in fp32, stored as the code q + 2^(bits-1);
 * x_hat = (code - 2^(bits-1)) * s.  inf/NaN: s = 0, code 2^(bits-1), flagged.
 *
 * NF4 caches ("Gör inference billig", the NF4 paragraph: sixteen levels at
 * the quantiles of a normal distribution, block scaling): level i is the
 * (i + 1/2)/16 quantile of N(0, 1) divided by the outermost one, as fp16;
 * per group s = max |x| (an fp16 value, exact); the code is the level
 * nearest x/s (fp32 quotient, ties to the lower code); x_hat = level * s.
 * A group of zeros stores s = 0 (no level is 0); inf/NaN: s = 0, flagged;
 * codes are 0 where s = 0.
 *
 * Axis-aware caches: a token at a sink position or in the residual window is
 * stored as fp16.  When a token completes block j, the block is quantized
 * from the window and the new tokens: each K channel over the block's g
 * tokens, and each V token per group of g channels, with the formulas
 * above.  The tokens that remain in the residual window are then written
 * to their slots.  One call is two kernel launches, in stream order.
 * Axis-aware caches take at most KVQ_MAX_BATCH sequences per call (larger:
 * KVQ_ERR_UNSUPPORTED before any launch).
 */
KVQ_API kvq_status kvq_append(const kvq_cache_desc* desc, const kvq_cache* cache,
                      int32_t batch, int32_t num_new,
                      const uint16_t* k_new, const uint16_t* v_new,
                      const int32_t* seq_lens_before, uint32_t* dev_status,
                      void* stream);

/*
 * Number of context splits kvq_decode_attn uses.  num_splits > 0 is taken
 * as given (capped so that every split holds at least one token tile);
 * num_splits == 0 lets the library choose from the SM count of the current
 * device (needs a device; returns 0 if none is available).
 */
KVQ_API int32_t kvq_decode_num_splits(const kvq_cache_desc* desc, int32_t batch,
                              int32_t num_q_heads, int32_t max_seq_len,
                              int32_t num_splits);

/*
 * Workspace bytes kvq_decode_attn needs for these arguments (0 when the
 * work runs in one split).  Same num_splits convention as above.
 */
KVQ_API size_t kvq_decode_workspace_size(const kvq_cache_desc* desc, int32_t batch,
                                 int32_t num_q_heads, int32_t max_seq_len,
                                 int32_t num_splits);

/*
 * Decode attention for one new query per sequence and query head.
 *
 *   q            device fp16 [batch][num_q_heads][head_dim]
 *   seq_lens     device int32 [batch]: cached tokens to attend over, the one
 *                just appended included.  0 gives a zero output row.
 *   max_seq_len  host upper bound on every seq_lens[b]; sizes the splits.
 *   num_splits   0 = library choice, else the split count (see above).
 *   softmax_scale  0 -> 1/sqrt(head_dim).
 *   out          device fp16 [batch][num_q_heads][head_dim]
 *   workspace    device scratch of kvq_decode_workspace_size() bytes
 *                (may be NULL when that size is 0); contents need no init.
 *
 * num_q_heads must be a multiple of num_kv_heads; query head h reads KV head
 * h / (num_q_heads / num_kv_heads).  For each (b, h):
 *   out = softmax(scale * q . k_hat_j) weighted sum of v_hat_j, j < seq_lens[b]
 * with k_hat = (q_k - z) * s dequantized in registers, fp32 accumulation,
 * an online softmax over token tiles and, when split, a log-sum-exp merge of
 * the per-split partials.  A length below 0 or above min(max_seq_len,
 * cache capacity) flags KVQ_FLAG_SEQ_LEN and yields a zero row; a token whose
 * page is unmapped flags KVQ_FLAG_BLOCK_TABLE and is left out.  batch is at
 * most KVQ_MAX_BATCH (one grid row per sequence); a larger batch returns
 * KVQ_ERR_UNSUPPORTED before any launch.
 */
KVQ_API kvq_status kvq_decode_attn(const kvq_cache_desc* desc, const kvq_cache* cache,
                           int32_t batch, int32_t num_q_heads,
                           const uint16_t* q, const int32_t* seq_lens,
                           int32_t max_seq_len, int32_t num_splits,
                           float softmax_scale, uint16_t* out,
                           void* workspace, size_t workspace_bytes,
                           uint32_t* dev_status, void* stream);

/*
 * One decode step in one call: kvq_append of one token per sequence followed
 * by kvq_decode_attn over the lengths seq_lens_before + 1 ("What actually
 * happens when you quantize a KV cache", section 3: the new K/V vectors are
 * quantized on arrival and attention then reads the quantized cache, the new
 * token included).
 *
 *   k_new, v_new     device fp16 [batch][num_kv_heads][head_dim]
 *   seq_lens_before  device int32 [batch]: tokens cached before this step; the
 *                    new token is written at position seq_lens_before[b] and
 *                    seq_lens_before[b] + 1 tokens are attended.
 *   max_seq_len      host upper bound on every seq_lens_before[b] + 1.
 *   the rest         as for kvq_decode_attn (same workspace size for the same
 *                    batch, num_q_heads, max_seq_len and num_splits).
 *
 * Cache contents and status flags are those of kvq_append (num_new = 1)
 * followed by kvq_decode_attn: the codes, scales and zero-points written are
 * bit-identical.  out is the same attention; it can differ from the two-call
 * result in fp32 rounding.  For per-token caches that the tensor-core kernel
 * takes (bits 4 and 8 and NF4 at head_dim 64 / 128, bits 2 at head_dim 128,
 * at most 8 query heads per KV head) this is one kernel launch (plus the
 * merge when split): the thread block that owns the new position quantizes
 * the token, stores it, and adds its dequantized K/V to the attention
 * directly.  Axis-aware caches of those shapes (group_size a multiple of 32,
 * bits 4 or 8) are one launch too when the call runs with one split: each
 * thread block, which owns one (sequence, KV head), first quantizes the
 * block its token completes (when it completes one) or reads the token from
 * k_new / v_new where the window would hold it, and stores it to its fp16
 * slot after attending.  Other shapes, and axis-aware caches split over the
 * context, run the append kernels and the decode in sequence.  Lengths are
 * not modified.
 */
KVQ_API kvq_status kvq_append_decode_attn(const kvq_cache_desc* desc, const kvq_cache* cache,
                                  int32_t batch, int32_t num_q_heads,
                                  const uint16_t* k_new, const uint16_t* v_new,
                                  const uint16_t* q, const int32_t* seq_lens_before,
                                  int32_t max_seq_len, int32_t num_splits,
                                  float softmax_scale, uint16_t* out,
                                  void* workspace, size_t workspace_bytes,
                                  uint32_t* dev_status, void* stream);

/* Size of the library's own split scratch used by kvq_decode_attn_static_ws. */
#define KVQ_STATIC_WORKSPACE_BYTES ((size_t)8 << 20)

/*
 * kvq_decode_attn without a caller workspace: the split partials go to a
 * static device array of KVQ_STATIC_WORKSPACE_BYTES inside the library.
 * The pages have no counterpart to this call. It exists for callers that
 * cannot allocate device memory around a decode call, such as a plugin that
 * is handed only its input and output buffers, or code whose device
 * footprint must stay fixed after start-up.
 *
 * Arguments, results and status flags are those of kvq_decode_attn. The
 * workspace is the library's array.
 *
 *   - Set-up: the first call on each device, with that device current,
 *     looks up the array's device address (cudaGetSymbolAddress) and keeps
 *     it with the identifier of the device's current context. This may load
 *     the library's device code on that device. Make that first call before
 *     any stream capture. A later call in a different context (after
 *     cudaDeviceReset, say) looks the address up again, since the array then
 *     lives elsewhere; make that call before any capture as well.
 *   - Size limit: when kvq_decode_workspace_size() for the same arguments
 *     exceeds KVQ_STATIC_WORKSPACE_BYTES, the call returns KVQ_ERR_WORKSPACE
 *     before any launch. Pass a smaller num_splits, or use kvq_decode_attn.
 *   - Allocation: none. No cudaMalloc, no cudaFree, no allocating library
 *     routine.
 *   - Initial contents: nothing in the array has to start at zero. Each
 *     call writes every partial it reads.
 *   - Concurrency: one array serves every call on a device. Calls whose
 *     kernels can overlap on the GPU race on it and give wrong results. That
 *     covers calls on different streams without ordering between them, and
 *     calls from several host threads. Calls on one stream are safe.
 */
KVQ_API kvq_status kvq_decode_attn_static_ws(const kvq_cache_desc* desc, const kvq_cache* cache,
                                     int32_t batch, int32_t num_q_heads,
                                     const uint16_t* q, const int32_t* seq_lens,
                                     int32_t max_seq_len, int32_t num_splits,
                                     float softmax_scale, uint16_t* out,
                                     uint32_t* dev_status, void* stream);

/*
 * Debug builds.  build(debug=True) in quantized_kv_decode_gb300/build.py
 * compiles the same sources with KVQ_DEBUG defined into libkvq_debug.so,
 * which exports the same entry points.  There each launch carries the byte
 * extent of every caller array it may touch, derived on the host from the
 * descriptor and the call's sizes:
 *   cache arrays   kvq_cache_array_bytes(desc, batch) each (DENSE: the
 *                  call's batch of sequences; PAGED: num_pages), the
 *                  windows kvq_cache_window_bytes(desc, batch) each;
 *   block_table    batch * max_blocks_per_seq int32;
 *   q, out         batch * num_q_heads * head_dim fp16 each;
 *   k_new, v_new   batch * num_new * num_kv_heads * head_dim fp16 each;
 *   seq_lens / seq_lens_before   batch int32;
 *   workspace      workspace_bytes (the static array for the
 *                  _static_ws call).
 * Every global load and store of the kernels first checks that its bytes lie
 * inside the extent of the array it addresses.  An access that does not is
 * skipped (a load yields zeros), and KVQ_FLAG_OOB is OR-ed into *dev_status
 * (when dev_status is not NULL).  The checks cost time; results are otherwise
 * those of the release library, which never sets KVQ_FLAG_OOB.
 */

/* 1 when the loaded library is a debug build (bounds checks compiled in). */
KVQ_API int32_t kvq_debug_checks(void);

/* The caller arrays a debug build checks, named for kvq_debug_shrink_extent. */
typedef enum {
  KVQ_ARRAY_K_CODES = 0,
  KVQ_ARRAY_V_CODES = 1,
  KVQ_ARRAY_K_SCALE = 2,
  KVQ_ARRAY_K_ZERO = 3,
  KVQ_ARRAY_V_SCALE = 4,
  KVQ_ARRAY_V_ZERO = 5,
  KVQ_ARRAY_K_WINDOW = 6,
  KVQ_ARRAY_V_WINDOW = 7,
  KVQ_ARRAY_BLOCK_TABLE = 8,
  KVQ_ARRAY_Q = 9,
  KVQ_ARRAY_K_NEW = 10,
  KVQ_ARRAY_V_NEW = 11,
  KVQ_ARRAY_SEQ_LENS = 12,   /* seq_lens or seq_lens_before */
  KVQ_ARRAY_OUT = 13,
  KVQ_ARRAY_WORKSPACE = 14,
  KVQ_ARRAY_COUNT = 15
} kvq_array;

/*
 * Tests the checks themselves (debug builds only; a release build returns
 * KVQ_ERR_UNSUPPORTED).  Every later launch checks array `array` (a
 * kvq_array) against an extent `bytes` shorter than the one the host derives
 * (bytes = 0 restores it).  Accesses to the array's last `bytes` bytes are
 * then skipped and flagged although they lie inside the caller's allocation.
 * Process-wide host state; not safe to call while another thread launches.
 * Returns KVQ_ERR_INVALID_ARG for an unknown array or bytes < 0.
 */
KVQ_API kvq_status kvq_debug_shrink_extent(int32_t array, int64_t bytes);

/* Static, human-readable name of a status code. */
KVQ_API const char* kvq_status_string(kvq_status status);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
