/*
 * kvq -- quantized paged KV cache for single-token decode (GB300, sm_103a).
 *
 * C ABI of libkvq.so.  Every argument is a plain pointer or size; device
 * pointers are CUDA device memory owned by the caller.  The library never
 * allocates or frees device memory, keeps no state between calls except a
 * per-device error word (kvq_get_device_error) and a cached SM count, and
 * enqueues all work asynchronously on the stream given (NULL = the legacy
 * default stream).  Entry points are thread-safe.
 *
 * Errors: every check that can be made on the host (null pointers, sizes,
 * unsupported shapes or formats, workspace too small, misalignment) returns
 * a status before anything is launched.  A failed launch returns
 * KVQ_ERR_CUDA.  Device-side data (slot ids, block ids) is range-checked in
 * the kernels: an out-of-range id skips the access and sets a bit in the
 * device error word instead of faulting.
 *
 * The operations follow the source pages:
 *  - "vllm-int8-kv-cache-for-ampere-sm86" (project summary): INT8 KV cache
 *    with per-layer scales, optional FP8-E4M3 for one of the two tensors;
 *  - vLLM PR #4893 "Load FP8 kv-cache scaling factors from checkpoints"
 *    (items 1-3, side note): --kv-cache-dtype fp8 / fp8_e4m3 / fp8_e5m2 with
 *    a kv_scale, 1.0 when uncalibrated; FP8 decode runs in the paged-attention
 *    kernel;
 *  - vLLM issue #4025 "Support for 4-bit KV Cache in paged-attention op"
 *    (section 'methods', items 1-3): scale/zero-point computation, int4
 *    storage in write_to_paged_cache, paged attention taking k_scale,
 *    k_zeropoint, v_scale, v_zeropoint;
 *  - "KVarN : le backend natif pour la quantification du cache KV" (section
 *    'Contexte Technique'): a Hadamard rotation and a variance normalisation
 *    before asymmetric codes, with no calibration step.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* kvq_stream_t;

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, misaligned buffer */
  KVQ_ERR_UNSUPPORTED = 2,      /* valid but not implemented (head_dim, block_size, format) */
  KVQ_ERR_WORKSPACE = 3,        /* workspace smaller than kvq_decode_workspace_size */
  KVQ_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
} kvq_status;

/* Stored code formats (the --kv-cache-dtype choices of PR #4893 item 1 plus
 * the INT8 and INT4 caches of the INT8 summary and issue #4025). */
typedef enum {
  KVQ_FMT_INT8 = 1,       /* int8, symmetric, one fp32 scale per tensor          */
  KVQ_FMT_FP8_E4M3 = 2,   /* OCP E4M3FN byte, one fp32 scale per tensor          */
  KVQ_FMT_FP8_E5M2 = 3,   /* OCP E5M2 byte, one fp32 scale per tensor            */
  KVQ_FMT_INT4_ASYM = 4,  /* 4-bit code, fp16 scale + zero point per token-head  */
  KVQ_FMT_UINT8_ASYM = 5, /* 8-bit code, fp16 scale + zero point per token-head  */
  KVQ_FMT_BF16 = 6,       /* the bf16 value itself, no scale (PR #4893 item 1's
                             --kv-cache-dtype auto: the unquantized 16-bit cache);
                             K and V both, no per-head scales, no rotation      */
} kvq_format;

/* KVarN pre-quantization (both tensors; asymmetric formats only): per
 * (token, kv-head) row, divide by its fp16 standard deviation sigma, flip
 * signs by d, apply the orthonormal Walsh-Hadamard transform; store sigma. */
#define KVQ_FLAG_VARNORM_ROTATE 1u

/*
 * Description of one layer's paged cache (all device memory caller-owned).
 *
 * Code arrays (passed separately to the calls):
 *   k_cache, v_cache: [num_blocks, block_size, num_kv_heads, row_bytes] bytes,
 *   row_bytes = head_dim for 8-bit formats, head_dim/2 for INT4 (element 2i
 *   in the low nibble of byte i, element 2i+1 in the high nibble), 2*head_dim
 *   for BF16 (little-endian bf16 values); int8 codes are two's complement.
 *   16-byte aligned.
 * Metadata (asymmetric formats only, else NULL):
 *   k_meta, v_meta: fp16 [num_blocks, num_kv_heads, F, block_size] with
 *   F = 2 fields (scale, zero point) or 3 (scale, zero point, sigma) with
 *   KVQ_FLAG_VARNORM_ROTATE.  16-byte aligned.
 *   Dequantization: x = (code * scale + zero_point) [* sigma, then the
 *   inverse rotation].
 * Per-tensor scales (symmetric formats): x = code_value * k_scale (v_scale).
 * Per-kv-head scales (symmetric formats, optional): k_head_scales /
 *   v_head_scales, device fp32 [num_kv_heads], 4-byte aligned, each > 0; when
 *   given, head h uses x = code_value * k_head_scales[h] (and codes
 *   rne(x * (1 / k_head_scales[h]))) in place of k_scale.  The per-tensor
 *   scales of the INT8 summary and PR #4893 made per attention head, as
 *   PR #4893's thread leaves for later.  NULL: the per-tensor scale.
 * signs: device int8 [head_dim] of +1 / -1 (the rotation's diagonal), or
 *   NULL for all +1; read only with KVQ_FLAG_VARNORM_ROTATE.
 */
typedef struct {
  int32_t k_fmt;        /* kvq_format */
  int32_t v_fmt;        /* kvq_format */
  int32_t num_kv_heads; /* >= 1 */
  int32_t head_dim;     /* 64 or 128 */
  int32_t block_size;   /* tokens per block: 8, 16, 32, 64 or 128 */
  int32_t num_blocks;   /* >= 1 */
  uint32_t flags;       /* KVQ_FLAG_* */
  float k_scale;        /* symmetric K formats: > 0 (1.0 = uncalibrated fp8); BF16: unused */
  float v_scale;        /* symmetric V formats: > 0; BF16: unused */
  void* k_meta;
  void* v_meta;
  const int8_t* signs;
  const float* k_head_scales; /* NULL or device fp32 [num_kv_heads] (symmetric K) */
  const float* v_head_scales; /* NULL or device fp32 [num_kv_heads] (symmetric V) */
} kvq_cache_desc;

/*
 * kvq_write_cache -- quantize bf16 keys/values and scatter them into the
 * paged cache ("write_to_paged_cache" of issue #4025, 'methods' items 1-2;
 * the INT8 / FP8 caches of the INT8 summary and PR #4893).
 *
 * key, value: device bf16 [num_tokens, num_kv_heads, head_dim]; heads and
 *   elements contiguous, consecutive tokens `key_stride` / `value_stride`
 *   elements apart (>= num_kv_heads*head_dim, multiple of 8); 16-byte aligned.
 * slot_mapping: device int64 [num_tokens]; token t is written at
 *   block = slot / block_size, offset = slot % block_size; slot < 0 skips the
 *   token; a slot past the cache sets KVQ_DEVERR_SLOT_RANGE and is skipped.
 *   Two tokens with the same slot: which one lands is unspecified.
 * Codes (fixed float32 arithmetic, IEEE round-to-nearest, no contraction):
 *   BF16:  x itself (the input's 16 bits)
 *   INT8:  clamp(rint(x * inv), -128, 127), inv = 1.0f / scale
 *   FP8:   E4M3 / E5M2 of (x * inv), round to nearest even, saturating to
 *          the largest finite magnitude
 *   ASYM:  s = fp16((max - min) / L) (1 if it is 0), z = fp16(min),
 *          code = clamp(rint((x - z) * (1.0f / s)), 0, L), L = 15 or 255.
 *   With KVQ_FLAG_VARNORM_ROTATE the ASYM step runs on the normalised,
 *   rotated row (see kvq_hadamard for the transform's definition).
 * Slots that are not written are left untouched.  num_tokens == 0 is a no-op.
 */
kvq_status kvq_write_cache(const kvq_cache_desc* cache, void* k_cache, void* v_cache,
                           const void* key, const void* value, int64_t key_stride,
                           int64_t value_stride, const int64_t* slot_mapping,
                           int64_t num_tokens, kvq_stream_t stream);

/*
 * kvq_decode_workspace_size -- bytes of device workspace kvq_paged_decode
 * needs for these sizes: partial results of sequences split between CTAs
 * (num_ctas * 2 * num_q_heads * (head_dim * 2 + 8) bytes: fp16 outputs and
 * fp32 (max, sum); 0 with one CTA)
 * six 8-byte tags and claims per (CTA, group of 8 kv-heads) and one 8-byte
 * merge claim per (sequence, group of 8 kv-heads).  Depends on the device's
 * SM count (current device).
 */
kvq_status kvq_decode_workspace_size(const kvq_cache_desc* cache, int32_t num_seqs,
                                     int32_t num_q_heads, int32_t max_context_len,
                                     size_t* bytes);

/*
 * kvq_paged_decode -- one new query token per sequence attends to its paged,
 * quantized context (issue #4025 'methods' item 3; PR #4893 side note).
 *
 * query: device bf16 [num_seqs, num_q_heads, head_dim], contiguous, 16-byte
 *   aligned.
 * out:   device bf16 [num_seqs, num_q_heads, head_dim], contiguous, 16-byte
 *   aligned.
 *   q-head h reads kv-head h / (num_q_heads / num_kv_heads); the ratio must be
 *   an integer <= 8.
 * block_table: device int32 [num_seqs, max_blocks_per_seq]; entries past
 *   ceil(context_len / block_size) are never read.
 * context_lens: device int32 [num_seqs], each in [0, max_context_len] (a length
 *   outside is clamped into it and sets KVQ_DEVERR_CONTEXT_RANGE).
 *   context_len 0 gives out = 0.
 * sm_scale: logits are sm_scale * <q, k>.
 * workspace: device memory of >= kvq_decode_workspace_size(...) bytes
 *   (may be NULL when that size is 0), 16-byte aligned; its contents on entry
 *   do not matter (its completion tags and claims carry a per-call value).  Two
 *   calls that overlap on the GPU must not share a workspace.
 * CUDA graphs: a call made while its stream is capturing first records a
 *   memset of the workspace's tags and claims (a few KB), so every replay of
 *   the graph starts from clear words (a replay reuses the recorded call's
 *   value).  This holds for kvq_paged_decode(_ex), kvq_decode_append,
 *   kvq_decode_mixed and kvq_paged_decode_static.
 * One kernel launch, stream-K: each CTA owns a contiguous range of the 16-token
 *   tiles of all sequences (for a group of up to 8 kv-heads), the ranges of
 *   equal weight when each sequence boundary is charged as four tiles.  A
 *   sequence split between CTAs leaves partial results that are merged
 *   (log-sum-exp) by a CTA that, after its own range, finds every other part
 *   published.  Results do not depend on the split beyond rounding.
 * out[s, h] = sum_t softmax_t(sm_scale <q, k_t>) v_t over the dequantized
 *   cache, computed with fp32 softmax and fp32 accumulation (keys and values
 *   enter the tensor cores as exact fp16 code values; the query is rounded to
 *   fp16, which is exact for bf16 values of magnitude 2^-14 .. 65504: smaller
 *   ones lose bits, larger ones overflow and set KVQ_DEVERR_QUERY_RANGE; the
 *   16-bit cache keeps the bf16 query).
 */
kvq_status kvq_paged_decode(const kvq_cache_desc* cache, const void* k_cache,
                            const void* v_cache, void* out, const void* query,
                            int32_t num_seqs, int32_t num_q_heads, const int32_t* block_table,
                            int32_t max_blocks_per_seq, const int32_t* context_lens,
                            int32_t max_context_len, float sm_scale, void* workspace,
                            size_t workspace_bytes, kvq_stream_t stream);

/*
 * kvq_paged_decode_ex -- kvq_paged_decode with an explicit number of CTAs
 * per group of 8 kv-heads (the stream-K ranges the tiles are split into,
 * 1..65535; 0 = the automatic choice: two per SM, one for the 16-bit cache).  The workspace must hold
 * kvq_decode_workspace_size_ex(...) bytes for the same num_ctas.
 */
kvq_status kvq_decode_workspace_size_ex(const kvq_cache_desc* cache, int32_t num_seqs,
                                        int32_t num_q_heads, int32_t max_context_len,
                                        int32_t num_ctas, size_t* bytes);
kvq_status kvq_paged_decode_ex(const kvq_cache_desc* cache, const void* k_cache,
                               const void* v_cache, void* out, const void* query,
                               int32_t num_seqs, int32_t num_q_heads,
                               const int32_t* block_table, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, int32_t max_context_len,
                               float sm_scale, int32_t num_ctas, void* workspace,
                               size_t workspace_bytes, kvq_stream_t stream);

/*
 * kvq_decode_append -- one decode step with the step's own key and value:
 * the new token of every sequence is quantized into the paged cache and the
 * query attends to the context including it, in one kernel launch (the
 * "write_to_paged_cache" store and the paged-attention read of issue #4025
 * 'Support for 4-bit KV Cache in paged-attention op', section 'methods',
 * items 2-3, for the decoding phase).
 *
 * new_key, new_value: device bf16 [num_seqs, num_kv_heads, head_dim]; heads
 *   and elements contiguous, consecutive sequences `key_stride` /
 *   `value_stride` elements apart (>= num_kv_heads*head_dim, multiple of 8);
 *   16-byte aligned.
 * context_lens counts the new token: for a sequence with context_len n > 0,
 *   row s is written at position n-1, i.e. at block block_table[s][(n-1) /
 *   block_size], offset (n-1) % block_size, and the attention runs over all
 *   n positions.  A sequence with n = 0 writes nothing (out = 0).  A block id
 *   outside [0, num_blocks) sets KVQ_DEVERR_BLOCK_RANGE and writes nothing.
 * Codes and metadata: exactly those kvq_write_cache stores for the same rows
 *   and slots (same formats, scales, per-head scales and KVarN transform).
 * Output: that of kvq_paged_decode_ex on the cache after the write.
 * The token at position n-1 must be written by this call alone: another call
 *   (or kernel) that writes the same slots or reads them while this one runs
 *   races with it.
 * The caches are written, so k_cache / v_cache (and the metadata in `cache`)
 *   must be writable.  Other arguments, the workspace and its size are those
 *   of kvq_paged_decode_ex (num_ctas included).
 */
kvq_status kvq_decode_append(const kvq_cache_desc* cache, void* k_cache, void* v_cache,
                             const void* new_key, const void* new_value, int64_t key_stride,
                             int64_t value_stride, void* out, const void* query,
                             int32_t num_seqs, int32_t num_q_heads,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             const int32_t* context_lens, int32_t max_context_len,
                             float sm_scale, int32_t num_ctas, void* workspace,
                             size_t workspace_bytes, kvq_stream_t stream);

/*
 * kvq_decode_mixed -- kvq_paged_decode_ex (new_key == NULL) or
 * kvq_decode_append over a cache whose sequences use pages of different sizes
 * (the variable page sizes that the KVarN article's section 'Perspective'
 * looks ahead to).
 *
 * Each page class is a pool of pages of one size: classes[c] describes it
 * (block_size 16, 32, 64 or 128 and num_blocks of its own, its own metadata
 * arrays; formats, num_kv_heads, head_dim, flags, scales, per-head scales and
 * signs equal to class 0's), with codes k_caches[c] / v_caches[c] (host
 * arrays of device pointers).  num_classes: 1 or 2.
 * seq_class: device uint8 [num_seqs], the class of each sequence; row s of
 *   block_table holds block ids of that class's pool, and max_blocks_per_seq
 *   must cover max_context_len at the smallest page size.  A class id outside
 *   [0, num_classes) sets KVQ_DEVERR_CLASS_RANGE and reads class 0.
 * Writes go through kvq_write_cache with each class's description, codes and
 *   slots (slot = block * class block_size + offset).
 * new_key, new_value, key_stride, value_stride: as in kvq_decode_append (the
 *   new row lands in the sequence's class), or NULL for a plain decode.
 * Everything else (workspace and its size, num_ctas, output) is that of
 * kvq_paged_decode_ex / kvq_decode_append for class 0's description.
 */
kvq_status kvq_decode_mixed(const kvq_cache_desc* classes, int32_t num_classes,
                            void* const* k_caches, void* const* v_caches,
                            const uint8_t* seq_class, const void* new_key, const void* new_value,
                            int64_t key_stride, int64_t value_stride, void* out,
                            const void* query, int32_t num_seqs, int32_t num_q_heads,
                            const int32_t* block_table, int32_t max_blocks_per_seq,
                            const int32_t* context_lens, int32_t max_context_len,
                            float sm_scale, int32_t num_ctas, void* workspace,
                            size_t workspace_bytes, kvq_stream_t stream);

/*
 * kvq_paged_decode_static -- kvq_paged_decode_ex for callers that cannot
 * allocate device memory.  None of the source pages has a counterpart of
 * this entry point: it exists for integration, not for the method.
 *
 * Who needs it: code that must not call cudaMalloc (or any allocator) once it
 * is running -- a plugin inside a host application or framework that owns
 * every byte of device memory through its own pool, or a latency-bound
 * serving loop where an allocation could block on the device or fail late.
 * Such a caller still owns the cache, query and output buffers, but has no way
 * to obtain the split-K workspace.
 *
 * Instead of a workspace, the call uses a scratch array of
 * kvq_paged_decode_static_capacity() bytes (16 MiB) compiled into the library:
 * every GPU that loads the library holds that memory until the process exits.
 * Sizes whose workspace (kvq_decode_workspace_size_ex) exceeds it return
 * KVQ_ERR_WORKSPACE before anything is launched.  The call allocates nothing
 * (no cudaMalloc, no cudaFree, no allocating library routine).
 *
 * The first call on a device looks up the scratch's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  The address is kept with the id of the context it belongs to, so
 * a call after cudaDeviceReset (a new primary context) looks it up again.
 * `stream` must belong to the current device: the scratch used is the current
 * device's copy.  All calls share the one array, and it keeps whatever the last
 * call left: nothing in it needs to start at zero (every value the combine
 * reads is written earlier in the same call), but two calls whose kernels
 * overlap on the GPU (different streams, or several host threads) race on it
 * and corrupt each other's results -- serialize them.
 * Arguments and results are those of kvq_paged_decode_ex (num_ctas included).
 */
kvq_status kvq_paged_decode_static(const kvq_cache_desc* cache, const void* k_cache,
                                   const void* v_cache, void* out, const void* query,
                                   int32_t num_seqs, int32_t num_q_heads,
                                   const int32_t* block_table, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, int32_t max_context_len,
                                   float sm_scale, int32_t num_ctas, kvq_stream_t stream);
/* Bytes of the scratch array kvq_paged_decode_static uses. */
size_t kvq_paged_decode_static_capacity(void);

/*
 * kvq_hadamard -- in-place orthonormal Walsh-Hadamard rotation of `rows`
 * rows of `head_dim` elements (KVarN article, 'Contexte Technique').
 *   forward (inverse = 0): x <- cR * H (d . x)
 *   inverse (inverse = 1): x <- d . (cR * H x)
 * H is the natural-order (Sylvester) Hadamard matrix, d = signs (NULL: all
 * +1), cR = float(1/sqrt(head_dim)).  H x is computed in float32 by the
 * butterfly stages h = 1, 2, 4, ..., head_dim/2 in that order, each pair
 * (i, i+h), i & h == 0, becoming (a + b, a - b).  dtype: 0 = float32,
 * 1 = bfloat16 (computed in float32, rounded to nearest even on store).
 * x: device, contiguous rows, 16-byte aligned.  head_dim: 64, 128 or 256.
 */
kvq_status kvq_hadamard(void* x, int32_t dtype, int64_t rows, int32_t head_dim,
                        const int8_t* signs, int32_t inverse, kvq_stream_t stream);

/*
 * kvq_calibrate_scale -- per-tensor scale = absmax(x) / qmax in float32
 * (1.0 when x is all zero): the per-layer scaling values of the INT8
 * summary (qmax 127) and the E4M3 kv_scale (qmax 448).
 * x: device bf16 [n], finite values; scale_out: device float, overwritten.
 */
kvq_status kvq_calibrate_scale(const void* x, int64_t n, float qmax, float* scale_out,
                               kvq_stream_t stream);

/*
 * kvq_calibrate_head_scales -- per-kv-head scales for the k_head_scales /
 * v_head_scales of kvq_cache_desc: scales_out[h] = absmax over tokens t and
 * dims d of x[t, h, d], divided by qmax in float32 (1.0 for an all-zero head).
 * x: device bf16 [num_tokens, num_kv_heads, head_dim], row stride `stride`
 * elements between tokens (>= num_kv_heads * head_dim, multiple of 8), 16-byte
 * aligned, finite values; scales_out: device float [num_kv_heads], 4-byte
 * aligned, overwritten.  head_dim: a multiple of 8.
 */
kvq_status kvq_calibrate_head_scales(const void* x, int64_t num_tokens, int32_t num_kv_heads,
                                     int32_t head_dim, int64_t stride, float qmax,
                                     float* scales_out, kvq_stream_t stream);

/* Device error word bits. */
#define KVQ_DEVERR_SLOT_RANGE 1u  /* a slot id past num_blocks*block_size */
#define KVQ_DEVERR_BLOCK_RANGE 2u /* a block-table entry outside [0, num_blocks) */
#define KVQ_DEVERR_CONTEXT_RANGE 4u /* a context length outside [0, max_context_len] */
#define KVQ_DEVERR_COMBINE 8u       /* a split-sequence merge counter update gave up */
#define KVQ_DEVERR_TIMEOUT 16u      /* a pipeline barrier wait gave up: the CTA stopped
                                       early, the launch's results are invalid */
#define KVQ_DEVERR_CLASS_RANGE 32u  /* a page class id outside the call's classes */
#define KVQ_DEVERR_QUERY_RANGE 64u  /* a query value not finite once converted: beyond
                                       fp16's range (65504) for the quantized formats,
                                       or an infinity or NaN; that row's output is not
                                       meaningful */

/*
 * kvq_debug_arm_wait_timeout -- test hook for the decode kernel's bounded
 * pipeline waits (every mbarrier wait gives up after a number of polls, sets
 * KVQ_DEVERR_TIMEOUT and makes its CTA stop loading, publish nothing and
 * return once no copy it issued is in flight).  It applies to the next decode
 * launch of the process (kvq_paged_decode*, kvq_decode_append) and then
 * disarms itself: that launch polls each wait at most `polls` times (>= 1),
 * and CTA `cta` of the first kv-head group never issues the loads of the
 * `tile`-th tile of its range (-1: every load is issued), so that the waits
 * for that tile run out with nothing in flight.  The launch's output is then
 * invalid.  For tests of the failure path only; a caller never needs it.
 */
kvq_status kvq_debug_arm_wait_timeout(int32_t polls, int32_t cta, int32_t tile);

/*
 * kvq_get_device_error -- synchronizes `stream`, then reads and clears the
 * current device's error word (OR of KVQ_DEVERR_* bits set since the last
 * read) into *bits.
 */
kvq_status kvq_get_device_error(kvq_stream_t stream, uint32_t* bits);

/* Static string for a status code. */
const char* kvq_status_string(kvq_status status);

/* Library version, e.g. "kvq 0.1.0 sm_103a". */
const char* kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
