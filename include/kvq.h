/*
 * kvq.h -- C ABI of the quantized paged KV store for GB300 (sm_103a).
 *
 * A paged, low-precision KV cache plus decode-phase GQA attention that reads
 * the cache directly and dequantizes in registers.
 *
 * Sources (web pages, cited by title and section):
 *   [QKV]   "Quantized KV Cache" (SGLang documentation, data-sketchers wiki)
 *           - Supported formats / FP8 formats, FP4 formats; Usage (format
 *             names); Scaling factors; Performance warning (dequantization not
 *             fused into attention is extremely slow).
 *   [NVFP4] "SGLang PR #21954 analysis: NVFP4 KV cache" (secrett2633 blog)
 *           - Code analysis 1: create_buffers, quantize_and_store,
 *             dequantize_prev_kv; NVFP4 two-level scaling; CUDA-graph
 *             compatibility (Review feedback).
 *   [TRAPS] "KV cache quantization: mechanism and traps" (hrletsgo.me)
 *           - When to enable (bytes per token, the scale-reuse trap).
 *   [VLLM]  "Quantized KV cache" (vLLM documentation, data-sketchers wiki)
 *           - Supported schemes (per-tensor scales); calibration (default 1.0).
 *
 * Conventions for every entry point
 *   - Return KVQ_OK or an error code; on error kvq_last_error_string() gives a
 *     message (thread-local).  Arguments are validated on the host before any
 *     device work; an invalid call changes nothing.
 *   - All array pointers are DEVICE pointers on the cache's device unless the
 *     parameter says "host".  The caller owns them; the library never frees,
 *     retains or reallocates them.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous.  No entry point except kvq_create_cache,
 *     kvq_destroy_cache and kvq_get_device_error allocates, frees or
 *     synchronizes the host.
 *   - Call with the cache's device current.
 *
 * Numerics (readings where the pages are silent; the CPU oracle follows the
 * same definitions):
 *   - FP8 E4M3 is the "fn" variant (max 448, no Inf); E5M2 max 57344.
 *     [QKV] prints +-240 for E4M3, the IEEE-style variant's range.
 *   - Encoding rounds to nearest, ties to even, and saturates to the largest
 *     finite magnitude; the sign is kept, so negatives that round to zero give
 *     the sign-set zero code.  FP8: NaN gives 0x7F with the input's sign.
 *   - FP8: code = enc(x / s), an IEEE fp32 division by the per-tensor scale.
 *   - FP4 block-16 ("fp4_mx_block16"): per 16 elements, E = clamp(floor(log2
 *     amax) - 2, -127, 127) (OCP MX shared-exponent rule, E2M1 emax = 2),
 *     stored as the E8M0 byte E + 127; codes = enc_E2M1(x * 2^-E).
 *   - NVFP4: given the fp32 global scale g, block scale byte
 *     sc = enc_E4M3(amax / (6 g)), S = dec(sc) * g (fp32), codes =
 *     enc_E2M1(x / S) (fp32 division); S == 0 stores all-zero codes.
 *   - FP4 packing: even head_dim index in the low nibble.
 *   - Non-finite K/V values are outside the contract of the FP4 formats.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers (same underlying type). */
struct CUstream_st;
typedef struct CUstream_st* kvq_stream;

/* Cache element formats ([QKV] Supported formats; names from [QKV] Usage). */
typedef enum {
  KVQ_BF16 = 0,        /* "bf16": unquantized reference path               */
  KVQ_FP8_E4M3 = 1,    /* "fp8_e4m3": E4M3fn + per-tensor fp32 scale        */
  KVQ_FP8_E5M2 = 2,    /* "fp8_e5m2": E5M2 + per-tensor fp32 scale          */
  KVQ_FP4_BLOCK16 = 3, /* "fp4_mx_block16": E2M1, one E8M0 per 16 elements  */
  KVQ_NVFP4 = 4        /* "nvfp4": E2M1, E4M3 per 16 + fp32 global scale    */
} kvq_format;

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,    /* bad pointer, size, layer, scale, ...           */
  KVQ_ERR_UNSUPPORTED = 2,    /* valid request this build does not implement    */
  KVQ_ERR_OOM = 3,            /* device allocation failed (kvq_create_cache)    */
  KVQ_ERR_CUDA = 4,           /* a CUDA runtime call failed                     */
  KVQ_ERR_SCALE_MISMATCH = 5, /* scales differ from the ones fixed for a layer  */
  KVQ_ERR_DEVICE_RANGE = 6,   /* a kernel saw an out-of-range slot/page/length  */
  KVQ_ERR_TIMEOUT = 7         /* a kernel's bounded wait ran out                */
} kvq_status;

typedef struct kvq_cache kvq_cache; /* opaque */

/*
 * Create a cache of `layers` layers, each holding K and V pools of
 * `num_pages` pages of `page_size` tokens for `kv_heads` heads of
 * `head_dim` elements ([NVFP4] create_buffers: data buffers plus block-scale
 * buffers; the FP8 dequantization workspace of that design is not needed
 * because attention dequantizes in registers).
 * Layout per layer and per K/V:
 *   data  [num_pages][kv_heads][page_size][row]   row = head_dim * 2 (bf16),
 *                                                 head_dim (fp8), head_dim/2 (fp4)
 *   scale [num_pages][kv_heads][page_size][head_dim / 16] bytes (FP4 formats)
 * One device allocation (owned by the cache, freed by kvq_destroy_cache),
 * zero-filled.  Requires head_dim % 16 == 0, page_size >= 1, all counts > 0.
 * Errors: INVALID_ARG, OOM, CUDA.  *out is set only on success.
 */
kvq_status kvq_create_cache(kvq_format fmt, int layers, int kv_heads, int head_dim,
                            int page_size, int num_pages, kvq_cache** out);

/* Free the cache's device memory (synchronizes the device).  NULL is a no-op. */
kvq_status kvq_destroy_cache(kvq_cache* cache);

/*
 * Quantize bf16 K/V rows and scatter them into the paged cache of `layer`
 * ([NVFP4] quantize_and_store; [QKV] Scaling factors).
 *   k_bf16, v_bf16: [num_tokens][kv_heads][head_dim] bf16, contiguous.
 *   slot_mapping:   int64 [num_tokens]; slot = page * page_size + offset;
 *                   -1 skips the token (padding).
 *   scales (host):  FP8: {k_scale, v_scale}; NVFP4: {g_k, g_v}; ignored (may
 *                   be NULL) for bf16 and fp4_mx_block16.  NULL for an FP8 or
 *                   NVFP4 format means 1.0 ([QKV] Scaling factors, [VLLM]:
 *                   the default scale is 1.0).  Must be finite and > 0.
 * The first store to a layer fixes its scales; a later store with different
 * values returns KVQ_ERR_SCALE_MISMATCH (guards the scale-reuse trap of
 * [TRAPS] When to enable).  Slots >= num_pages * page_size are skipped and
 * raise KVQ_ERR_DEVICE_RANGE in the device error word.
 * num_tokens == 0 is a valid no-op.
 */
kvq_status kvq_quantize_and_store(kvq_cache* cache, int layer, const void* k_bf16,
                                  const void* v_bf16, const int64_t* slot_mapping,
                                  int num_tokens, const float* scales, kvq_stream stream);

/*
 * kvq_quantize_and_store with one scale per kv head ([VLLM] Supported
 * schemes: per-attention-head quantization, k/v_scale = [num_kv_heads]).
 *   k_scales, v_scales (host): [kv_heads] floats, finite and > 0 -- the FP8
 *                   scales or the NVFP4 global scales of each kv head; ignored
 *                   (may be NULL) for bf16 and fp4_mx_block16.
 * Every kv head h is quantized as with kvq_quantize_and_store and scale
 * k_scales[h] / v_scales[h]; attention and kvq_dequantize use the same scale
 * per head.  Equal scales on every head are exactly the per-tensor case.  The
 * first store of a layer that stores tokens fixes its scales (with either
 * entry point, or kvq_calibrate_scales); a later store whose scales differ on
 * any head returns KVQ_ERR_SCALE_MISMATCH.  Other errors as for
 * kvq_quantize_and_store.
 */
kvq_status kvq_quantize_and_store_per_head(kvq_cache* cache, int layer, const void* k_bf16,
                                           const void* v_bf16, const int64_t* slot_mapping,
                                           int num_tokens, const float* k_scales,
                                           const float* v_scales, kvq_stream stream);

/*
 * Fix the scales of `layer` from a batch of bf16 K and V rows on the device
 * ([VLLM] Scale calibration approaches: scales estimated on the fly from one
 * batch of tokens, then fixed; [QKV] Scaling factors).
 *   k_bf16, v_bf16: [num_tokens][kv_heads][head_dim] bf16 device rows, 16-byte
 *                   aligned, num_tokens >= 1.
 *   per_head:       0: one scale per tensor (K and V each); 1: one per kv head.
 * scale = amax / M over the finite values (per tensor or per kv head), fp32
 * division, M = 448 (E4M3), 57344 (E5M2), 6 * 448 = 2688 (NVFP4 global scale:
 * the largest block scale lands on the E4M3 maximum); amax == 0 gives 1.0.
 * Stream-ordered, no host synchronization, no allocation; every layer has its
 * own reduction scratch, so calibrations of different layers may run on
 * different streams at the same time.  Only valid on a
 * layer whose scales are not fixed yet (else KVQ_ERR_SCALE_MISMATCH); for bf16
 * and fp4_mx_block16 it fixes nothing but marks the layer as set.  Later
 * stores of the layer pass scales == NULL to kvq_quantize_and_store (explicit
 * scales return KVQ_ERR_SCALE_MISMATCH: the host does not see the values).
 * Errors: INVALID_ARG, SCALE_MISMATCH, CUDA.
 */
kvq_status kvq_calibrate_scales(kvq_cache* cache, int layer, const void* k_bf16,
                                const void* v_bf16, int num_tokens, int per_head,
                                kvq_stream stream);

/*
 * Decode attention of one query token per sequence over the cache of
 * `layer`, dequantizing in registers ([QKV] Performance warning; [NVFP4]
 * XQA decode path, here fused).  For sequence b and q head j, with
 * h = j / (num_q_heads / kv_heads) (consecutive q heads share a kv head):
 *   out[b][j] = sum_t softmax_t(sm_scale * q[b][j] . K^[t]) V^[t],
 *   t < seq_lens[b], token t in page page_table[b][t / page_size] at
 *   offset t % page_size; a sequence with seq_lens[b] == 0 gives zeros.
 *   q_bf16:      [batch][num_q_heads][head_dim] bf16.
 *   page_table:  int32 [batch][max_pages_per_seq].
 *   seq_lens:    int32 [batch], 0 <= seq_lens[b] <= max_pages_per_seq * page_size.
 *   out_bf16:    [batch][num_q_heads][head_dim] bf16 (round to nearest even).
 *   workspace:   device scratch of at least kvq_decode_workspace_size(...)
 *                bytes, 16-byte aligned, used only during the call (split-K
 *                partial outputs and log-sum-exps).
 * sm_scale: any finite value (a negative one is folded into the query's sign).
 * Supported: head_dim == 128, page_size % 16 == 0, num_q_heads % kv_heads == 0
 * with group size (num_q_heads / kv_heads) <= 16.  Page ids outside
 * [0, num_pages) or out-of-range lengths raise KVQ_ERR_DEVICE_RANGE in the
 * device error word and zero the affected sequence's output.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
kvq_status kvq_decode_attention(kvq_cache* cache, int layer, const void* q_bf16, int num_q_heads,
                                const int32_t* page_table, int max_pages_per_seq,
                                const int32_t* seq_lens, int batch, float sm_scale,
                                void* out_bf16, void* workspace, size_t workspace_bytes,
                                kvq_stream stream);

/*
 * Extend (chunked-prefill) attention over the cache of `layer` ([NVFP4] Code
 * analysis 1: the prefill / extend path reads the previously stored,
 * quantized KV; here it is read in place instead of through a dequantized
 * workspace).  Query token i belongs to sequence q_seq[i] and attends to that
 * sequence's tokens [0, q_len[i]) -- its causal prefix, itself included, so
 * the new tokens must be stored first:
 *   out[i][j] = sum_t softmax_t(sm_scale * q[i][j] . K^[t]) V^[t],
 *   t < q_len[i], token t in page page_table[q_seq[i]][t / page_size].
 *   q_bf16, out_bf16: [num_q_tokens][num_q_heads][head_dim] bf16.
 *   q_seq, q_len:     int32 [num_q_tokens] device arrays; 0 <= q_seq[i] <
 *                     num_seqs, 0 <= q_len[i] <= max_pages_per_seq * page_size.
 *   page_table:       int32 [num_seqs][max_pages_per_seq].
 *   workspace:        device scratch, 16-byte aligned, of
 *                     kvq_extend_workspace_size(...) bytes for the fastest
 *                     plan: each sequence's context is split across CTAs and
 *                     the splits' partial outputs are merged.  A smaller
 *                     workspace (or NULL / 0) is valid: the call then uses
 *                     fewer splits (none without a workspace).
 * Every K/V chunk of a sequence is read and dequantized once per 128 (query,
 * q head) rows of a kv head, shared by those rows' queries (16 queries at 8 q
 * heads per kv head); QK^T and PV run on the tcgen05 tensor cores with fp32
 * accumulators in tensor memory.  Out-of-range
 * q_seq, q_len or page ids raise KVQ_ERR_DEVICE_RANGE in the device error word
 * and zero that query's output.  Other rules and errors as for
 * kvq_decode_attention.
 */
kvq_status kvq_extend_attention(kvq_cache* cache, int layer, const void* q_bf16, int num_q_heads,
                                int num_q_tokens, const int32_t* q_seq, const int32_t* q_len,
                                const int32_t* page_table, int num_seqs, int max_pages_per_seq,
                                float sm_scale, void* out_bf16, void* workspace,
                                size_t workspace_bytes, kvq_stream stream);

/*
 * Decode attention in the FP8 domain with a quantized query ([VLLM] FP8 KV
 * cache overview: with an FP8 KV cache on the Flash Attention 3 backend the
 * attention itself is computed in the quantized (FP8) domain and the query is
 * quantized to FP8 together with keys and values; [VLLM] Supported schemes:
 * q_scale is [1] per tensor or [num_heads] per attention head).
 *   q_scales (host): num_q_scales = 1 (per tensor) or num_q_heads floats
 *                    (per q head), finite and > 0, at most 256.
 * Every q head j is quantized to E4M3 with the store's rule: code =
 * enc_E4M3(q / q_scale_j) (fp32 division, nearest, ties to even, saturating),
 * and QK^T runs on FP8 tensor cores over the query codes and the cache's FP8
 * codes unconverted; the softmax weights and the PV product keep f16/fp32
 * precision (they are not quantized).  The result is attention over the
 * dequantized query q^ = dec(code) * q_scale_j:
 *   out[b][j] = sum_t softmax_t(sm_scale * q^[b][j] . K^[t]) V^[t].
 * Only for fp8_e4m3 and fp8_e5m2 caches (others: KVQ_ERR_UNSUPPORTED).  All
 * other arguments, the workspace (same size as kvq_decode_attention's), the
 * rules and the errors are those of kvq_decode_attention.
 */
kvq_status kvq_decode_attention_fp8q(kvq_cache* cache, int layer, const void* q_bf16,
                                     int num_q_heads, const float* q_scales, int num_q_scales,
                                     const int32_t* page_table, int max_pages_per_seq,
                                     const int32_t* seq_lens, int batch, float sm_scale,
                                     void* out_bf16, void* workspace, size_t workspace_bytes,
                                     kvq_stream stream);

/*
 * The query quantization of kvq_decode_attention_fp8q on its own ([VLLM] FP8
 * KV cache overview; Supported schemes), for callers that keep the FP8 query:
 *   q_bf16:   [rows][num_q_heads][head_dim] bf16 device rows, 16-byte aligned.
 *   q_scales: host, 1 or num_q_heads floats (finite, > 0, at most 256).
 *   q_codes:  [rows][num_q_heads][head_dim] E4M3 bytes (device, 16-byte
 *             aligned): enc_E4M3(q / q_scale) per element, NaN -> 0x7F with
 *             its sign.
 * head_dim % 16 == 0.  No cache needed.  Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
kvq_status kvq_quantize_query(const void* q_bf16, int rows, int num_q_heads, int head_dim,
                              const float* q_scales, int num_q_scales, void* q_codes,
                              kvq_stream stream);

/* Bytes of workspace kvq_extend_attention uses at most for these sizes (0 when
 * it needs none, or on invalid arguments; see kvq_last_error_string). */
size_t kvq_extend_workspace_size(const kvq_cache* cache, int num_q_tokens, int num_q_heads,
                                 int max_pages_per_seq);

/* Bytes of workspace kvq_decode_attention needs for these sizes (0 on invalid
 * arguments; see kvq_last_error_string). */
size_t kvq_decode_workspace_size(const kvq_cache* cache, int batch, int num_q_heads,
                                 int max_pages_per_seq);

/* Size of the static scratch array of kvq_decode_attention_noalloc (16 MiB). */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * kvq_decode_attention without a workspace argument, for callers that cannot
 * allocate device memory when they decode: an application that must not call
 * cudaMalloc/cudaFree after start-up (those calls may synchronize the device
 * and can fail once memory is committed), or a plugin whose host framework
 * owns all device memory and gives it no allocator.  The pages have no
 * counterpart of this call; it is an addition of this library.
 * Same arguments, semantics and errors as kvq_decode_attention, minus the
 * workspace.  The split-K scratch is a file-scope static device array of
 * KVQ_NOALLOC_SCRATCH_BYTES that every GPU loading the library keeps until the
 * process exits; this call allocates nothing.  Sizes whose workspace
 * (kvq_decode_workspace_size) exceeds that array are rejected with
 * KVQ_ERR_UNSUPPORTED and a message.  The first call on a device resolves the
 * array's device address (cudaGetSymbolAddress) with that device current, so
 * make that first call before any stream capture.  All calls share the array:
 * calls that overlap on the GPU (other streams or host threads) race.
 */
kvq_status kvq_decode_attention_noalloc(kvq_cache* cache, int layer, const void* q_bf16,
                                        int num_q_heads, const int32_t* page_table,
                                        int max_pages_per_seq, const int32_t* seq_lens, int batch,
                                        float sm_scale, void* out_bf16, kvq_stream stream);

/*
 * Gather and dequantize rows back to bf16 ([NVFP4] dequantize_prev_kv, here
 * to bf16 instead of an FP8 workspace; a test and debugging utility):
 *   k_out_bf16[i][h][d] = bf16_RNE(fp32(dec(code) * S)), S the element's fp32
 *   scale (s, 2^E, or dec(sc) * g).
 *   slot_mapping: int64 [num_tokens]; -1 (and out-of-range slots, which also
 *   raise KVQ_ERR_DEVICE_RANGE) give zero rows.
 *   k_out_bf16, v_out_bf16: [num_tokens][kv_heads][head_dim] bf16.
 */
kvq_status kvq_dequantize(kvq_cache* cache, int layer, const int64_t* slot_mapping,
                          int num_tokens, void* k_out_bf16, void* v_out_bf16, kvq_stream stream);

/*
 * Device addresses of a layer's pools (for tests and external kernels).
 * strides (host, may be NULL) receives, in bytes: [0] one page of a data pool,
 * [1] one (page, kv_head) slab of a data pool, [2] one token row of a data
 * pool, [3] one token row of a scale plane (0 for formats without block
 * scales).  Scale pointers are NULL for formats without block scales.
 */
kvq_status kvq_cache_layout(const kvq_cache* cache, int layer, void** k_data, void** v_data,
                            void** k_scales, void** v_scales, size_t strides[4]);

/* The per-tensor scales fixed for `layer` (host out[2] = {K, V}); returns
 * KVQ_ERR_INVALID_ARG if the layer has no scales yet or its kv heads have
 * different scales (read those with kvq_layer_head_scales).  For a calibrated
 * layer it synchronizes the device first. */
kvq_status kvq_layer_scales(const kvq_cache* cache, int layer, float out[2]);

/* The per-kv-head scales of a layer (k_out, v_out: host [kv_heads] each):
 * the values its first store fixed, or, for a calibrated layer, the values
 * the device computed (this synchronizes `stream` first).  INVALID_ARG if the
 * layer has no scales yet. */
kvq_status kvq_layer_head_scales(const kvq_cache* cache, int layer, float* k_out, float* v_out,
                                 kvq_stream stream);

/* Cache bytes per token for a model: 2 (K, V) x layers x kv_heads x bytes per
 * head row, including one scale byte per 16 elements for the FP4 formats
 * ([TRAPS] When to enable; [QKV] Memory savings: 4.5 bits per element).
 * Per-layer global scales are not per-token and are not counted.  0 on
 * invalid arguments.  Host only. */
size_t kvq_bytes_per_token(kvq_format fmt, int layers, int kv_heads, int head_dim);

/* Format <-> name ([QKV] Usage: "bf16", "fp8_e4m3", "fp8_e5m2",
 * "fp4_mx_block16", "nvfp4").  Host only. */
kvq_status kvq_format_from_name(const char* name, kvq_format* out);
const char* kvq_format_name(kvq_format fmt); /* NULL for an unknown value */

/* Synchronize `stream`, then read and clear the cache's device error word:
 * KVQ_OK, KVQ_ERR_DEVICE_RANGE or KVQ_ERR_TIMEOUT (or KVQ_ERR_CUDA if the
 * synchronization itself fails). */
kvq_status kvq_get_device_error(kvq_cache* cache, kvq_stream stream);

/* Message for the last error on this thread (never NULL). */
const char* kvq_last_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
