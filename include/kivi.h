/*
 * kivi.h - C ABI of the GB300 (sm_103a) KIVI KV-cache library.
 *
 * KIVI stores the key cache quantized per channel and the value cache
 * quantized per token, asymmetric min/max, 2 (or 4) bits, with the newest
 * tokens kept unquantized in a residual window ("KIVI: A Tuning-Free
 * Asymmetric 2bit Quantization for KV Cache", abstract; "KIVI: Asymmetric
 * 2-Bit KV Cache Quantization Guide", section "The Three Structural
 * Innovations of KIVI"). This library holds the data-parallel hot path:
 * the codec, the append + group flush of a decode step or a prefill, and
 * split-K decode attention that reads the packed cache directly.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument named *_dev, and every buffer inside kivi_seq,
 *    is DEVICE memory of the current CUDA device, allocated and owned by the
 *    caller, 16-byte aligned. Configuration structs (kivi_cfg) are host memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). All work is enqueued on it; no entry point synchronizes, and
 *    the library allocates no device memory. The only state it keeps between
 *    calls is per-device launch settings (each attention kernel's shared
 *    memory limit, raised on its first launch on a device, and its count of
 *    resident CTAs), held in atomic per-device slots, so it is safe to call
 *    from several host threads (kivi_decode_attn_static, described at its
 *    declaration, adds a device array that its calls share).
 *  - Argument errors are found on the host before anything is launched and
 *    returned synchronously (KIVI_ERR_ARG, KIVI_ERR_UNSUPPORTED,
 *    KIVI_ERR_WORKSPACE). A failed launch returns KIVI_ERR_CUDA.
 *    Data-dependent errors found on the device are written to the caller's
 *    status word (*status_dev) with an atomic compare-and-swap from 0, so
 *    the first error code sticks until the caller clears the word; the
 *    library never clears it. No kernel traps or asserts.
 *  - fp16 scale and zero bit patterns are stored as uint16_t.
 *
 * Quantization rule (the codec; the guide's "Step 1" with the zero point
 * taken as the group minimum itself). For a group of G values x_i,
 * widened exactly to fp32:
 *     mn = min x_i, mx = max x_i
 *     s  = fp16_rn( (mx - mn) / qmax )     qmax = 2^bits - 1, IEEE fp32 sub/div
 *     z  = fp16_rn( mn )
 *     c_i = clamp( rint( (x_i - float(z)) / float(s) ), 0, qmax )  (c_i = 0 if s == 0)
 *     dequantized value = c_i * s + z
 * Keys: one group per (kv head, G consecutive tokens aligned to position 0,
 * channel), coded at k_bits. Values: one group per (kv head, token, G
 * consecutive channels), coded at v_bits. Domain: finite inputs with
 * |x| <= 65504 (scale and zero are fp16).
 *
 * Packing rule: a token row holds its D codes, channel d in byte
 * d*bits/8 at bit offset (d mod (8/bits))*bits, lowest bits first
 * (four 2-bit codes, or two 4-bit codes, per byte); bits is k_bits for key
 * rows and v_bits for value rows.
 *
 * Cache state of one sequence holding L tokens (a pure function of L):
 *     n_packed(L) = G * floor(max(L - R, 0) / G)     packed tokens [0, n_packed)
 *     r(L)        = L - n_packed(L)                 residual tokens, in [R, R+G-1] once L >= R
 * Residual position p lives in ring slot p mod (R + G). When an append makes
 * the residual reach R + G tokens, the oldest G are quantized and packed
 * (the guide's fp16 window that is "grouped and packed" once tokens slide
 * past it; G = 32 and R = 128 by default, "KV cache quantization with KIVI
 * INT2 setup guide 2026", section "KIVI: Per-Channel Key, Per-Token Value
 * Quantization Explained"; G = 64, R = 64 and separate k_bits / v_bits in
 * the config example of "KV-Cache Quantization: I Ran the Experiments So You
 * Don't Have To", section "Component 4" (serving architecture and manifests)).
 */
#ifndef KIVI_H
#define KIVI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KIVI_ABI_VERSION 3

typedef enum kivi_status {
    KIVI_OK = 0,
    KIVI_ERR_ARG = 1,          /* invalid argument or configuration; nothing launched */
    KIVI_ERR_UNSUPPORTED = 2,  /* valid configuration this library does not implement */
    KIVI_ERR_CAPACITY = 3,     /* device: an append would need more than cap_tokens packed tokens */
    KIVI_ERR_WORKSPACE = 4,    /* workspace pointer NULL or smaller than required */
    KIVI_ERR_CUDA = 5,         /* a CUDA launch or runtime call failed */
    KIVI_ERR_LENGTH = 6        /* device: kv_len or n_new out of the range the call allows */
} kivi_status;

typedef enum kivi_dtype {
    KIVI_F16 = 0,   /* IEEE binary16 */
    KIVI_BF16 = 1   /* bfloat16 */
} kivi_dtype;

/* Configuration (host memory). */
typedef struct kivi_cfg {
    int32_t k_bits;        /* key code width: 2 or 4 */
    int32_t v_bits;        /* value code width: 2 or 4 */
    int32_t group;         /* G: 32 or 64 */
    int32_t residual;      /* R: residual window, a positive multiple of G */
    int32_t head_dim;      /* D: multiple of G, at most 256 (decode attention: 128) */
    int32_t num_q_heads;   /* Hq (attention only), a multiple of num_kv_heads */
    int32_t num_kv_heads;  /* Hkv */
    int32_t dtype;         /* kivi_dtype of K, V, q and the residual ring */
} kivi_cfg;

/*
 * Buffers of one sequence (an array of these lives in device memory).
 * cap = cap_tokens, a multiple of G: packed capacity in tokens. A sequence
 * can hold up to cap + R + G - 1 tokens.
 *
 * Contiguous layout (flags = 0): the packed buffers belong to this sequence.
 *   k_codes [Hkv][cap][D*k_bits/8]  u8   packed key rows
 *   k_scale [Hkv][cap/G][D]       fp16   per (key group, channel)
 *   k_zero  [Hkv][cap/G][D]       fp16
 *   v_codes [Hkv][cap][D*v_bits/8]  u8   packed value rows
 *   v_scale [Hkv][cap][D/G]       fp16   per (token, channel group)
 *   v_zero  [Hkv][cap][D/G]       fp16
 *
 * Paged layout (flags = KIVI_SEQ_PAGED): the six packed buffers are pools of
 * pages that any number of sequences may share. A page holds one packed group
 * of G tokens for every kv head, laid out like a contiguous sequence with
 * cap = G:
 *   k_codes [pages][Hkv][G][D*k_bits/8], k_scale, k_zero [pages][Hkv][D],
 *   v_codes [pages][Hkv][G][D*v_bits/8], v_scale, v_zero [pages][Hkv][G][D/G]
 * block_table [cap/G] int32 (device memory) gives the page of each packed
 * group of the sequence, in order; the caller keeps the pages of different
 * sequences apart. Packed groups are written once (when they leave the
 * residual window) and only read afterwards, so a table may be extended
 * between calls.
 *
 * Both layouts:
 *   k_res   [Hkv][R+G][D]         dtype  residual ring (slot p mod (R+G))
 *   v_res   [Hkv][R+G][D]         dtype
 * Ring slots that hold no live residual position have unspecified contents.
 * This paging is not on the pages that describe KIVI; it maps the packed cache
 * onto the fixed-size blocks of a paged serving cache.
 */
#define KIVI_SEQ_PAGED 1
typedef struct kivi_seq {
    uint8_t* k_codes;
    uint16_t* k_scale;
    uint16_t* k_zero;
    uint8_t* v_codes;
    uint16_t* v_scale;
    uint16_t* v_zero;
    void* k_res;
    void* v_res;
    int32_t cap_tokens;
    int32_t flags;                 /* 0 or KIVI_SEQ_PAGED */
    const int32_t* block_table;    /* KIVI_SEQ_PAGED only; else unused */
} kivi_seq;

/* ---------------------------------------------------------------- codec */

/*
 * Per-channel key quantization ("The Three Structural Innovations of KIVI",
 * item 1: key elements grouped along the sequence for each channel).
 *   x     [n_streams][n_tokens][D] dtype, n_tokens a multiple of G
 *   codes [n_streams][n_tokens][D*k_bits/8]
 *   scale, zero [n_streams][n_tokens/G][D] fp16
 * Errors: KIVI_ERR_ARG for a bad config, NULL pointers, negative sizes or
 * n_tokens % G != 0. n_streams == 0 or n_tokens == 0 is a no-op.
 */
kivi_status kivi_quant_keys(const kivi_cfg* cfg, int32_t n_streams, int32_t n_tokens,
                            const void* x_dev, uint8_t* codes_dev, uint16_t* scale_dev,
                            uint16_t* zero_dev, void* stream);

/*
 * Per-token value quantization (same section, item 2: value elements
 * grouped along the channels of each token), G channels per group.
 *   x     [n_streams][n_tokens][D] dtype, any n_tokens >= 0
 *   codes [n_streams][n_tokens][D*v_bits/8]
 *   scale, zero [n_streams][n_tokens][D/G] fp16
 */
kivi_status kivi_quant_values(const kivi_cfg* cfg, int32_t n_streams, int32_t n_tokens,
                              const void* x_dev, uint8_t* codes_dev, uint16_t* scale_dev,
                              uint16_t* zero_dev, void* stream);

/* ---------------------------------------------------------------- state update */

/*
 * Append new tokens to each sequence and flush every group of G tokens that
 * leaves the residual window (same section, item 3). A decode step is
 * n_new = 1; a prefill is kv_len = 0, n_new = L. The result is bit-identical
 * to appending the tokens one at a time.
 *   seqs_dev   [nseq] kivi_seq
 *   kv_len_dev [nseq] int32, in/out: tokens held; increased by n_new on success
 *   k_new_dev, v_new_dev [nseq] device pointers, sequence b's new tokens as
 *              [Hkv][n_new_b][D] dtype (may be NULL where n_new_b == 0)
 *   n_new_dev  [nseq] int32, 0 <= n_new_b <= max_new
 *   max_new    host bound on every n_new_b (sizes the grid)
 *   status_dev one int32 (see the conventions above)
 * Device errors: KIVI_ERR_CAPACITY when sequence b would need more than
 * cap_tokens packed tokens, KIVI_ERR_LENGTH when n_new_b is outside
 * [0, max_new] or kv_len_b < 0; such a sequence is left unchanged.
 * Concurrent appends to the same sequence race.
 */
kivi_status kivi_append_flush(const kivi_cfg* cfg, int32_t nseq, const kivi_seq* seqs_dev,
                              int32_t* kv_len_dev, const void* const* k_new_dev,
                              const void* const* v_new_dev, const int32_t* n_new_dev,
                              int32_t max_new, int32_t* status_dev, void* stream);

/* ---------------------------------------------------------------- attention */

/*
 * Split-K decode attention over the packed cache, one query token per
 * sequence, dequantizing on the fly inside the kernel ("Production Serving
 * and vLLM Deployment Trade-offs in 2026": on-the-fly dequantization in
 * SRAM). Query head hq reads kv head hq / (Hq / Hkv).
 *   out[b][hq][:] = sum_t softmax_t(softmax_scale * q[b][hq] . k_t) v_t
 * over all kv_len_b tokens of sequence b (packed tokens dequantized as
 * c*s + z, residual tokens as stored). fp32 accumulation and output.
 *   q_dev      [nseq][Hq][D] dtype
 *   out_dev    [nseq][Hq][D] fp32
 *   max_kv_len host bound on every kv_len_b (sizes the grid and the workspace)
 *   workspace_dev, workspace_bytes: at least kivi_decode_workspace_bytes()
 *              bytes, zero-filled before its first use; every call leaves it
 *              zero-filled again (every partial record is cleared by the
 *              kernel that merges it, and split tickets are reset), so one
 *              workspace serves any sequence of decode and multi-query calls
 *              whose sizes it covers. Calls that share a workspace must not
 *              overlap.
 *   status_dev one int32 (may be NULL)
 * A sequence with kv_len 0 gets zeros. Device error KIVI_ERR_LENGTH: kv_len_b
 * outside [0, max_kv_len] or more tokens than the sequence can hold; that
 * sequence's output rows are set to NaN. Domain of q: finite, with
 * |softmax_scale * q| <= 2^100 (far beyond it fp32 logits overflow anyway).
 * Query groups 1, 2, 4 and 8 run on a persistent tensor-core kernel (a group of
 * 8 as one stream of eight heads per kv head), followed on the same stream by
 * a small kernel that merges the partial records of the sequences and kv
 * heads it split over several CTAs; any other group up to 32 runs on the
 * multi-query kernel with one query.
 * Errors: KIVI_ERR_UNSUPPORTED unless D == 128 and Hq/Hkv <= 32.
 */
kivi_status kivi_decode_attn(const kivi_cfg* cfg, int32_t nseq, const kivi_seq* seqs_dev,
                             const int32_t* kv_len_dev, const void* q_dev, float* out_dev,
                             float softmax_scale, int32_t max_kv_len, void* workspace_dev,
                             size_t workspace_bytes, int32_t* status_dev, void* stream);

/* Workspace bytes kivi_decode_attn needs for (nseq, max_kv_len); 0 on a bad config. */
size_t kivi_decode_workspace_bytes(const kivi_cfg* cfg, int32_t nseq, int32_t max_kv_len);

/*
 * Multi-query attention over the packed cache: the n_query newest tokens of
 * each sequence (already appended with kivi_append_flush) attend causally, as
 * when a target model verifies n_query draft tokens (speculative decoding) or
 * a prefill runs in chunks. The pages that describe KIVI show one query per
 * step; this entry point reads the same cache the same way ("KIVI: Asymmetric
 * 2-Bit KV Cache Quantization Guide", section "Step 2": dequantize during
 * attention), with the causal mask as this library's reading.
 *   out[b][i][hq][:] = sum_{t <= p_i} softmax_t(softmax_scale * q[b][i][hq] . k_t) v_t,
 *   p_i = kv_len_b - n_query + i
 * Query head hq reads kv head hq / (Hq / Hkv). Packed tokens are dequantized as
 * c*s + z, residual tokens read as stored; every masked token lies in the
 * residual window. fp32 accumulation and output.
 *   q_dev      [nseq][n_query][Hq][D] dtype
 *   out_dev    [nseq][n_query][Hq][D] fp32
 *   n_query    queries per sequence, 1 <= n_query and n_query * Hq / Hkv <= 32
 *   max_kv_len, workspace_dev, workspace_bytes, status_dev: as kivi_decode_attn, with
 *              kivi_decode_multi_workspace_bytes() for the size
 * Device error KIVI_ERR_LENGTH: kv_len_b < n_query, kv_len_b > max_kv_len or
 * more tokens than the sequence can hold; that sequence's output rows are NaN.
 * Domain of q: as kivi_decode_attn.
 * Errors: KIVI_ERR_ARG for n_query < 1; KIVI_ERR_UNSUPPORTED unless D == 128
 * and n_query * Hq / Hkv <= 32.
 * n_query == 1 with Hq / Hkv of 1, 2, 4 or 8 runs the kernels of kivi_decode_attn
 * (one query attends to every token), and so do calls with several queries at
 * Hq / Hkv of 4 or 8 and with two queries at Hq / Hkv of 1 or 2 (one stream of
 * the group's heads per query and kv head, each ending its residual range at its
 * query's causal end); the length errors above apply. Other calls run on a
 * multi-query kernel that unpacks each tile once for all (query, head) pairs of
 * its kv head.
 */
kivi_status kivi_decode_multi_attn(const kivi_cfg* cfg, int32_t nseq, const kivi_seq* seqs_dev,
                                   const int32_t* kv_len_dev, int32_t n_query, const void* q_dev,
                                   float* out_dev, float softmax_scale, int32_t max_kv_len,
                                   void* workspace_dev, size_t workspace_bytes, int32_t* status_dev,
                                   void* stream);

/* Workspace bytes kivi_decode_multi_attn needs; 0 on a bad config or n_query < 1. */
size_t kivi_decode_multi_workspace_bytes(const kivi_cfg* cfg, int32_t nseq, int32_t n_query,
                                         int32_t max_kv_len);

/*
 * Decode attention that allocates nothing and takes no workspace argument.
 * The pages that describe KIVI have no counterpart of this entry point; it
 * exists for callers that cannot call cudaMalloc: processes whose device
 * memory is already reserved by another allocator (a serving framework's
 * memory pool), latency-critical paths that must not allocate or free
 * (cudaFree synchronizes the whole device), and plugin hosts whose interface
 * passes only input and output buffers.
 * Same arguments, results and errors as kivi_decode_attn, except that the
 * workspace is a fixed array of KIVI_STATIC_WORKSPACE_BYTES bytes in the
 * library's own device memory: every GPU that loads the library holds it
 * until the process exits. Calls whose kivi_decode_workspace_bytes(cfg, nseq,
 * max_kv_len) exceeds that size return KIVI_ERR_WORKSPACE and launch nothing.
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before any stream
 * capture. The cached address belongs to the device's primary context: after
 * cudaDeviceReset on a device, do not call this entry point on it again. The entry point calls no cudaMalloc, cudaFree or other allocating
 * routine. All calls on a device share the array: each call clears the part
 * that must start at zero (with an asynchronous memset on `stream`), and calls
 * that overlap on the GPU race and give wrong results.
 */
#define KIVI_STATIC_WORKSPACE_BYTES (16u << 20)
kivi_status kivi_decode_attn_static(const kivi_cfg* cfg, int32_t nseq, const kivi_seq* seqs_dev,
                                    const int32_t* kv_len_dev, const void* q_dev, float* out_dev,
                                    float softmax_scale, int32_t max_kv_len, int32_t* status_dev,
                                    void* stream);

/* ---------------------------------------------------------------- sizes and helpers */

/*
 * Bytes of each buffer of one sequence at capacity cap_tokens, in kivi_seq
 * field order (k_codes, k_scale, k_zero, v_codes, v_scale, v_zero, k_res,
 * v_res). Returns KIVI_ERR_ARG for a bad config or cap_tokens % G != 0.
 */
kivi_status kivi_seq_buffer_bytes(const kivi_cfg* cfg, int32_t cap_tokens, size_t bytes_out[8]);

/* Total bytes of one sequence's buffers (the sum of the above), -1 on error. */
int64_t kivi_seq_bytes(const kivi_cfg* cfg, int32_t cap_tokens);

/*
 * KV-cache bytes with no quantization metadata and no residual window: the
 * closed form the pages use for cache size, 2 (K and V) x layers x kv_heads x
 * head_dim x bits / 8 x tokens x batch ("KV-Cache Quantization: I Ran the
 * Experiments So You Don't Have To", section "Component 1", the table under
 * Figure 3 and the figures beside it: 128 KiB per token for Llama-3-8B at fp16,
 * about 275 GB for 64 requests of 32K tokens; section "The memory math
 * (verified)"). bits is 2, 4, 8 or 16. Compare kivi_seq_bytes, which counts the
 * scales, zeros and ring this library stores. Returns -1 for bits outside that
 * set, a negative size, or a product beyond int64.
 */
int64_t kivi_kv_bytes_plain(int32_t layers, int32_t num_kv_heads, int32_t head_dim, int32_t bits, int64_t tokens,
                            int64_t batch);

/* n_packed(L) for this config (see above), -1 on a bad config or L < 0. */
int64_t kivi_n_packed(const kivi_cfg* cfg, int64_t kv_len);

/* Static description of a status code. */
const char* kivi_status_string(int32_t status);

/* KIVI_ABI_VERSION of the loaded library. */
int32_t kivi_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KIVI_H */
