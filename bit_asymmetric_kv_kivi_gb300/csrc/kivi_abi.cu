// The extern "C" boundary of the KIVI library: argument validation on the
// host, sizes and workspace planning, and the launches. Every entry point
// checks its arguments before anything is enqueued, so an invalid call
// launches nothing and returns an error code.
#include <math.h>
#include <string.h>

#include "kivi_internal.cuh"

namespace {

bool cfg_ok(const kivi_cfg* c) {
    if (c == nullptr) return false;
    if (c->k_bits != 2 && c->k_bits != 4) return false;
    if (c->v_bits != 2 && c->v_bits != 4) return false;
    if (c->group != 32 && c->group != 64) return false;
    if (c->residual <= 0 || c->residual % c->group != 0) return false;
    if (c->head_dim <= 0 || c->head_dim % c->group != 0 || c->head_dim > kivi::kMaxHeadDim) return false;
    if (c->num_kv_heads <= 0 || c->num_kv_heads > 65535) return false;
    if (c->num_q_heads <= 0 || c->num_q_heads % c->num_kv_heads != 0) return false;
    if (c->dtype != KIVI_F16 && c->dtype != KIVI_BF16) return false;
    return true;
}

kivi_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KIVI_OK : KIVI_ERR_CUDA; }

kivi_status codec_common(const kivi_cfg* cfg, int bits, int32_t n_streams, int32_t n_tokens, const void* x,
                         uint8_t* codes, uint16_t* scale, uint16_t* zero, kivi::CodecArgs* a) {
    if (!cfg_ok(cfg)) return KIVI_ERR_ARG;
    if (n_streams < 0 || n_tokens < 0 || n_streams > 65535) return KIVI_ERR_ARG;
    if (n_streams > 0 && n_tokens > 0 &&
        (x == nullptr || codes == nullptr || scale == nullptr || zero == nullptr))
        return KIVI_ERR_ARG;
    a->bits = bits;
    a->G = cfg->group;
    a->D = cfg->head_dim;
    a->dtype = cfg->dtype;
    a->n_streams = n_streams;
    a->n_tokens = n_tokens;
    a->x = x;
    a->codes = codes;
    a->scale = scale;
    a->zero = zero;
    return KIVI_OK;
}

}  // namespace

extern "C" {

kivi_status kivi_quant_keys(const kivi_cfg* cfg, int32_t n_streams, int32_t n_tokens, const void* x_dev,
                            uint8_t* codes_dev, uint16_t* scale_dev, uint16_t* zero_dev, void* stream) {
    kivi::CodecArgs a;
    const kivi_status st = codec_common(cfg, cfg ? cfg->k_bits : 0, n_streams, n_tokens, x_dev, codes_dev, scale_dev,
                                        zero_dev, &a);
    if (st != KIVI_OK) return st;
    if (n_tokens % cfg->group != 0) return KIVI_ERR_ARG;
    return from_cuda(kivi::launch_quant_keys(a, static_cast<cudaStream_t>(stream)));
}

kivi_status kivi_quant_values(const kivi_cfg* cfg, int32_t n_streams, int32_t n_tokens, const void* x_dev,
                              uint8_t* codes_dev, uint16_t* scale_dev, uint16_t* zero_dev, void* stream) {
    kivi::CodecArgs a;
    const kivi_status st = codec_common(cfg, cfg ? cfg->v_bits : 0, n_streams, n_tokens, x_dev, codes_dev, scale_dev,
                                        zero_dev, &a);
    if (st != KIVI_OK) return st;
    return from_cuda(kivi::launch_quant_values(a, static_cast<cudaStream_t>(stream)));
}

kivi_status kivi_append_flush(const kivi_cfg* cfg, int32_t nseq, const kivi_seq* seqs_dev, int32_t* kv_len_dev,
                              const void* const* k_new_dev, const void* const* v_new_dev,
                              const int32_t* n_new_dev, int32_t max_new, int32_t* status_dev, void* stream) {
    if (!cfg_ok(cfg)) return KIVI_ERR_ARG;
    if (nseq < 0 || nseq > 65535 || max_new < 0) return KIVI_ERR_ARG;
    if (nseq == 0) return KIVI_OK;
    if (seqs_dev == nullptr || kv_len_dev == nullptr || k_new_dev == nullptr || v_new_dev == nullptr ||
        n_new_dev == nullptr || status_dev == nullptr)
        return KIVI_ERR_ARG;
    kivi::AppendArgs a;
    a.kb = cfg->k_bits;
    a.vb = cfg->v_bits;
    a.G = cfg->group;
    a.D = cfg->head_dim;
    a.R = cfg->residual;
    a.H = cfg->num_kv_heads;
    a.dtype = cfg->dtype;
    a.nseq = nseq;
    a.max_new = max_new;
    a.seqs = seqs_dev;
    a.kv_len = kv_len_dev;
    a.k_new = k_new_dev;
    a.v_new = v_new_dev;
    a.n_new = n_new_dev;
    a.status = status_dev;
    return from_cuda(kivi::launch_append_flush(a, static_cast<cudaStream_t>(stream)));
}

size_t kivi_decode_workspace_bytes(const kivi_cfg* cfg, int32_t nseq, int32_t max_kv_len) {
    if (!cfg_ok(cfg) || nseq < 0 || max_kv_len < 0) return 0;
    int chunk, max_splits;
    size_t cb, pb;
    kivi::decode_plan(nseq, cfg->num_kv_heads, cfg->num_q_heads, cfg->head_dim, max_kv_len, &chunk,
                      &max_splits, &cb, &pb);
    return cb + pb;
}

kivi_status kivi_decode_attn(const kivi_cfg* cfg, int32_t nseq, const kivi_seq* seqs_dev,
                             const int32_t* kv_len_dev, const void* q_dev, float* out_dev, float softmax_scale,
                             int32_t max_kv_len, void* workspace_dev, size_t workspace_bytes,
                             int32_t* status_dev, void* stream) {
    if (!cfg_ok(cfg)) return KIVI_ERR_ARG;
    if (nseq < 0 || nseq > 65535 || max_kv_len < 0 || !isfinite(softmax_scale)) return KIVI_ERR_ARG;
    const int g = cfg->num_q_heads / cfg->num_kv_heads;
    if (cfg->head_dim != 128 || g > 32) return KIVI_ERR_UNSUPPORTED;
    if (nseq == 0) return KIVI_OK;
    if (seqs_dev == nullptr || kv_len_dev == nullptr || q_dev == nullptr || out_dev == nullptr)
        return KIVI_ERR_ARG;
    kivi::DecodeArgs a;
    size_t cb, pb;
    kivi::decode_plan(nseq, cfg->num_kv_heads, cfg->num_q_heads, cfg->head_dim, max_kv_len, &a.chunk,
                      &a.max_splits, &cb, &pb);
    if (workspace_dev == nullptr || workspace_bytes < cb + pb) return KIVI_ERR_WORKSPACE;
    a.kb = cfg->k_bits;
    a.vb = cfg->v_bits;
    a.G = cfg->group;
    a.D = cfg->head_dim;
    a.R = cfg->residual;
    a.Hq = cfg->num_q_heads;
    a.H = cfg->num_kv_heads;
    a.dtype = cfg->dtype;
    a.nseq = nseq;
    a.max_kv_len = max_kv_len;
    a.n_query = 0;
    a.seqs = seqs_dev;
    a.kv_len = kv_len_dev;
    a.q = q_dev;
    a.out = out_dev;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.counters = static_cast<int32_t*>(workspace_dev);
    a.partials = reinterpret_cast<float*>(static_cast<char*>(workspace_dev) + cb);
    a.status = status_dev;
    return from_cuda(kivi::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

// Multi-query calls that run on the persistent decode kernel: one query with a query group
// of 1, 2, 4 or 8 (decode attention; kv_len 0 stays a length error), several queries at a
// group of 4 or 8, and two queries at a group of 1 or 2 (one stream of the group's heads per
// query and kv head, each stopping at its query's causal end). Below four or eight (query,
// head) pairs per kv head that beat the multi-query kernel, whose shared unpack wins beyond.
static bool multi_is_decode(const kivi_cfg* cfg, int32_t n_query) {
    const int g = cfg->num_q_heads / cfg->num_kv_heads;
    return (n_query == 1 && (g == 1 || g == 2 || g == 4 || g == 8)) || (n_query > 1 && (g == 4 || g == 8)) ||
           (n_query == 2 && (g == 1 || g == 2));
}

static void multi_or_decode_plan(const kivi_cfg* cfg, int32_t nseq, int32_t n_query, int32_t max_kv_len, int* chunk,
                                 int* max_splits, size_t* cb, size_t* pb) {
    if (multi_is_decode(cfg, n_query) && n_query == 1) {
        kivi::decode_plan(nseq, cfg->num_kv_heads, cfg->num_q_heads, cfg->head_dim, max_kv_len, chunk, max_splits, cb,
                          pb);
    } else if (multi_is_decode(cfg, n_query)) {
        *chunk = 0;   // n_query streams of the group's heads per kv head
        *max_splits = 0;
        kivi::mma_plan(nseq, cfg->num_kv_heads, cfg->head_dim, cfg->num_q_heads / cfg->num_kv_heads, n_query, cb, pb);
    } else
        kivi::multi_plan(nseq, cfg->num_kv_heads, cfg->num_q_heads, cfg->head_dim, n_query, max_kv_len, chunk,
                         max_splits, cb, pb);
}

size_t kivi_decode_multi_workspace_bytes(const kivi_cfg* cfg, int32_t nseq, int32_t n_query, int32_t max_kv_len) {
    if (!cfg_ok(cfg) || nseq < 0 || max_kv_len < 0 || n_query < 1) return 0;
    int chunk, max_splits;
    size_t cb, pb;
    multi_or_decode_plan(cfg, nseq, n_query, max_kv_len, &chunk, &max_splits, &cb, &pb);
    return cb + pb;
}

kivi_status kivi_decode_multi_attn(const kivi_cfg* cfg, int32_t nseq, const kivi_seq* seqs_dev,
                                   const int32_t* kv_len_dev, int32_t n_query, const void* q_dev, float* out_dev,
                                   float softmax_scale, int32_t max_kv_len, void* workspace_dev,
                                   size_t workspace_bytes, int32_t* status_dev, void* stream) {
    if (!cfg_ok(cfg)) return KIVI_ERR_ARG;
    if (nseq < 0 || nseq > 65535 || max_kv_len < 0 || n_query < 1 || !isfinite(softmax_scale)) return KIVI_ERR_ARG;
    const int g = cfg->num_q_heads / cfg->num_kv_heads;
    if (cfg->head_dim != 128 || static_cast<int64_t>(n_query) * g > 32) return KIVI_ERR_UNSUPPORTED;
    if (nseq == 0) return KIVI_OK;
    if (seqs_dev == nullptr || kv_len_dev == nullptr || q_dev == nullptr || out_dev == nullptr)
        return KIVI_ERR_ARG;
    kivi::DecodeArgs a;
    size_t cb, pb;
    multi_or_decode_plan(cfg, nseq, n_query, max_kv_len, &a.chunk, &a.max_splits, &cb, &pb);
    if (workspace_dev == nullptr || workspace_bytes < cb + pb) return KIVI_ERR_WORKSPACE;
    a.kb = cfg->k_bits;
    a.vb = cfg->v_bits;
    a.G = cfg->group;
    a.D = cfg->head_dim;
    a.R = cfg->residual;
    a.Hq = cfg->num_q_heads;
    a.H = cfg->num_kv_heads;
    a.dtype = cfg->dtype;
    a.nseq = nseq;
    a.max_kv_len = max_kv_len;
    a.n_query = n_query;
    a.seqs = seqs_dev;
    a.kv_len = kv_len_dev;
    a.q = q_dev;
    a.out = out_dev;
    a.scale_log2 = softmax_scale * 1.4426950408889634f;
    a.counters = static_cast<int32_t*>(workspace_dev);
    a.partials = reinterpret_cast<float*>(static_cast<char*>(workspace_dev) + cb);
    a.status = status_dev;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    return from_cuda(multi_is_decode(cfg, n_query) ? kivi::launch_decode(a, st) : kivi::launch_multi(a, st));
}

kivi_status kivi_seq_buffer_bytes(const kivi_cfg* cfg, int32_t cap_tokens, size_t bytes_out[8]) {
    if (!cfg_ok(cfg) || cap_tokens < 0 || cap_tokens % cfg->group != 0 || bytes_out == nullptr) return KIVI_ERR_ARG;
    const size_t H = cfg->num_kv_heads, D = cfg->head_dim, cap = cap_tokens, G = cfg->group;
    const size_t esz = 2;  // fp16 and bf16
    const size_t kcodes = H * cap * D * cfg->k_bits / 8, vcodes = H * cap * D * cfg->v_bits / 8;
    const size_t kmeta = H * (cap / G) * D * 2;
    const size_t vmeta = H * cap * (D / G) * 2;
    const size_t ring = H * (cfg->residual + G) * D * esz;
    const size_t sizes[8] = {kcodes, kmeta, kmeta, vcodes, vmeta, vmeta, ring, ring};
    memcpy(bytes_out, sizes, sizeof(sizes));
    return KIVI_OK;
}

int64_t kivi_seq_bytes(const kivi_cfg* cfg, int32_t cap_tokens) {
    size_t b[8];
    if (kivi_seq_buffer_bytes(cfg, cap_tokens, b) != KIVI_OK) return -1;
    int64_t total = 0;
    for (int i = 0; i < 8; ++i) total += static_cast<int64_t>(b[i]);
    return total;
}

int64_t kivi_kv_bytes_plain(int32_t layers, int32_t num_kv_heads, int32_t head_dim, int32_t bits, int64_t tokens,
                            int64_t batch) {
    if (bits != 2 && bits != 4 && bits != 8 && bits != 16) return -1;
    if (layers < 0 || num_kv_heads < 0 || head_dim < 0 || tokens < 0 || batch < 0) return -1;
    // bits of one token of one layer (K and V), then bytes: every factor is checked against
    // overflow before it is applied
    const int64_t lim = INT64_MAX;
    int64_t v = 2 * static_cast<int64_t>(num_kv_heads) * head_dim * bits;   // < 2^49
    const int64_t f[3] = {layers, tokens, batch};
    for (int i = 0; i < 3; ++i) {
        if (f[i] != 0 && v > lim / f[i]) return -1;
        v *= f[i];
    }
    return v / 8;
}

int64_t kivi_n_packed(const kivi_cfg* cfg, int64_t kv_len) {
    if (!cfg_ok(cfg) || kv_len < 0) return -1;
    return kivi::n_packed(kv_len, cfg->residual, cfg->group);
}

const char* kivi_status_string(int32_t status) {
    switch (status) {
        case KIVI_OK: return "ok";
        case KIVI_ERR_ARG: return "invalid argument or configuration";
        case KIVI_ERR_UNSUPPORTED: return "configuration not supported by this library";
        case KIVI_ERR_CAPACITY: return "append exceeds the packed capacity of a sequence";
        case KIVI_ERR_WORKSPACE: return "workspace missing or too small";
        case KIVI_ERR_CUDA: return "CUDA launch or runtime error";
        case KIVI_ERR_LENGTH: return "sequence length or new-token count out of range";
        default: return "unknown status";
    }
}

int32_t kivi_abi_version(void) { return KIVI_ABI_VERSION; }

}  // extern "C"
