// Decode attention for callers that cannot allocate device memory.
//
// kivi_decode_attn needs a caller-provided workspace (split partials and
// combine tickets). Some callers cannot allocate one: a process whose device
// memory is already reserved by another allocator (for example a serving
// framework's memory pool), a latency-critical path that must not call
// cudaMalloc/cudaFree (cudaFree synchronizes the whole device), or a plugin
// host whose interface hands over only input and output buffers. For them,
// kivi_decode_attn_static runs the same kernels with the workspace taken from
// a fixed-size array in this library's own device memory, which exists from
// the time the library's device code is loaded until the process exits.
// There is no counterpart of this entry point in the pages that describe KIVI.
//
// The array is shared by every call on a device and keeps what the last call
// left there; the entry point clears the part that must start at zero
// before each launch. Calls on the same device that overlap on the GPU race
// on it and give wrong results.
#include <math.h>

#include <mutex>

#include "kivi_internal.cuh"

namespace {

// The workspace of kivi_decode_attn_static. In host code this name is only a
// host-side stand-in for the symbol, not a device address: a kernel given it
// would fault or, where the GPU can reach host memory, silently use the wrong
// memory. Host code passes the address from cudaGetSymbolAddress instead.
static __device__ __align__(256) unsigned char g_static_ws[KIVI_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_ws_ptr[kMaxDevices] = {};   // device address of g_static_ws, per device

// Device address of the array on the current device, looked up once per
// device (with that device current) and cached for the life of the process.
// cudaDeviceReset tears down the context that holds the array, so after it the
// cached address is stale: a process that resets a device must not call
// kivi_decode_attn_static on that device again.
kivi_status static_workspace(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KIVI_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_ws_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr) return KIVI_ERR_CUDA;
        g_ws_ptr[dev] = p;
    }
    *out = g_ws_ptr[dev];
    return KIVI_OK;
}

}  // namespace

extern "C" kivi_status kivi_decode_attn_static(const kivi_cfg* cfg, int32_t nseq, const kivi_seq* seqs_dev,
                                               const int32_t* kv_len_dev, const void* q_dev, float* out_dev,
                                               float softmax_scale, int32_t max_kv_len, int32_t* status_dev,
                                               void* stream) {
    if (cfg == nullptr || nseq < 0 || max_kv_len < 0) return KIVI_ERR_ARG;
    if (nseq == 0)  // validates the config; launches nothing
        return kivi_decode_attn(cfg, 0, seqs_dev, kv_len_dev, q_dev, out_dev, softmax_scale, max_kv_len, nullptr, 0,
                                status_dev, stream);
    // Every check kivi_decode_attn makes before launching, made here before the memset below.
    const size_t need = kivi_decode_workspace_bytes(cfg, nseq, max_kv_len);
    if (need == 0 || seqs_dev == nullptr || kv_len_dev == nullptr || q_dev == nullptr || out_dev == nullptr ||
        !isfinite(softmax_scale) || nseq > 65535)
        return KIVI_ERR_ARG;
    const int g = cfg->num_q_heads / cfg->num_kv_heads;
    if (cfg->head_dim != 128 || g > 32) return KIVI_ERR_UNSUPPORTED;
    if (need > KIVI_STATIC_WORKSPACE_BYTES) return KIVI_ERR_WORKSPACE;
    void* ws = nullptr;
    const kivi_status st = static_workspace(&ws);
    if (st != KIVI_OK) return st;
    // The split-combine tickets at the front of the workspace must start at zero.
    int chunk, max_splits;
    size_t counter_bytes, partial_bytes;
    kivi::decode_plan(nseq, cfg->num_kv_heads, cfg->num_q_heads, cfg->head_dim, max_kv_len, &chunk, &max_splits,
                      &counter_bytes, &partial_bytes);
    if (cudaMemsetAsync(ws, 0, counter_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KIVI_ERR_CUDA;
    return kivi_decode_attn(cfg, nseq, seqs_dev, kv_len_dev, q_dev, out_dev, softmax_scale, max_kv_len, ws,
                            KIVI_STATIC_WORKSPACE_BYTES, status_dev, stream);
}
