// Internal declarations shared by the CUDA translation units of the KIVI
// library: device helpers for the storage formats, the quantizer of one
// min/max group, and the internal launchers called by the C ABI layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kivi.h"

namespace kivi {

// G (tokens per key group, channels per value group) is 32 or 64. Kernels work in
// tiles of 32 tokens: a packed group is one or two whole tiles.
constexpr int kTile = 32;
constexpr int kMaxHeadDim = 256;

// ---------------------------------------------------------------- formats

template <int DT>
__device__ __forceinline__ float widen(uint16_t v) {
    if constexpr (DT == KIVI_BF16) {
        return __uint_as_float(static_cast<uint32_t>(v) << 16);
    } else {
        return __half2float(__ushort_as_half(v));
    }
}

__device__ __forceinline__ float f16_bits_to_float(uint16_t v) {
    return __half2float(__ushort_as_half(v));
}

// ---------------------------------------------------------------- quantizer

// Scale and zero of one group from its min and max: s = fp16(fp32(mx - mn) / qmax),
// z = fp16(mn), both round-to-nearest-even, with one IEEE fp32 subtraction and one
// IEEE fp32 division. Returns the stored fp16 patterns and their fp32 widening.
struct GroupParams {
    uint16_t s16, z16;
    float s, z;
};

__device__ __forceinline__ GroupParams group_params(float mn, float mx, int qmax) {
    const float s32 = __fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(qmax));
    const __half hs = __float2half_rn(s32);
    const __half hz = __float2half_rn(mn);
    GroupParams p;
    p.s16 = __half_as_ushort(hs);
    p.z16 = __half_as_ushort(hz);
    p.s = __half2float(hs);
    p.z = __half2float(hz);
    return p;
}

// Code of one element: clamp(rint((x - z) / s), 0, qmax), IEEE fp32 subtraction and
// division, round half to even; 0 when s == 0.
__device__ __forceinline__ uint32_t encode(float x, float z, float s, int qmax) {
    if (s == 0.0f) return 0u;
    float t = rintf(__fdiv_rn(__fsub_rn(x, z), s));
    t = fminf(fmaxf(t, 0.0f), static_cast<float>(qmax));
    return static_cast<uint32_t>(t);
}

// ---------------------------------------------------------------- cache state

__host__ __device__ __forceinline__ int64_t n_packed(int64_t L, int R, int G) {
    const int64_t over = L - R;
    return over <= 0 ? 0 : (over / G) * G;
}

// Addresses of packed group j of kv head h of a sequence, in either layout of kivi.h:
// its G key code rows (kb bits per code), D key scales and zeros, G value code rows (vb
// bits per code) and G x (D / G) value scales and zeros. page is block_table[j] for a
// paged sequence (ignored otherwise).
struct GroupAddr {
    uint8_t* kc;
    uint16_t* ks;
    uint16_t* kz;
    uint8_t* vc;
    uint16_t* vs;
    uint16_t* vz;
};

__device__ __forceinline__ bool seq_paged(const kivi_seq& sq) { return (sq.flags & KIVI_SEQ_PAGED) != 0; }

__device__ __forceinline__ GroupAddr group_addr(const kivi_seq& sq, int H, int h, int64_t j, int32_t page, int D,
                                                int kb, int vb, int G) {
    const int64_t ng = D / G;
    int64_t row0, meta;   // first code row of the group, and its (head, group) metadata row
    if (seq_paged(sq)) {
        const int64_t pg = static_cast<int64_t>(page) * H + h;
        row0 = pg * G;
        meta = pg;
    } else {
        const int64_t cap = sq.cap_tokens;
        row0 = h * cap + j * G;
        meta = h * (cap / G) + j;
    }
    GroupAddr a;
    a.kc = sq.k_codes + row0 * (static_cast<int64_t>(D) * kb / 8);
    a.ks = sq.k_scale + meta * D;
    a.kz = sq.k_zero + meta * D;
    a.vc = sq.v_codes + row0 * (static_cast<int64_t>(D) * vb / 8);
    a.vs = sq.v_scale + row0 * ng;
    a.vz = sq.v_zero + row0 * ng;
    return a;
}

__device__ __forceinline__ int32_t group_page(const kivi_seq& sq, int64_t j) {
    return seq_paged(sq) ? sq.block_table[j] : 0;
}

// The same for 32-token tile jt of the packed tokens (group jt / (G / 32)): its code
// rows and value metadata rows, and the key scales and zeros of its group.
__device__ __forceinline__ GroupAddr tile_addr(const kivi_seq& sq, int H, int h, int64_t jt, int D, int kb, int vb,
                                               int G) {
    const int tpg = G / kTile;
    const int64_t j = jt / tpg, sub = (jt - j * tpg) * kTile;
    GroupAddr a = group_addr(sq, H, h, j, group_page(sq, j), D, kb, vb, G);
    a.kc += sub * (static_cast<int64_t>(D) * kb / 8);
    a.vc += sub * (static_cast<int64_t>(D) * vb / 8);
    a.vs += sub * (D / G);
    a.vz += sub * (D / G);
    return a;
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- launchers

struct CodecArgs {
    int bits, G, D, dtype;
    int n_streams, n_tokens;
    const void* x;
    uint8_t* codes;
    uint16_t* scale;
    uint16_t* zero;
};

cudaError_t launch_quant_keys(const CodecArgs& a, cudaStream_t stream);
cudaError_t launch_quant_values(const CodecArgs& a, cudaStream_t stream);

struct AppendArgs {
    int kb, vb, G, D, R, H, dtype;
    int nseq, max_new;
    const kivi_seq* seqs;
    int32_t* kv_len;
    const void* const* k_new;
    const void* const* v_new;
    const int32_t* n_new;
    int32_t* status;
};

cudaError_t launch_append_flush(const AppendArgs& a, cudaStream_t stream);

struct DecodeArgs {
    int kb, vb, G, D, R, Hq, H, dtype;
    int nseq, max_kv_len;
    int n_query;                    // queries per sequence of multi-query attention (0: decode)
    int chunk, max_splits;          // tokens per split (multiple of 32), splits per sequence
    const kivi_seq* seqs;
    const int32_t* kv_len;
    const void* q;
    float* out;
    float scale_log2;               // softmax_scale * log2(e)
    int32_t* counters;              // [nseq][H] split tickets (workspace)
    float* partials;                // [nseq][Hq][max_splits][D + 4] (workspace)
    int32_t* status;
};

// Bound on the persistent decode grid (CTAs); sizes its workspace.
constexpr int kDecodeMaxCtas = 1024;

// Workspace of decode_mma_kernel: tickets (unused by it), then records for streams of `per`
// query heads, streams_per_kv_head per (sequence, kv head).
void mma_plan(int nseq, int H, int D, int per, int streams_per_kv_head, size_t* counter_bytes, size_t* partial_bytes);

// Split policy and workspace layout shared by kivi_decode_workspace_bytes and the launch.
void decode_plan(int nseq, int H, int Hq, int D, int max_kv_len, int* chunk, int* max_splits,
                 size_t* counter_bytes, size_t* partial_bytes);

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// Multi-query attention (kivi_decode_multi_attn): split plan and workspace, and the launch.
void multi_plan(int nseq, int H, int Hq, int D, int n_query, int max_kv_len, int* chunk, int* max_splits,
                size_t* counter_bytes, size_t* partial_bytes);
cudaError_t launch_multi(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_multi_k2v2(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_multi_k2v4(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_multi_k4v2(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_multi_k4v4(const DecodeArgs& a, cudaStream_t stream);
// One per pair of key / value code widths, each in a translation unit of its own.
cudaError_t launch_decode_k2v2(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_k2v4(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_k4v2(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_k4v4(const DecodeArgs& a, cudaStream_t stream);

}  // namespace kivi
