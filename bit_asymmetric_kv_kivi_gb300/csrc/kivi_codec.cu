// KIVI codec kernels for sm_103a: per-channel key quantization, per-token
// value quantization, and the append + group flush of a decode step or a
// prefill.
//
// Method: "KIVI: Asymmetric 2-Bit KV Cache Quantization Guide", section "The
// Three Structural Innovations of KIVI" (keys grouped along tokens per
// channel, values grouped along channels per token, a residual FIFO window
// whose overflow is grouped and packed) and its "Step 1" min/max quantizer;
// group and window sizes from "KV cache quantization with KIVI INT2 setup
// guide 2026" (G = 32, R = 128).
//
// Design. One CTA of 128 threads quantizes one 32-token group tile of one
// kv head: the tile (32 x D, 16-bit) is staged into shared memory with
// 16-byte loads, per-group min/max and the fp16 scale/zero are computed
// there, and every thread then emits whole 32-bit words of packed codes, so
// the code rows leave the SM as coalesced word stores. These kernels stream
// 16 bits in and 3 (2-bit) bits out per element; they are HBM-bound.
#include "kivi_internal.cuh"

namespace kivi {
namespace {

constexpr int kThreads = 128;
constexpr int kPad = 8;  // row padding of the shared tile, in 16-bit elements (keeps 16-byte rows)

// Copies rows [0, nrows) of a 32 x D tile of 16-bit elements into shared memory.
// row_src(t) returns the global address of row t (16-byte aligned).
template <typename RowSrc>
__device__ __forceinline__ void stage_tile(uint16_t* tile, int D, int nrows, RowSrc row_src) {
    const int chunks_per_row = D / 8;  // 16-byte chunks
    for (int c = threadIdx.x; c < nrows * chunks_per_row; c += kThreads) {
        const int t = c / chunks_per_row, part = c - t * chunks_per_row;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(row_src(t)) + part);
        *reinterpret_cast<uint4*>(tile + t * (D + kPad) + part * 8) = v;
    }
}

// Keys of one group (32 tokens x D channels in `tile`): per channel min/max
// over the 32 tokens, fp16 scale and zero into scale[d], zero[d], and the 32
// packed code rows into codes (row stride D*BITS/8 bytes).
template <int BITS, int DT>
__device__ void quantize_key_group(const uint16_t* tile, int D, uint8_t* codes, uint16_t* scale,
                                   uint16_t* zero, float* s_s, float* s_z) {
    constexpr int qmax = (1 << BITS) - 1;
    const int ld = D + kPad;
    for (int d = threadIdx.x; d < D; d += kThreads) {
        float mn = widen<DT>(tile[d]), mx = mn;
#pragma unroll 8
        for (int t = 1; t < kGroup; ++t) {
            const float v = widen<DT>(tile[t * ld + d]);
            mn = v < mn ? v : mn;   // first-seen wins on ties (+0 / -0), in token order
            mx = v > mx ? v : mx;
        }
        const GroupParams p = group_params(mn, mx, qmax);
        scale[d] = p.s16;
        zero[d] = p.z16;
        s_s[d] = p.s;
        s_z[d] = p.z;
    }
    __syncthreads();
    constexpr int per_word = 32 / BITS;
    const int wpr = D / per_word;  // 32-bit words per code row
    uint32_t* out = reinterpret_cast<uint32_t*>(codes);
    for (int w = threadIdx.x; w < kGroup * wpr; w += kThreads) {
        const int t = w / wpr, k = w - t * wpr;
        const int d0 = k * per_word;
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < per_word; ++i) {
            const int d = d0 + i;
            word |= encode(widen<DT>(tile[t * ld + d]), s_z[d], s_s[d], qmax) << (i * BITS);
        }
        out[w] = word;
    }
}

// Values of up to 32 tokens (rows [0, ntok) of `tile`): per token and per
// group of 32 channels, min/max, fp16 scale and zero into scale/zero
// [ntok][D/32], and the packed code rows.
template <int BITS, int DT>
__device__ void quantize_value_rows(const uint16_t* tile, int D, int ntok, uint8_t* codes,
                                    uint16_t* scale, uint16_t* zero, float* s_s, float* s_z) {
    constexpr int qmax = (1 << BITS) - 1;
    const int ld = D + kPad, ng = D / kGroup;
    for (int i = threadIdx.x; i < ntok * ng; i += kThreads) {
        const int t = i / ng, k = i - t * ng;
        const uint16_t* x = tile + t * ld + k * kGroup;
        float mn = widen<DT>(x[0]), mx = mn;
#pragma unroll 8
        for (int c = 1; c < kGroup; ++c) {
            const float v = widen<DT>(x[c]);
            mn = v < mn ? v : mn;   // first-seen wins on ties, in channel order
            mx = v > mx ? v : mx;
        }
        const GroupParams p = group_params(mn, mx, qmax);
        scale[i] = p.s16;
        zero[i] = p.z16;
        s_s[i] = p.s;
        s_z[i] = p.z;
    }
    __syncthreads();
    constexpr int per_word = 32 / BITS;
    const int wpr = D / per_word;
    uint32_t* out = reinterpret_cast<uint32_t*>(codes);
    for (int w = threadIdx.x; w < ntok * wpr; w += kThreads) {
        const int t = w / wpr, k = w - t * wpr;
        const int d0 = k * per_word;
        const float s = s_s[t * ng + d0 / kGroup], z = s_z[t * ng + d0 / kGroup];
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < per_word; ++i)
            word |= encode(widen<DT>(tile[t * ld + d0 + i]), z, s, qmax) << (i * BITS);
        out[w] = word;
    }
}

// ---------------------------------------------------------------- standalone codec

template <int BITS, int DT>
__global__ void __launch_bounds__(kThreads) quant_keys_kernel(CodecArgs a) {
    __shared__ __align__(16) uint16_t tile[kGroup * (kMaxHeadDim + kPad)];
    __shared__ float s_s[kMaxHeadDim], s_z[kMaxHeadDim];
    const int j = blockIdx.x, st = blockIdx.y, D = a.D;
    const int64_t tok0 = static_cast<int64_t>(st) * a.n_tokens + static_cast<int64_t>(j) * kGroup;
    const uint16_t* x = static_cast<const uint16_t*>(a.x);
    stage_tile(tile, D, kGroup, [&](int t) { return x + (tok0 + t) * D; });
    __syncthreads();
    const int64_t g = static_cast<int64_t>(st) * (a.n_tokens / kGroup) + j;
    quantize_key_group<BITS, DT>(tile, D, a.codes + tok0 * (D * BITS / 8), a.scale + g * D, a.zero + g * D,
                                 s_s, s_z);
}

template <int BITS, int DT>
__global__ void __launch_bounds__(kThreads) quant_values_kernel(CodecArgs a) {
    __shared__ __align__(16) uint16_t tile[kGroup * (kMaxHeadDim + kPad)];
    __shared__ float s_s[kGroup * (kMaxHeadDim / kGroup)], s_z[kGroup * (kMaxHeadDim / kGroup)];
    const int j = blockIdx.x, st = blockIdx.y, D = a.D;
    const int t_begin = j * kGroup;
    const int ntok = min(kGroup, a.n_tokens - t_begin);
    const int64_t tok0 = static_cast<int64_t>(st) * a.n_tokens + t_begin;
    const uint16_t* x = static_cast<const uint16_t*>(a.x);
    stage_tile(tile, D, ntok, [&](int t) { return x + (tok0 + t) * D; });
    __syncthreads();
    quantize_value_rows<BITS, DT>(tile, D, ntok, a.codes + tok0 * (D * BITS / 8),
                                  a.scale + tok0 * (D / kGroup), a.zero + tok0 * (D / kGroup), s_s, s_z);
}

// ---------------------------------------------------------------- append + flush

struct SeqState {
    bool ok;
    int64_t L, L1, np0, np1;
};

// Validity and flush range of one sequence for this append; identical in both kernels.
__device__ __forceinline__ SeqState seq_state(const AppendArgs& a, int b, int cap) {
    SeqState s;
    s.L = a.kv_len[b];
    const int64_t n = a.n_new[b];
    s.L1 = s.L + n;
    s.np0 = n_packed(s.L, a.R);
    s.np1 = n_packed(s.L1, a.R);
    s.ok = s.L >= 0 && n >= 0 && n <= a.max_new && s.np1 <= cap;
    return s;
}

// One CTA per (group slot, kv head, sequence): quantizes the gi-th group that
// this append makes leave the residual window. Tokens older than kv_len come
// from the ring, newer ones straight from the caller's new-token buffers.
template <int BITS, int DT>
__global__ void __launch_bounds__(kThreads) append_pack_kernel(AppendArgs a) {
    __shared__ __align__(16) uint16_t tk[kGroup * (kMaxHeadDim + kPad)];
    __shared__ __align__(16) uint16_t tv[kGroup * (kMaxHeadDim + kPad)];
    __shared__ float s_s[kMaxHeadDim], s_z[kMaxHeadDim];
    const int gi = blockIdx.x, h = blockIdx.y, b = blockIdx.z, D = a.D;
    const kivi_seq& sq = a.seqs[b];
    const int cap = sq.cap_tokens;
    const SeqState st = seq_state(a, b, cap);
    if (!st.ok) {
        if (gi == 0 && h == 0 && threadIdx.x == 0) {
            const bool len_bad = st.L < 0 || st.L1 < st.L || st.L1 - st.L > a.max_new;
            set_status(a.status, len_bad ? KIVI_ERR_LENGTH : KIVI_ERR_CAPACITY);
        }
        return;
    }
    const int64_t p0 = st.np0 + static_cast<int64_t>(gi) * kGroup;  // first token of the group
    if (p0 >= st.np1) return;
    const int ring = a.R + kGroup;
    const int64_t n = st.L1 - st.L;
    const uint16_t* kres = static_cast<const uint16_t*>(sq.k_res) + static_cast<int64_t>(h) * ring * D;
    const uint16_t* vres = static_cast<const uint16_t*>(sq.v_res) + static_cast<int64_t>(h) * ring * D;
    const uint16_t* knew = static_cast<const uint16_t*>(a.k_new[b]);
    const uint16_t* vnew = static_cast<const uint16_t*>(a.v_new[b]);
    auto src = [&](const uint16_t* res, const uint16_t* nw, int t) -> const uint16_t* {
        const int64_t p = p0 + t;
        if (p < st.L) return res + (p % ring) * D;
        return nw + (static_cast<int64_t>(h) * n + (p - st.L)) * D;
    };
    stage_tile(tk, D, kGroup, [&](int t) { return src(kres, knew, t); });
    stage_tile(tv, D, kGroup, [&](int t) { return src(vres, vnew, t); });
    __syncthreads();
    const int row_bytes = D * BITS / 8;
    const int64_t tok = static_cast<int64_t>(h) * cap + p0;
    const int64_t kg = static_cast<int64_t>(h) * (cap / kGroup) + p0 / kGroup;
    quantize_key_group<BITS, DT>(tk, D, sq.k_codes + tok * row_bytes, sq.k_scale + kg * D, sq.k_zero + kg * D,
                                 s_s, s_z);
    __syncthreads();
    quantize_value_rows<BITS, DT>(tv, D, kGroup, sq.v_codes + tok * row_bytes, sq.v_scale + tok * (D / kGroup),
                                  sq.v_zero + tok * (D / kGroup), s_s, s_z);
}

// One CTA per sequence: writes the new tokens that stay in the residual window
// into their ring slots, then advances kv_len. Runs after append_pack_kernel
// on the same stream, so every ring slot that a flush still had to read has
// been read before it is overwritten here.
__global__ void __launch_bounds__(256) append_ring_kernel(AppendArgs a) {
    const int b = blockIdx.x, D = a.D, H = a.H;
    const kivi_seq& sq = a.seqs[b];
    const SeqState st = seq_state(a, b, sq.cap_tokens);
    if (!st.ok) return;
    const int ring = a.R + kGroup;
    const int64_t n = st.L1 - st.L;
    const int64_t first = st.L > st.np1 ? st.L : st.np1;  // first position that stays in the ring
    const int64_t count = st.L1 - first;
    if (count > 0) {
        const uint16_t* knew = static_cast<const uint16_t*>(a.k_new[b]);
        const uint16_t* vnew = static_cast<const uint16_t*>(a.v_new[b]);
        uint16_t* kres = static_cast<uint16_t*>(sq.k_res);
        uint16_t* vres = static_cast<uint16_t*>(sq.v_res);
        const int cpr = D / 8;  // 16-byte chunks per row
        const int64_t total = count * H * cpr;
        for (int64_t c = threadIdx.x; c < total; c += blockDim.x) {
            const int part = static_cast<int>(c % cpr);
            const int64_t rowi = c / cpr;
            const int h = static_cast<int>(rowi % H);
            const int64_t p = first + rowi / H;
            const int64_t src = (static_cast<int64_t>(h) * n + (p - st.L)) * D + part * 8;
            const int64_t dst = (static_cast<int64_t>(h) * ring + p % ring) * D + part * 8;
            *reinterpret_cast<uint4*>(kres + dst) = __ldg(reinterpret_cast<const uint4*>(knew + src));
            *reinterpret_cast<uint4*>(vres + dst) = __ldg(reinterpret_cast<const uint4*>(vnew + src));
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) a.kv_len[b] = static_cast<int32_t>(st.L1);
}

}  // namespace

cudaError_t launch_quant_keys(const CodecArgs& a, cudaStream_t stream) {
    if (a.n_streams == 0 || a.n_tokens == 0) return cudaSuccess;
    const dim3 grid(a.n_tokens / kGroup, a.n_streams);
    if (a.bits == 2 && a.dtype == KIVI_F16) quant_keys_kernel<2, KIVI_F16><<<grid, kThreads, 0, stream>>>(a);
    else if (a.bits == 2) quant_keys_kernel<2, KIVI_BF16><<<grid, kThreads, 0, stream>>>(a);
    else if (a.dtype == KIVI_F16) quant_keys_kernel<4, KIVI_F16><<<grid, kThreads, 0, stream>>>(a);
    else quant_keys_kernel<4, KIVI_BF16><<<grid, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_quant_values(const CodecArgs& a, cudaStream_t stream) {
    if (a.n_streams == 0 || a.n_tokens == 0) return cudaSuccess;
    const dim3 grid((a.n_tokens + kGroup - 1) / kGroup, a.n_streams);
    if (a.bits == 2 && a.dtype == KIVI_F16) quant_values_kernel<2, KIVI_F16><<<grid, kThreads, 0, stream>>>(a);
    else if (a.bits == 2) quant_values_kernel<2, KIVI_BF16><<<grid, kThreads, 0, stream>>>(a);
    else if (a.dtype == KIVI_F16) quant_values_kernel<4, KIVI_F16><<<grid, kThreads, 0, stream>>>(a);
    else quant_values_kernel<4, KIVI_BF16><<<grid, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_append_flush(const AppendArgs& a, cudaStream_t stream) {
    if (a.nseq == 0) return cudaSuccess;
    const int max_groups = (a.max_new + kGroup - 1) / kGroup;
    if (max_groups > 0) {
        const dim3 grid(max_groups, a.H, a.nseq);
        if (a.bits == 2 && a.dtype == KIVI_F16) append_pack_kernel<2, KIVI_F16><<<grid, kThreads, 0, stream>>>(a);
        else if (a.bits == 2) append_pack_kernel<2, KIVI_BF16><<<grid, kThreads, 0, stream>>>(a);
        else if (a.dtype == KIVI_F16) append_pack_kernel<4, KIVI_F16><<<grid, kThreads, 0, stream>>>(a);
        else append_pack_kernel<4, KIVI_BF16><<<grid, kThreads, 0, stream>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    append_ring_kernel<<<a.nseq, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kivi
