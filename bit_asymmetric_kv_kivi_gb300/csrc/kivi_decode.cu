// Split-K decode attention over the KIVI packed cache (sm_103a).
//
// One query token per sequence attends to every cached token: packed tokens
// are dequantized on the fly as c*s + z (keys: scale/zero per (group of 32
// tokens, channel); values: per (token, group of 32 channels)), residual
// tokens are read as stored. "KIVI: Asymmetric 2-Bit KV Cache Quantization
// Guide", sections "Step 2" (dequantize during attention) and "Production
// Serving and vLLM Deployment Trade-offs in 2026" (on-the-fly dequantization
// in SRAM); "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache",
// abstract (decode is bound by loading the cache).
//
// Work decomposition. A CTA owns one (sequence b, kv head h, split) where a
// split is a range of `chunk` tokens (a multiple of 32, so every 32-token tile
// is either wholly packed, i.e. one key group, or wholly residual). Its four
// warps take 32-token tiles round-robin, lane = token. All g = Hq/Hkv query
// heads of the kv head are handled together, so the cache is read once per
// kv head. Each warp keeps an online-softmax state (running max m, sum l and
// the fp32 accumulator of its 4 channels per lane), the warps are merged in
// shared memory, and the split's (m, l, acc) goes to the workspace. The last
// CTA of (b, h) to finish (an atomic ticket, no waiting) merges the splits
// with the usual log-sum-exp rescaling and writes the fp32 output.
//
// Key side per packed tile: q'[hq][d] = q[hq][d] * s_k[d] (the softmax scale
// and log2(e) folded into q) and bias[hq] = sum_d q[hq][d] * z_k[d] are formed
// once per group, so each token's score is bias + sum_d q'[d] * c[d].
#include <math_constants.h>

#include "kivi_internal.cuh"

namespace kivi {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kD = 128;          // head_dim handled by this kernel
constexpr int kCpl = kD / 32;    // channels per lane in the value accumulator

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int BITS, int DT, int GQ>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(DecodeArgs a) {
    constexpr int qmax = (1 << BITS) - 1;
    constexpr int kRowWords = kD * BITS / 32;     // 32-bit words per packed row
    constexpr int kPerWord = 32 / BITS;           // codes per word
    constexpr int kNg = kD / kGroup;              // value channel groups per token

    __shared__ float qs[GQ][kD];                                  // q * scale * log2(e)
    __shared__ float qk[kWarps][GQ][kD];                          // per warp: q' of the current key group
    __shared__ uint32_t vcode[kWarps][kGroup][kRowWords];         // per warp: value code rows of the tile
    __shared__ float vsc[kWarps][kGroup][kNg], vzr[kWarps][kGroup][kNg];
    __shared__ float red_m[kWarps][GQ], red_l[kWarps][GQ];
    __shared__ int s_last;

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hq = a.Hq, ring = a.R + kGroup;
    const kivi_seq& sq = a.seqs[b];
    const int cap = sq.cap_tokens;
    const int64_t L = a.kv_len[b];
    float* out_bh = a.out + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(h) * GQ) * kD;

    const bool bad = L < 0 || L > a.max_kv_len || n_packed(L, a.R) > cap;
    if (bad || L == 0) {
        if (split == 0) {
            for (int i = tid; i < GQ * kD; i += kThreads) out_bh[i] = bad ? CUDART_NAN_F : 0.0f;
            if (bad && h == 0 && tid == 0) set_status(a.status, KIVI_ERR_LENGTH);
        }
        return;
    }
    const int nsplit = static_cast<int>((L + a.chunk - 1) / a.chunk);
    if (split >= nsplit) return;
    const int64_t t0 = static_cast<int64_t>(split) * a.chunk;
    const int64_t t1 = min(t0 + a.chunk, L);
    const int64_t np = n_packed(L, a.R);

    const uint16_t* q = static_cast<const uint16_t*>(a.q) + (static_cast<int64_t>(b) * Hq + h * GQ) * kD;
    for (int i = tid; i < GQ * kD; i += kThreads) (&qs[0][0])[i] = widen<DT>(q[i]) * a.scale_log2;
    __syncthreads();

    float m[GQ], l[GQ], acc[GQ][kCpl];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        m[hh] = -CUDART_INF_F;
        l[hh] = 0.0f;
#pragma unroll
        for (int c = 0; c < kCpl; ++c) acc[hh][c] = 0.0f;
    }

    const uint16_t* kres = static_cast<const uint16_t*>(sq.k_res) + static_cast<int64_t>(h) * ring * kD;
    const uint16_t* vres = static_cast<const uint16_t*>(sq.v_res) + static_cast<int64_t>(h) * ring * kD;

    for (int64_t ts = t0 + 32 * warp; ts < t1; ts += 32 * kWarps) {
        const int64_t p = ts + lane;
        const bool valid = p < t1;
        const bool packed = ts < np;   // whole tile: np and ts are multiples of 32
        float sc[GQ];
        if (packed) {
            const int64_t j = ts / kGroup;
            const uint16_t* ksc = sq.k_scale + (static_cast<int64_t>(h) * (cap / kGroup) + j) * kD;
            const uint16_t* kzr = sq.k_zero + (static_cast<int64_t>(h) * (cap / kGroup) + j) * kD;
            float bias[GQ];
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) bias[hh] = 0.0f;
#pragma unroll
            for (int i = 0; i < kD / 32; ++i) {
                const int d = lane + 32 * i;
                const float s = f16_bits_to_float(ksc[d]), z = f16_bits_to_float(kzr[d]);
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                    qk[warp][hh][d] = qs[hh][d] * s;
                    bias[hh] = fmaf(qs[hh][d], z, bias[hh]);
                }
            }
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) sc[hh] = warp_sum(bias[hh]);
            // this lane's value codes and value scale/zero into the warp's tile
            const int64_t tok = static_cast<int64_t>(h) * cap + p;
            const uint4* vrow = reinterpret_cast<const uint4*>(sq.v_codes + tok * (kD * BITS / 8));
#pragma unroll
            for (int w = 0; w < kRowWords / 4; ++w)
                *reinterpret_cast<uint4*>(&vcode[warp][lane][4 * w]) = __ldg(vrow + w);
#pragma unroll
            for (int k = 0; k < kNg; ++k) {
                vsc[warp][lane][k] = f16_bits_to_float(sq.v_scale[tok * kNg + k]);
                vzr[warp][lane][k] = f16_bits_to_float(sq.v_zero[tok * kNg + k]);
            }
            __syncwarp();
            const uint4* krow = reinterpret_cast<const uint4*>(sq.k_codes + tok * (kD * BITS / 8));
#pragma unroll
            for (int w4 = 0; w4 < kRowWords / 4; ++w4) {
                const uint4 v4 = __ldg(krow + w4);
                const uint32_t words[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
#pragma unroll
                    for (int i = 0; i < kPerWord; ++i) {
                        const int d = (4 * w4 + e) * kPerWord + i;
                        const float c = static_cast<float>((words[e] >> (i * BITS)) & qmax);
#pragma unroll
                        for (int hh = 0; hh < GQ; ++hh) sc[hh] = fmaf(qk[warp][hh][d], c, sc[hh]);
                    }
                }
            }
        } else {
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) sc[hh] = 0.0f;
            if (valid) {
                const uint4* krow = reinterpret_cast<const uint4*>(kres + (p % ring) * kD);
#pragma unroll 4
                for (int w = 0; w < kD / 8; ++w) {
                    const uint4 v4 = __ldg(krow + w);
                    const uint32_t words[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float k0 = widen<DT>(static_cast<uint16_t>(words[e] & 0xffffu));
                        const float k1 = widen<DT>(static_cast<uint16_t>(words[e] >> 16));
                        const int d = 8 * w + 2 * e;
#pragma unroll
                        for (int hh = 0; hh < GQ; ++hh)
                            sc[hh] = fmaf(qs[hh][d + 1], k1, fmaf(qs[hh][d], k0, sc[hh]));
                    }
                }
            }
        }

        // online softmax over this tile (base 2: the scale already holds log2(e))
        float pr[GQ];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
            const float tmax = warp_max(valid ? sc[hh] : -CUDART_INF_F);
            const float mnew = fmaxf(m[hh], tmax);
            const float alpha = exp2f(m[hh] - mnew);
            pr[hh] = valid ? exp2f(sc[hh] - mnew) : 0.0f;
            l[hh] = l[hh] * alpha + warp_sum(pr[hh]);
#pragma unroll
            for (int c = 0; c < kCpl; ++c) acc[hh][c] *= alpha;
            m[hh] = mnew;
        }

        if (packed) {
            // lane owns channels [4 lane, 4 lane + 4): value channel group lane / 8
            const int kg = (lane * kCpl) / kGroup;
            for (int tau = 0; tau < 32; ++tau) {
                const uint32_t bitsv = (vcode[warp][tau][(lane * kCpl * BITS) / 32] >> ((lane * kCpl * BITS) % 32));
                const float s = vsc[warp][tau][kg], z = vzr[warp][tau][kg];
                float v[kCpl];
#pragma unroll
                for (int c = 0; c < kCpl; ++c) v[c] = fmaf(static_cast<float>((bitsv >> (c * BITS)) & qmax), s, z);
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                    const float pt = __shfl_sync(0xffffffffu, pr[hh], tau);
#pragma unroll
                    for (int c = 0; c < kCpl; ++c) acc[hh][c] = fmaf(pt, v[c], acc[hh][c]);
                }
            }
        } else {
            const int ntok = static_cast<int>(t1 - ts < 32 ? t1 - ts : 32);
            for (int tau = 0; tau < ntok; ++tau) {
                const uint2 raw = __ldg(reinterpret_cast<const uint2*>(vres + ((ts + tau) % ring) * kD + lane * kCpl));
                const float v[kCpl] = {widen<DT>(static_cast<uint16_t>(raw.x & 0xffffu)),
                                       widen<DT>(static_cast<uint16_t>(raw.x >> 16)),
                                       widen<DT>(static_cast<uint16_t>(raw.y & 0xffffu)),
                                       widen<DT>(static_cast<uint16_t>(raw.y >> 16))};
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                    const float pt = __shfl_sync(0xffffffffu, pr[hh], tau);
#pragma unroll
                    for (int c = 0; c < kCpl; ++c) acc[hh][c] = fmaf(pt, v[c], acc[hh][c]);
                }
            }
        }
        __syncwarp();
    }

    // merge the four warps (the per-warp key tiles are reused as the accumulator exchange)
    __syncthreads();
    float* red_acc = &qk[0][0][0];   // [kWarps][GQ][kD]
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        if (lane == 0) {
            red_m[warp][hh] = m[hh];
            red_l[warp][hh] = l[hh];
        }
#pragma unroll
        for (int c = 0; c < kCpl; ++c) red_acc[(warp * GQ + hh) * kD + lane * kCpl + c] = acc[hh][c];
    }
    __syncthreads();
    const int64_t rec_stride = kD + 4;
    float* part_bh = a.partials + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(h) * GQ) * a.max_splits * rec_stride;
    for (int i = tid; i < GQ * kD; i += kThreads) {
        const int hh = i / kD, d = i - hh * kD;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w][hh]);
        float den = 0.0f, num = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = exp2f(red_m[w][hh] - M);
            den = fmaf(red_l[w][hh], f, den);
            num = fmaf(red_acc[(w * GQ + hh) * kD + d], f, num);
        }
        if (nsplit == 1) {
            out_bh[i] = num / den;
        } else {
            float* rec = part_bh + (static_cast<int64_t>(hh) * a.max_splits + split) * rec_stride;
            rec[d] = num;
            if (d == 0) {
                rec[kD] = M;
                rec[kD + 1] = den;
            }
        }
    }
    if (nsplit == 1) return;

    // split combine: the last CTA of (b, h) to arrive merges every split
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int ticket = atomicAdd(&a.counters[static_cast<int64_t>(b) * a.H + h], 1);
        s_last = ticket == nsplit - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int i = tid; i < GQ * kD; i += kThreads) {
        const int hh = i / kD, d = i - hh * kD;
        const float* rec = part_bh + static_cast<int64_t>(hh) * a.max_splits * rec_stride;
        float M = -CUDART_INF_F, den = 0.0f, num = 0.0f;
        for (int s = 0; s < nsplit; ++s) {
            const float ms = __ldcg(rec + s * rec_stride + kD);
            const float Mn = fmaxf(M, ms);
            const float fo = exp2f(M - Mn), fs = exp2f(ms - Mn);
            den = den * fo + __ldcg(rec + s * rec_stride + kD + 1) * fs;
            num = num * fo + __ldcg(rec + s * rec_stride + d) * fs;
            M = Mn;
        }
        out_bh[i] = num / den;
    }
    if (tid == 0) a.counters[static_cast<int64_t>(b) * a.H + h] = 0;
}

template <int BITS, int DT>
cudaError_t launch_gq(const DecodeArgs& a, dim3 grid, cudaStream_t stream) {
    switch (a.Hq / a.H) {
        case 1: decode_split_kernel<BITS, DT, 1><<<grid, kThreads, 0, stream>>>(a); break;
        case 2: decode_split_kernel<BITS, DT, 2><<<grid, kThreads, 0, stream>>>(a); break;
        case 4: decode_split_kernel<BITS, DT, 4><<<grid, kThreads, 0, stream>>>(a); break;
        case 8: decode_split_kernel<BITS, DT, 8><<<grid, kThreads, 0, stream>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

void decode_plan(int nseq, int H, int Hq, int D, int max_kv_len, int* chunk, int* max_splits,
                 size_t* counter_bytes, size_t* partial_bytes) {
    // Split size: about an eighth of the longest sequence, in whole 256-token
    // steps, between 512 and 8192 tokens.
    const int64_t eighth = (static_cast<int64_t>(max_kv_len) + 7) / 8;
    int64_t c = ((eighth + 255) / 256) * 256;
    c = c < 512 ? 512 : (c > 8192 ? 8192 : c);
    const int64_t ms = max_kv_len <= 0 ? 1 : (max_kv_len + c - 1) / c;
    *chunk = static_cast<int>(c);
    *max_splits = static_cast<int>(ms);
    *counter_bytes = ((static_cast<size_t>(nseq) * H * sizeof(int32_t) + 255) / 256) * 256;
    *partial_bytes = static_cast<size_t>(nseq) * Hq * ms * (D + 4) * sizeof(float);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    if (a.nseq == 0) return cudaSuccess;
    const dim3 grid(a.max_splits, a.H, a.nseq);
    if (a.bits == 2 && a.dtype == KIVI_F16) return launch_gq<2, KIVI_F16>(a, grid, stream);
    if (a.bits == 2) return launch_gq<2, KIVI_BF16>(a, grid, stream);
    if (a.dtype == KIVI_F16) return launch_gq<4, KIVI_F16>(a, grid, stream);
    return launch_gq<4, KIVI_BF16>(a, grid, stream);
}

}  // namespace kivi
