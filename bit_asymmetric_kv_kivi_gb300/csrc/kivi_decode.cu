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
// Two kernels share the split bookkeeping:
//
//  * decode_mma_kernel (Hq/Hkv = 1, 2, 4): the dot products run on the tensor
//    cores (mma.sync m16n8k16, f16 operands, fp32 accumulation). A CTA owns a
//    range of whole 32-token key groups of one (sequence, kv head), or the
//    residual tokens of it (a split of its own). Each of its four warps
//    streams its groups through a private cp.async ring of shared-memory
//    stages and keeps its own online-softmax state.
//      - Scores: S[token][head] = sum_d c[token][d] * Q[d][head] + bias[head],
//        Q = q * s_k (softmax scale and log2(e) folded into q). Codes are the
//        A operand, unpacked to exact f16 integers (one lop3 + one fma per
//        pair). Q is the B operand as an f16 hi + lo pair (two columns per
//        head), built with an exact-error product in f16, so the sum carries
//        about 22 bits; bias = sum_d q z_k is one more small MMA.
//      - Values: O[d][head] += sum_t c[t][d] * P'[t][head] with
//        P' = p * s_v[t][group(d)] (hi + lo again), channels as M; the
//        sum_t p z_v term is a small MMA of its own.
//    q is rescaled by a power of two so that max|q| lies in (1/2, 1]; with
//    |x| <= 65504 no f16 operand can overflow.
//  * decode_split_kernel (any Hq/Hkv, used for 8): CUDA-core FMAs, lane = token.
//
// Every split writes (m, l, acc[128]) for its query heads to the workspace;
// the last CTA of a (sequence, kv head) to finish (an atomic ticket, no
// waiting) merges the splits with the log-sum-exp rescaling and writes the
// fp32 output.
#include <math_constants.h>

#include "kivi_internal.cuh"

namespace kivi {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kD = 128;          // head_dim handled by these kernels
constexpr int kCpl = kD / 32;    // channels per lane in the lane-layout value accumulator
constexpr int kStages = 4;       // cp.async ring depth per warp (decode_mma_kernel)
constexpr int kPtLd = 40;        // row stride (floats) of the per-warp probability transpose
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// f16x2 from two floats (round to nearest even): `lo` in bits 0-15, `hi` in 16-31.
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ float h2_lo(uint32_t v) { return __half2float(__ushort_as_half(static_cast<uint16_t>(v))); }
__device__ __forceinline__ float h2_hi(uint32_t v) { return __half2float(__ushort_as_half(static_cast<uint16_t>(v >> 16))); }

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Codes at bits I*BITS and 16 + I*BITS of w as an exact f16 pair (low, high half).
// The field is OR-ed into the mantissa of 1024.0 and the 1024 removed by one fma
// (the field's position scaled away by a power of two); fields that reach past the
// 10 mantissa bits are taken from ws = w >> (DIRECT * BITS).
template <int BITS, int I>
__device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t ws) {
    constexpr int kDirect = (10 - BITS) / BITS + 1;               // fields wholly inside bits 0..9
    constexpr int kPos = I < kDirect ? I * BITS : (I - kDirect) * BITS;
    constexpr uint32_t kMask = ((((1u << BITS) - 1u) << kPos) * 0x00010001u);
    constexpr uint32_t kScale = static_cast<uint32_t>((15 - kPos) << 10) * 0x00010001u;          // 2^-pos
    constexpr uint32_t kBias = static_cast<uint32_t>(0x8000 | ((25 - kPos) << 10)) * 0x00010001u;  // -2^(10-pos)
    const uint32_t src = I < kDirect ? w : ws;
    uint32_t h;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(h) : "r"(src), "r"(kMask), "r"(0x64006400u));  // (src & mask) | magic
    return hfma2(h, kScale, kBias);
}

// code_pair for a slot index known only after unrolling (folds to one case).
template <int BITS>
__device__ __forceinline__ uint32_t code_slot(uint32_t w, uint32_t ws, int s) {
    constexpr int kN = 16 / BITS;
    switch (s % kN) {
        case 0: return code_pair<BITS, 0>(w, ws);
        case 1: return code_pair<BITS, 1 % kN>(w, ws);
        case 2: return code_pair<BITS, 2 % kN>(w, ws);
        case 3: return code_pair<BITS, 3 % kN>(w, ws);
        case 4: return code_pair<BITS, 4 % kN>(w, ws);
        case 5: return code_pair<BITS, 5 % kN>(w, ws);
        case 6: return code_pair<BITS, 6 % kN>(w, ws);
        default: return code_pair<BITS, 7 % kN>(w, ws);
    }
}

template <int BITS>
struct CodeShift {
    static constexpr int kValue = ((10 - BITS) / BITS + 1) * BITS;   // 10 (2-bit), 8 (4-bit)
};

// ---------------------------------------------------------------- lane-layout pieces

// One 32-token tile of residual tokens [ts, min(ts+32, t1)) for one warp, lane = token:
// scores against the widened stored keys, online-softmax update and value accumulation
// into the lane-layout state (lane owns channels [4 lane, 4 lane + 4)).
template <int DT, int GQ>
__device__ __forceinline__ void residual_tile(const uint16_t* kres, const uint16_t* vres, int ring, int64_t ts,
                                              int64_t t1, const float* qs, int lane, float (&m)[GQ], float (&l)[GQ],
                                              float (&acc)[GQ][kCpl]) {
    const int64_t p = ts + lane;
    const bool valid = p < t1;
    float sc[GQ];
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
                for (int hh = 0; hh < GQ; ++hh) sc[hh] = fmaf(qs[hh * kD + d + 1], k1, fmaf(qs[hh * kD + d], k0, sc[hh]));
            }
        }
    }
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
    const int ntok = static_cast<int>(t1 - ts < 32 ? t1 - ts : 32);
    for (int tau = 0; tau < ntok; ++tau) {
        const uint2 raw = __ldg(reinterpret_cast<const uint2*>(vres + ((ts + tau) % ring) * kD + lane * kCpl));
        const float v[kCpl] = {widen<DT>(static_cast<uint16_t>(raw.x & 0xffffu)),
                               widen<DT>(static_cast<uint16_t>(raw.x >> 16)),
                               widen<DT>(static_cast<uint16_t>(raw.y & 0xffffu)),
                               widen<DT>(static_cast<uint16_t>(raw.y >> 16))};
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
            const float pt = __shfl_sync(kFull, pr[hh], tau);
#pragma unroll
            for (int c = 0; c < kCpl; ++c) acc[hh][c] = fmaf(pt, v[c], acc[hh][c]);
        }
    }
}

// Lane-layout warp state into the CTA merge arrays.
template <int GQ>
__device__ __forceinline__ void store_lane_state(int warp, int lane, const float (&m)[GQ], const float (&l)[GQ],
                                                 const float (&acc)[GQ][kCpl], float* red_m, float* red_l,
                                                 float* red_acc) {
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        if (lane == 0) {
            red_m[warp * GQ + hh] = m[hh];
            red_l[warp * GQ + hh] = l[hh];
        }
#pragma unroll
        for (int c = 0; c < kCpl; ++c) red_acc[(warp * GQ + hh) * kD + lane * kCpl + c] = acc[hh][c];
    }
}

// Merges the four warps' states of this split (red_* in shared memory, filled and
// synchronized by the caller), then either writes the output (single split) or
// the split's partial record; the last CTA of (b, h) to arrive merges all splits.
template <int GQ>
__device__ __forceinline__ void finish_split(const DecodeArgs& a, int b, int h, int split, int nsplit,
                                             float* out_bh, const float* red_m, const float* red_l,
                                             const float* red_acc, int* s_last) {
    const int tid = threadIdx.x;
    const int64_t rec_stride = kD + 4;
    float* part_bh =
        a.partials + (static_cast<int64_t>(b) * a.Hq + static_cast<int64_t>(h) * GQ) * a.max_splits * rec_stride;
    for (int i = tid; i < GQ * kD; i += kThreads) {
        const int hh = i / kD, d = i - hh * kD;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * GQ + hh]);
        float den = 0.0f, num = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = exp2f(red_m[w * GQ + hh] - M);
            den = fmaf(red_l[w * GQ + hh], f, den);
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
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int ticket = atomicAdd(&a.counters[static_cast<int64_t>(b) * a.H + h], 1);
        *s_last = ticket == nsplit - 1;
    }
    __syncthreads();
    if (!*s_last) return;
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

// ---------------------------------------------------------------- CUDA-core kernel

// Splits over [0, L) in chunks of a.chunk tokens; four warps take 32-token tiles
// round-robin, lane = token. Key side per packed tile: q'[hq][d] = q[hq][d] * s_k[d]
// and bias[hq] = sum_d q[hq][d] * z_k[d], so a token's score is bias + sum_d q'[d] c[d].
template <int BITS, int DT, int GQ>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(DecodeArgs a) {
    constexpr int qmax = (1 << BITS) - 1;
    constexpr int kRowWords = kD * BITS / 32;     // 32-bit words per packed row
    constexpr int kPerWord = 32 / BITS;           // codes per word
    constexpr int kNg = kD / kGroup;              // value channel groups per token

    __shared__ float qs[GQ * kD];                                 // q * scale * log2(e)
    __shared__ float qk[kWarps][GQ][kD];                          // per warp: q' of the current key group
    __shared__ uint32_t vcode[kWarps][kGroup][kRowWords];         // per warp: value code rows of the tile
    __shared__ float vsc[kWarps][kGroup][kNg], vzr[kWarps][kGroup][kNg];
    __shared__ float red_m[kWarps * GQ], red_l[kWarps * GQ];
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
    for (int i = tid; i < GQ * kD; i += kThreads) qs[i] = widen<DT>(q[i]) * a.scale_log2;
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
        if (ts >= np) {   // residual tile (np and ts are multiples of 32)
            residual_tile<DT, GQ>(kres, vres, ring, ts, t1, qs, lane, m, l, acc);
            __syncwarp();
            continue;
        }
        const int64_t p = ts + lane;   // packed tiles are always full
        const int64_t j = ts / kGroup;
        const uint16_t* ksc = sq.k_scale + (static_cast<int64_t>(h) * (cap / kGroup) + j) * kD;
        const uint16_t* kzr = sq.k_zero + (static_cast<int64_t>(h) * (cap / kGroup) + j) * kD;
        float sc[GQ], bias[GQ];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) bias[hh] = 0.0f;
#pragma unroll
        for (int i = 0; i < kD / 32; ++i) {
            const int d = lane + 32 * i;
            const float s = f16_bits_to_float(ksc[d]), z = f16_bits_to_float(kzr[d]);
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
                qk[warp][hh][d] = qs[hh * kD + d] * s;
                bias[hh] = fmaf(qs[hh * kD + d], z, bias[hh]);
            }
        }
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) sc[hh] = warp_sum(bias[hh]);
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
        float pr[GQ];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
            const float tmax = warp_max(sc[hh]);
            const float mnew = fmaxf(m[hh], tmax);
            const float alpha = exp2f(m[hh] - mnew);
            pr[hh] = exp2f(sc[hh] - mnew);
            l[hh] = l[hh] * alpha + warp_sum(pr[hh]);
#pragma unroll
            for (int c = 0; c < kCpl; ++c) acc[hh][c] *= alpha;
            m[hh] = mnew;
        }
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
                const float pt = __shfl_sync(kFull, pr[hh], tau);
#pragma unroll
                for (int c = 0; c < kCpl; ++c) acc[hh][c] = fmaf(pt, v[c], acc[hh][c]);
            }
        }
        __syncwarp();
    }

    __syncthreads();
    float* red_acc = &qk[0][0][0];   // [kWarps][GQ][kD]
    store_lane_state<GQ>(warp, lane, m, l, acc, red_m, red_l, red_acc);
    __syncthreads();
    finish_split<GQ>(a, b, h, split, nsplit, out_bh, red_m, red_l, red_acc, &s_last);
}

// ---------------------------------------------------------------- tensor-core kernel

template <int BITS>
struct MmaLayout {
    static constexpr int kRowBytes = kD * BITS / 8;                      // packed row: 32 or 64 bytes
    // kc, vc, ks, kz, vs, vz; each 64-byte channel span of ks and kz is padded to 80 bytes so
    // that the four spans read together fall on distinct shared-memory banks
    static constexpr int kMetaPad = 320;
    static constexpr int kStage = 2 * kGroup * kRowBytes + 2 * kMetaPad + 2 * 256;
    static constexpr int kChunks = (2 * kGroup * kRowBytes + 4 * 256) / 16;   // 16-byte cp.async pieces
    static constexpr int kNslot = 16 / BITS;                             // code pairs per 32-bit word
    static constexpr int kStageBytes = kWarps * kStages * kStage;
    static constexpr int kSmemBytes(int gq) {
        return kStageBytes + (gq * kD + kWarps * 4 * kPtLd + 2 * kWarps * gq + 8) * 4;
    }
};

// Splits: ceil(n_packed / chunk) ranges of whole key groups, then one split for the
// residual tokens. Thread (gid = lane / 4, t = lane % 4) follows the mma.sync
// m16n8k16 fragment layout. Logical k index 2t+8e+{0,1} of key k-step ks maps to
// the code pair of slot s = 2 ks + e in thread t's 32-channel span of the row:
// channels 32t + m*2*NSLOT + i and + NSLOT, with m = s / NSLOT, i = s % NSLOT.
template <int BITS, int DT, int GQ>
__global__ void __launch_bounds__(kThreads, BITS == 2 ? 3 : 2) decode_mma_kernel(DecodeArgs a) {
    static_assert(GQ == 1 || GQ == 2 || GQ == 4, "one n8 tile holds hi and lo of up to four heads");
    using Lay = MmaLayout<BITS>;
    constexpr int RB = Lay::kRowBytes;
    constexpr int STAGE = Lay::kStage;
    constexpr int NSLOT = Lay::kNslot;
    constexpr int SHIFT = CodeShift<BITS>::kValue;

    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* stages = smem;                                               // [warp][stage][STAGE]
    float* qs = reinterpret_cast<float*>(smem + Lay::kStageBytes);             // [GQ][kD]
    float* pt_all = qs + GQ * kD;                                               // [warp][4][kPtLd]
    float* red_m = pt_all + kWarps * 4 * kPtLd;                                 // [warp][GQ]
    float* red_l = red_m + kWarps * GQ;                                         // [warp][GQ]
    int* s_misc = reinterpret_cast<int*>(red_l + kWarps * GQ);                 // [8]
    float* red_acc = reinterpret_cast<float*>(smem);                           // [warp][GQ][kD], after the loop

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
    const int64_t np = n_packed(L, a.R);
    const int nsp = static_cast<int>((np + a.chunk - 1) / a.chunk);   // packed splits
    const int nsplit = nsp + 1;                                         // + the residual split
    if (split >= nsplit) return;

    const uint16_t* q = static_cast<const uint16_t*>(a.q) + (static_cast<int64_t>(b) * Hq + h * GQ) * kD;
    for (int i = tid; i < GQ * kD; i += kThreads) qs[i] = widen<DT>(q[i]) * a.scale_log2;
    __syncthreads();

    if (split == nsp) {
        // ---------------- residual split: tokens [np, L), lane-layout CUDA-core path
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
        for (int64_t ts = np + 32 * warp; ts < L; ts += 32 * kWarps) {
            residual_tile<DT, GQ>(kres, vres, ring, ts, L, qs, lane, m, l, acc);
            __syncwarp();
        }
        store_lane_state<GQ>(warp, lane, m, l, acc, red_m, red_l, red_acc);
        __syncthreads();
        finish_split<GQ>(a, b, h, split, nsplit, out_bh, red_m, red_l, red_acc, &s_misc[0]);
        return;
    }

    // ---------------- packed split: key groups [g0, g1)
    const int gid = lane >> 2, t = lane & 3;
    const int hh = gid >> 1, part = gid & 1;     // B column gid = (head hh, hi/lo part)
    const bool hv = GQ >= 4 || hh < GQ;   // this thread's B column belongs to a real head

    // q prescale: a power of two putting max |q| in (1/2, 1]
    float qmax_abs = 0.0f;
    for (int i = tid; i < GQ * kD; i += kThreads) qmax_abs = fmaxf(qmax_abs, fabsf(qs[i]));
    qmax_abs = warp_max(qmax_abs);
    if (lane == 0) reinterpret_cast<float*>(s_misc)[1 + warp] = qmax_abs;
    __syncthreads();
    qmax_abs = fmaxf(fmaxf(reinterpret_cast<float*>(s_misc)[1], reinterpret_cast<float*>(s_misc)[2]),
                     fmaxf(reinterpret_cast<float*>(s_misc)[3], reinterpret_cast<float*>(s_misc)[4]));
    int qexp = 0;
    if (qmax_abs > 0.0f) frexpf(qmax_abs, &qexp);
    const float qpre = ldexpf(1.0f, -qexp), qpost = ldexpf(1.0f, qexp);

    // per-thread constants of the key-side B operand (column gid, thread t's span)
    uint32_t cY[16], cX[16], cZ[16], cB[16];
#pragma unroll
    for (int s = 0; s < 16; ++s) {
        const int c0 = 32 * t + (s / NSLOT) * 2 * NSLOT + (s % NSLOT), c1 = c0 + NSLOT;
        const float v0 = hv ? qs[(hv ? hh : 0) * kD + c0] * qpre : 0.0f;
        const float v1 = hv ? qs[(hv ? hh : 0) * kD + c1] * qpre : 0.0f;
        const uint32_t qh = pack_h2(v0, v1);
        const uint32_t ql = pack_h2(v0 - h2_lo(qh), v1 - h2_hi(qh));
        cY[s] = qh;
        cX[s] = part ? ql : 0u;
        cZ[s] = part ? (qh ^ 0x80008000u) : 0u;
        cB[s] = part ? ql : qh;
    }
    // value side: byte / half-word selectors of this thread's four channels per channel group
    const uint32_t g3 = static_cast<uint32_t>(gid & 3);
    const uint32_t sel_v = BITS == 2 ? (g3 | (g3 << 4) | ((4 + g3) << 8) | ((4 + g3) << 12))
                                     : ((gid & 1) ? 0x7632u : 0x5410u);
    const int vbyte = BITS == 2 ? 4 * (gid >> 2) : 4 * (gid >> 1);   // byte offset of the word in a group's block
    const uint32_t sel_z = (gid & 1) ? 0x7632u : 0x5410u;

    float m_run = -CUDART_INF_F, l_run = 0.0f;
    float cv[8][4], cz[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) cv[i][0] = cv[i][1] = cv[i][2] = cv[i][3] = 0.0f;
    cz[0] = cz[1] = cz[2] = cz[3] = 0.0f;

    const int64_t g0 = static_cast<int64_t>(split) * a.chunk / kGroup;
    const int64_t g1 = min(static_cast<int64_t>(split + 1) * a.chunk, np) / kGroup;
    const int64_t gfirst = g0 + warp;
    const int n_my = gfirst < g1 ? static_cast<int>((g1 - gfirst + kWarps - 1) / kWarps) : 0;
    unsigned char* my_st = stages + warp * kStages * STAGE;
    float* pt = pt_all + warp * 4 * kPtLd;

    const unsigned char* kc_base = sq.k_codes + static_cast<int64_t>(h) * cap * RB;
    const unsigned char* vc_base = sq.v_codes + static_cast<int64_t>(h) * cap * RB;
    const unsigned char* ks_base = reinterpret_cast<const unsigned char*>(sq.k_scale + static_cast<int64_t>(h) * (cap / kGroup) * kD);
    const unsigned char* kz_base = reinterpret_cast<const unsigned char*>(sq.k_zero + static_cast<int64_t>(h) * (cap / kGroup) * kD);
    const unsigned char* vs_base = reinterpret_cast<const unsigned char*>(sq.v_scale + static_cast<int64_t>(h) * cap * (kD / kGroup));
    const unsigned char* vz_base = reinterpret_cast<const unsigned char*>(sq.v_zero + static_cast<int64_t>(h) * cap * (kD / kGroup));

    // Per-lane cp.async plan of one group: code rows as 16-byte chunks (lane + 32k), then one
    // chunk of key scale / zero (lanes 0-15 / 16-31) and one of value scale / zero.
    constexpr int kCodeChunks = 2 * RB / 32;                // per lane, per code block
    const int half = lane >> 4, off16 = (lane & 15) * 16;
    const unsigned char* kc_lane = kc_base + lane * 16;
    const unsigned char* vc_lane = vc_base + lane * 16;
    const unsigned char* km_lane = (half ? kz_base : ks_base) + off16;
    const unsigned char* vm_lane = (half ? vz_base : vs_base) + off16;
    const int km_dst = 2 * kGroup * RB + half * Lay::kMetaPad + (off16 >> 6) * 80 + (off16 & 63);
    const int vm_dst = 2 * kGroup * RB + 2 * Lay::kMetaPad + half * 256 + off16;
    auto issue = [&](int slot, int64_t j) {
        unsigned char* dst = my_st + slot * STAGE;
        const int64_t code_off = j * kGroup * RB, meta_off = j * 256;
#pragma unroll
        for (int k = 0; k < kCodeChunks; ++k) {
            cp_async16(dst + lane * 16 + 512 * k, kc_lane + code_off + 512 * k);
            cp_async16(dst + kGroup * RB + lane * 16 + 512 * k, vc_lane + code_off + 512 * k);
        }
        cp_async16(dst + km_dst, km_lane + meta_off);
        cp_async16(dst + vm_dst, vm_lane + meta_off);
    };

#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) {
        if (i < n_my) issue(i, gfirst + static_cast<int64_t>(kWarps) * i);
        cp_async_commit();
    }

    for (int it = 0; it < n_my; ++it) {
        {
            const int nxt = it + kStages - 1;
            if (nxt < n_my) issue(nxt % kStages, gfirst + static_cast<int64_t>(kWarps) * nxt);
            cp_async_commit();
        }
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const unsigned char* st = my_st + (it % kStages) * STAGE;
        const unsigned char* kc = st;
        const unsigned char* vc = st + kGroup * RB;
        const unsigned char* ksm = st + 2 * kGroup * RB;
        const unsigned char* kzm = ksm + Lay::kMetaPad;
        const unsigned char* vsm = kzm + Lay::kMetaPad;    // [32 tokens][4] fp16
        const unsigned char* vzm = vsm + 256;

        // ---- key scale / zero pairs of this thread's span
        uint32_t sp[16], zp[16];
        {
            uint32_t R[16], Z[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 r4 = *reinterpret_cast<const uint4*>(ksm + 80 * t + 16 * i);
                const uint4 z4 = *reinterpret_cast<const uint4*>(kzm + 80 * t + 16 * i);
                R[4 * i] = r4.x; R[4 * i + 1] = r4.y; R[4 * i + 2] = r4.z; R[4 * i + 3] = r4.w;
                Z[4 * i] = z4.x; Z[4 * i + 1] = z4.y; Z[4 * i + 2] = z4.z; Z[4 * i + 3] = z4.w;
            }
#pragma unroll
            for (int s = 0; s < 16; ++s) {
                const int rel = (s / NSLOT) * 2 * NSLOT + (s % NSLOT);
                const uint32_t sel = (rel & 1) ? 0x7632u : 0x5410u;
                sp[s] = prmt(R[rel >> 1], R[(rel + NSLOT) >> 1], sel);
                zp[s] = prmt(Z[rel >> 1], Z[(rel + NSLOT) >> 1], sel);
            }
        }

        // ---- bias: every row of A is z_k, B = q (hi / lo column)
        // two accumulators (even / odd k-steps) halve the dependent MMA chain
        float cb[4] = {0.0f, 0.0f, 0.0f, 0.0f}, cb2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int ks = 0; ks < 8; ks += 2) {
            mma_f16(cb, zp[2 * ks], zp[2 * ks], zp[2 * ks + 1], zp[2 * ks + 1], cB[2 * ks], cB[2 * ks + 1]);
            mma_f16(cb2, zp[2 * ks + 2], zp[2 * ks + 2], zp[2 * ks + 3], zp[2 * ks + 3], cB[2 * ks + 2], cB[2 * ks + 3]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) cb[i] += cb2[i];

        // ---- scores: A = key codes (tokens gid + 8r), B = (q * s_k) hi / lo
        float c0[4] = {cb[0], cb[1], cb[2], cb[3]}, c1[4] = {cb[0], cb[1], cb[2], cb[3]};
        float c0o[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c1o[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // odd k-steps
        {
            uint32_t cw[4][BITS], cws[4][BITS];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const unsigned char* row = kc + (gid + 8 * r) * RB;
                if constexpr (BITS == 2) {
                    const uint2 v = *reinterpret_cast<const uint2*>(row + 8 * t);
                    cw[r][0] = v.x; cw[r][1] = v.y;
                } else {
                    const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * t);
                    cw[r][0] = v.x; cw[r][1] = v.y; cw[r][2] = v.z; cw[r][3] = v.w;
                }
#pragma unroll
                for (int w = 0; w < BITS; ++w) cws[r][w] = cw[r][w] >> SHIFT;
            }
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int s0 = 2 * ks, s1 = 2 * ks + 1;
                const uint32_t b0 = hfma2(cX[s0], sp[s0], hfma2(cY[s0], sp[s0], hmul2(cZ[s0], sp[s0])));
                const uint32_t b1 = hfma2(cX[s1], sp[s1], hfma2(cY[s1], sp[s1], hmul2(cZ[s1], sp[s1])));
                const int w0 = s0 / NSLOT, w1 = s1 / NSLOT;
                uint32_t a0, a1, a2, a3;
a0 = code_slot<BITS>(cw[0][w0], cws[0][w0], s0);
                a1 = code_slot<BITS>(cw[1][w0], cws[1][w0], s0);
                a2 = code_slot<BITS>(cw[0][w1], cws[0][w1], s1);
                a3 = code_slot<BITS>(cw[1][w1], cws[1][w1], s1);
                if (ks & 1) mma_f16(c0o, a0, a1, a2, a3, b0, b1); else mma_f16(c0, a0, a1, a2, a3, b0, b1);
                a0 = code_slot<BITS>(cw[2][w0], cws[2][w0], s0);
                a1 = code_slot<BITS>(cw[3][w0], cws[3][w0], s0);
                a2 = code_slot<BITS>(cw[2][w1], cws[2][w1], s1);
                a3 = code_slot<BITS>(cw[3][w1], cws[3][w1], s1);
                if (ks & 1) mma_f16(c1o, a0, a1, a2, a3, b0, b1); else mma_f16(c1, a0, a1, a2, a3, b0, b1);
            }
        }

        // ---- online softmax for head t over tokens gid, gid+8, gid+16, gid+24
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            c0[i] += c0o[i];
            c1[i] += c1o[i];
        }
        float S[4] = {(c0[0] + c0[1]) * qpost, (c0[2] + c0[3]) * qpost, (c1[0] + c1[1]) * qpost,
                      (c1[2] + c1[3]) * qpost};
        float tmax = fmaxf(fmaxf(S[0], S[1]), fmaxf(S[2], S[3]));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 4));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
        tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
        const float mnew = fmaxf(m_run, tmax);
        if (__any_sync(kFull, mnew > m_run)) {
            const float alpha = exp2f(m_run - mnew);
            l_run *= alpha;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                cv[i][0] *= alpha; cv[i][1] *= alpha; cv[i][2] *= alpha; cv[i][3] *= alpha;
            }
            cz[0] *= alpha; cz[1] *= alpha; cz[2] *= alpha; cz[3] *= alpha;
            m_run = mnew;
        }
        float p[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) p[r] = (GQ >= 4 || t < GQ) ? exp2f(S[r] - m_run) : 0.0f;
        l_run += (p[0] + p[1]) + (p[2] + p[3]);
#pragma unroll
        // token 8r + j goes to column 8r + 2 (j % 4) + j / 4: the value side pairs tokens
        // (8r + t', 8r + t' + 4), which then sit side by side
        for (int r = 0; r < 4; ++r) pt[t * kPtLd + 8 * r + 2 * (gid & 3) + (gid >> 2)] = p[r];
        __syncwarp();

        // ---- value side B operands: P' = p * s_v (hi / lo), and p (hi / lo) for the z_v term
        uint32_t vb[2][2][4], bp[2][2], za[2][2];
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tau0 = 16 * k2 + 8 * e + t;      // pair (tau0, tau0 + 4)
                const float2 pp = hv ? *reinterpret_cast<const float2*>(pt + (hv ? hh : 0) * kPtLd + 16 * k2 + 8 * e + 2 * t)
                                     : make_float2(0.0f, 0.0f);
                const uint32_t ph = pack_h2(pp.x, pp.y);
                const uint32_t pl = pack_h2(pp.x - h2_lo(ph), pp.y - h2_hi(ph));
                const uint32_t xp = part ? pl : 0u, zn = part ? (ph ^ 0x80008000u) : 0u;
                bp[k2][e] = part ? pl : ph;
                const uint2 s0w = *reinterpret_cast<const uint2*>(vsm + tau0 * 8);
                const uint2 s1w = *reinterpret_cast<const uint2*>(vsm + (tau0 + 4) * 8);
#pragma unroll
                for (int kg = 0; kg < 4; ++kg) {
                    const uint32_t a_w = kg < 2 ? s0w.x : s0w.y, b_w = kg < 2 ? s1w.x : s1w.y;
                    const uint32_t svp = prmt(a_w, b_w, (kg & 1) ? 0x7632u : 0x5410u);
                    vb[k2][e][kg] = hfma2(xp, svp, hfma2(ph, svp, hmul2(zn, svp)));
                }
                const uint32_t zw0 = *reinterpret_cast<const uint32_t*>(vzm + tau0 * 8 + 4 * ((gid & 3) >> 1));
                const uint32_t zw1 = *reinterpret_cast<const uint32_t*>(vzm + (tau0 + 4) * 8 + 4 * ((gid & 3) >> 1));
                za[k2][e] = gid < 4 ? prmt(zw0, zw1, sel_z) : 0u;
            }
        }
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) mma_f16(cz, za[k2][0], 0u, za[k2][1], 0u, bp[k2][0], bp[k2][1]);

        // ---- value codes (A = codes^T, rows = channels of one channel group) and P' V
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
#pragma unroll
            for (int kg = 0; kg < 4; ++kg) {
                uint32_t wv[2], wvs[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tau0 = 16 * k2 + 8 * e + t;
                    const int off = kg * (RB / 4) + vbyte;
                    const uint32_t x0 = *reinterpret_cast<const uint32_t*>(vc + tau0 * RB + off);
                    const uint32_t x1 = *reinterpret_cast<const uint32_t*>(vc + (tau0 + 4) * RB + off);
                    wv[e] = prmt(x0, x1, sel_v);
                    wvs[e] = wv[e] >> SHIFT;
                }
                // m-tile 2kg + u: rows gid (slot 2u) and gid + 8 (slot 2u + 1)
                mma_f16(cv[2 * kg], code_pair<BITS, 0>(wv[0], wvs[0]), code_pair<BITS, 1>(wv[0], wvs[0]),
                        code_pair<BITS, 0>(wv[1], wvs[1]), code_pair<BITS, 1>(wv[1], wvs[1]), vb[k2][0][kg],
                        vb[k2][1][kg]);
                mma_f16(cv[2 * kg + 1], code_pair<BITS, 2>(wv[0], wvs[0]), code_pair<BITS, 3>(wv[0], wvs[0]),
                        code_pair<BITS, 2>(wv[1], wvs[1]), code_pair<BITS, 3>(wv[1], wvs[1]), vb[k2][0][kg],
                        vb[k2][1][kg]);
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();

    // ---- warp state -> merge arrays (red_acc aliases the stages: wait for every warp)
    float l_tot = l_run;
    l_tot += __shfl_xor_sync(kFull, l_tot, 4);
    l_tot += __shfl_xor_sync(kFull, l_tot, 8);
    l_tot += __shfl_xor_sync(kFull, l_tot, 16);
    float zk[4];
    const float zmine = cz[0] + cz[1];     // (channel group gid, head t) for gid < 4
#pragma unroll
    for (int kg = 0; kg < 4; ++kg) zk[kg] = __shfl_sync(kFull, zmine, 4 * kg + t);
    __syncthreads();
    if (GQ >= 4 || t < GQ) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int kg = mt >> 1;
            const int ch = 32 * kg + 4 * gid + 2 * (mt & 1);
            red_acc[(warp * GQ + t) * kD + ch] = cv[mt][0] + cv[mt][1] + zk[kg];
            red_acc[(warp * GQ + t) * kD + ch + 1] = cv[mt][2] + cv[mt][3] + zk[kg];
        }
        if (gid == 0) {
            red_m[warp * GQ + t] = m_run;
            red_l[warp * GQ + t] = l_tot;
        }
    }
    __syncthreads();
    finish_split<GQ>(a, b, h, split, nsplit, out_bh, red_m, red_l, red_acc, &s_misc[0]);
}

template <int BITS, int DT, int GQ>
cudaError_t launch_mma(const DecodeArgs& a, dim3 grid, cudaStream_t stream) {
    constexpr int smem = MmaLayout<BITS>::kSmemBytes(GQ);
    const cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<BITS, DT, GQ>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    decode_mma_kernel<BITS, DT, GQ><<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int BITS, int DT>
cudaError_t launch_gq(const DecodeArgs& a, dim3 grid, cudaStream_t stream) {
    switch (a.Hq / a.H) {
        case 1: return launch_mma<BITS, DT, 1>(a, grid, stream);
        case 2: return launch_mma<BITS, DT, 2>(a, grid, stream);
        case 4: return launch_mma<BITS, DT, 4>(a, grid, stream);
        case 8: decode_split_kernel<BITS, DT, 8><<<grid, kThreads, 0, stream>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace

void decode_plan(int nseq, int H, int Hq, int D, int max_kv_len, int* chunk, int* max_splits,
                 size_t* counter_bytes, size_t* partial_bytes) {
    // Split size: about an eighth of the longest sequence, in whole 256-token
    // steps, between 2048 and 4096 tokens; one more split for the residual tokens.
    // Below 2048 tokens (16 groups per warp) the per-CTA setup and merge dominate;
    // measured on the workloads, 2048..4096 is within 1 % of the best fixed size.
    const int64_t eighth = (static_cast<int64_t>(max_kv_len) + 7) / 8;
    int64_t c = ((eighth + 255) / 256) * 256;
    c = c < 2048 ? 2048 : (c > 4096 ? 4096 : c);
    const int64_t ms = (max_kv_len <= 0 ? 1 : (max_kv_len + c - 1) / c) + 1;
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
