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
// Design. One warp quantizes one G-token group tile (or, for values, up to 32
// tokens) over a slice of up to 128 channels, entirely in registers: no shared
// memory and no block barriers. G is 32 or 64 (a template parameter). For keys a
// lane owns four channels and loads them from every token row (each load
// instruction reads whole rows, coalesced); for values a lane owns one token row.
// Minimum and maximum run on packed pairs (min/max.f16x2 or .bf16x2). The codes
// come from a fused multiply-add with a rounding constant (twice, with 1/s
// bracketed, to mark the rare elements whose code the exact division must decide)
// and reach their bit position through the accumulating add. These kernels stream
// 16 bits in and 2.5 (2-bit) bits out per element and are meant to run at the HBM
// bound.
#include "kivi_internal.cuh"

namespace kivi {
namespace {

constexpr int kThreads = 256;   // 8 warps per CTA, one tile slice per warp
constexpr int kWarps = kThreads / 32;

// Channels one warp covers of a D-channel tile. Values: 64 where that divides D, else 32
// (a 64-channel slice holds 32 registers of elements per lane, so that three CTAs of
// eight warps fit on an SM; D is a multiple of G, so G = 64 always gets 64). Keys, G =
// 32: 128 where that divides D (then a lane owns four channels over all 32 tokens and no
// lane repeats another's per-channel scale and zero; two CTAs per SM; measured 6 % faster
// on the flush), else as values; G = 64: 64 (four channels of 32 of the 64 tokens per
// lane, the same 64 registers).
__host__ __device__ constexpr int slice_width(int D) { return D % 64 == 0 ? 64 : 32; }
__host__ __device__ constexpr int key_slice_width(int D, int G) {
    return G == 64 ? 64 : (D % 128 == 0 ? 128 : slice_width(D));
}
// Registers of elements per lane: DS * TOK / 64 for a DS-channel, TOK-token tile. Tiles
// of 64 registers run two CTAs of eight warps per SM, smaller ones three; so do 4-bit
// bf16 value tiles, whose fully unrolled 64 codes per lane do not fit 80 registers.
template <int DS, int TOK, int BITS = 2, int DT = KIVI_F16>
struct CtasPerSm {
    static constexpr int kValue = DS * TOK / 64 >= 64 || (BITS == 4 && DT == KIVI_BF16 && DS >= 64) ? 2 : 3;
};

template <int DT>
__device__ __forceinline__ uint32_t hmin2(uint32_t a, uint32_t b) {
    uint32_t r;
    if constexpr (DT == KIVI_F16) asm("min.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    else asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
template <int DT>
__device__ __forceinline__ uint32_t hmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    if constexpr (DT == KIVI_F16) asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    else asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t lo16(uint32_t w) { return w & 0xffffu; }
__device__ __forceinline__ uint32_t hi16(uint32_t w) { return w >> 16; }
__device__ __forceinline__ bool is_zero16(uint32_t h) { return (h & 0x7fffu) == 0; }

// Smaller / larger of two 16-bit floats of the same group (either one when equal).
template <int DT>
__device__ __forceinline__ uint32_t pick_min(uint32_t a, uint32_t b) {
    return widen<DT>(static_cast<uint16_t>(b)) < widen<DT>(static_cast<uint16_t>(a)) ? b : a;
}
template <int DT>
__device__ __forceinline__ uint32_t pick_max(uint32_t a, uint32_t b) {
    return widen<DT>(static_cast<uint16_t>(b)) > widen<DT>(static_cast<uint16_t>(a)) ? b : a;
}

// The fp32 quantizer of one group: zero z, scale s, and r_lo, r_hi: r = 1/s (correctly
// rounded; 0 when s is 0 or inf) moved down and up by 2^-21 of itself.
struct Quantizer {
    float z, s, r_lo, r_hi;
};

__device__ __forceinline__ Quantizer make_quantizer(const GroupParams& gp) {
    Quantizer q;
    q.z = gp.z;
    q.s = gp.s;
    const float r = gp.s != 0.0f ? __frcp_rn(gp.s) : 0.0f;
    q.r_lo = __fmul_rn(r, 1.0f - 0x1p-21f);
    q.r_hi = __fmul_rn(r, 1.0f + 0x1p-21f);
    return q;
}

// Adding 1.5 * 2^23 to an fp32 value t with |t| < 2^22 rounds it to the integer
// rint(t) (half to even) in the low mantissa bits.
constexpr float kMagic = 12582912.0f;
constexpr uint32_t kMagicBits = 0x4B400000u;
// What n encodings of kMagic + code, shifted to bit offsets 0, B, 2B, ..., sum to
// beyond the codes themselves; subtracted up front, so the sum is the packed codes.
__host__ __device__ constexpr uint32_t magic_offset(int n, int bits) {
    uint32_t o = 0;
    for (int e = 0; e < n; ++e) o += kMagicBits << (e * bits);
    return 0u - o;
}

// The code of encode() as kMagic + code (an fp32 bit pattern), with the IEEE division
// replaced by products with a bracket of 1/s, and a mark where that may give a
// different code. fma(d, r_x, kMagic) is kMagic + rint(d r_x) for the exact product
// d r_x. The correctly rounded quotient t = d / s lies within 2^-22 |t| of d / s's
// exact value and of d r (r is 1/s correctly rounded), so inside [d r_lo, d r_hi] (the
// bracket is 2^-21 wide on each side, less at most 2^-24 from rounding r_lo and r_hi).
// rint is monotone, so when the two ends round to the same integer, so does t. When
// they differ (a half-integer lies in the bracket) the bits of the two results differ
// and are OR-ed into `mark`: the caller recomputes with the exact division. There is no
// clamp: the caller checks with codes_in_range() that every element of the group lands
// in [0, qmax] and otherwise recomputes the group exactly. r == 0 (s == 0 or s = inf)
// gives code 0, as the division does.
template <int BITS>
__device__ __forceinline__ uint32_t code_bits(float x, const Quantizer& q, uint32_t& mark) {
    const float d = __fsub_rn(x, q.z);
    const uint32_t y_lo = __float_as_uint(__fmaf_rn(d, q.r_lo, kMagic));
    const uint32_t y_hi = __float_as_uint(__fmaf_rn(d, q.r_hi, kMagic));
    mark |= y_lo ^ y_hi;
    return y_hi;
}

// Whether code_bits() gives codes in [0, qmax] for every element of a group with this
// minimum and maximum: x -> fma(x - z, r_hi, kMagic) is monotone (r_hi >= 0), so
// checking the two ends suffices. False only where the fp16 rounding of z or s pushes an
// end more than half a step out (for instance inputs below the fp16 normal range).
template <int BITS>
__device__ __forceinline__ bool codes_in_range(float mn, float mx, const Quantizer& q) {
    constexpr float qmax = static_cast<float>((1 << BITS) - 1);
    const float ylo = __fmaf_rn(__fsub_rn(mn, q.z), q.r_hi, kMagic);
    const float yhi = __fmaf_rn(__fsub_rn(mx, q.z), q.r_hi, kMagic);
    return ylo >= kMagic && yhi <= kMagic + qmax;
}

template <int DT>
__device__ __forceinline__ float half_at(uint32_t w, int hi) {
    return widen<DT>(static_cast<uint16_t>(hi ? w >> 16 : w & 0xffffu));
}

__device__ __forceinline__ uint2 ld_nc_u2(const uint16_t* p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_nc_u4(const uint16_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Rare paths, kept out of line so that the unrolled main loops stay small in the
// instruction cache; they re-read their inputs from global memory.

// Codes of four consecutive key channels at p (one per channel quantizer), with the
// IEEE division: the product path found one of them near a rounding tie.
template <int BITS, int DT>
__device__ __noinline__ uint32_t keys_exact4(const uint16_t* p, float z0, float z1, float z2, float z3, float s0,
                                             float s1, float s2, float s3) {
    constexpr int qmax = (1 << BITS) - 1;
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    return encode(half_at<DT>(v.x, 0), z0, s0, qmax) | encode(half_at<DT>(v.x, 1), z1, s1, qmax) << BITS |
           encode(half_at<DT>(v.y, 0), z2, s2, qmax) << (2 * BITS) | encode(half_at<DT>(v.y, 1), z3, s3, qmax) << (3 * BITS);
}

// One lane's share of a TOK-row x DS-channel tile of 16-bit elements, in registers.
// Keys (TOK = G): lane l owns channels 4 (l mod DS/4) .. +3 of the slice and the tokens
// j, j + TS, ... (j = l / (DS/4), TS = 128 / DS): w[2 i], w[2 i + 1] hold token i TS + j.
// Values (TOK = 32): lane l owns token l, w[c] holding channels 2 c and 2 c + 1.
template <int DS, int TOK>
struct Tile {
    uint32_t w[DS * TOK / 64];
};

// Loads a key tile. row(t) is token t's row at the slice's first channel; where
// `contiguous` is set (the same on every lane) the rows are known to be row(0) + t * D.
template <int DS, int G, typename RowFn>
__device__ __forceinline__ void keys_load(RowFn row, bool contiguous, int D, Tile<DS, G>& x) {
    constexpr int LPR = DS / 4, TS = 32 / LPR, NT = G / TS;
    const int lane = threadIdx.x & 31, cq = lane % LPR, j = lane / LPR;
    if (contiguous) {
        const uint16_t* p = row(j) + 4 * cq;
        const int64_t step = static_cast<int64_t>(TS) * D;
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const uint2 v = ld_nc_u2(p + i * step);
            x.w[2 * i] = v.x;
            x.w[2 * i + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const uint2 v = ld_nc_u2(row(i * TS + j) + 4 * cq);
            x.w[2 * i] = v.x;
            x.w[2 * i + 1] = v.y;
        }
    }
}

// Keys of one G-token group over one DS-channel slice, by one warp, from a tile that
// keys_load() filled; row() as there (used again only on the rare exact paths). codes,
// scale and zero point at the slice's first channel of token 0's code row and of the
// group's scale and zero rows. The minimum and maximum come from packed min/max over
// token pairs and a shuffle across token subsets; where one is a zero, the rule "the
// first value seen wins" is applied by finding the sign of the first zero in token order.
template <int BITS, int DT, int DS, int G, typename RowFn>
__device__ __forceinline__ void keys_compute(const Tile<DS, G>& x, RowFn row, uint8_t* codes, int code_ld,
                                             uint16_t* scale, uint16_t* zero) {
    constexpr int LPR = DS / 4, TS = 32 / LPR, NT = G / TS;
    static_assert(NT <= 32, "rows to redo are kept in one 32-bit mask");
    const int lane = threadIdx.x & 31, cq = lane % LPR, j = lane / LPR;
    uint32_t mn0 = x.w[0], mx0 = x.w[0], mn1 = x.w[1], mx1 = x.w[1];
#pragma unroll
    for (int i = 1; i < NT; ++i) {
        mn0 = hmin2<DT>(mn0, x.w[2 * i]);
        mx0 = hmax2<DT>(mx0, x.w[2 * i]);
        mn1 = hmin2<DT>(mn1, x.w[2 * i + 1]);
        mx1 = hmax2<DT>(mx1, x.w[2 * i + 1]);
    }
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1) {
        mn0 = hmin2<DT>(mn0, __shfl_xor_sync(0xffffffffu, mn0, o));
        mx0 = hmax2<DT>(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mn1 = hmin2<DT>(mn1, __shfl_xor_sync(0xffffffffu, mn1, o));
        mx1 = hmax2<DT>(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    uint32_t mn[4] = {lo16(mn0), hi16(mn0), lo16(mn1), hi16(mn1)};
    uint32_t mx[4] = {lo16(mx0), hi16(mx0), lo16(mx1), hi16(mx1)};
    bool fix = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) fix |= is_zero16(mn[e]) || is_zero16(mx[e]);
    if (__any_sync(0xffffffffu, fix)) {
        // 2 t + sign of this lane's first zero, per channel
        uint32_t first[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
#pragma unroll 1
        for (int i = NT - 1; i >= 0; --i) {
            const uint2 v = *reinterpret_cast<const uint2*>(row(i * TS + j) + 4 * cq);
            const uint32_t hv[4] = {lo16(v.x), hi16(v.x), lo16(v.y), hi16(v.y)};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (is_zero16(hv[e])) first[e] = 2u * (i * TS + j) + (hv[e] >> 15);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
#pragma unroll
            for (int o = LPR; o < 32; o <<= 1) first[e] = min(first[e], __shfl_xor_sync(0xffffffffu, first[e], o));
            const uint32_t zs = (first[e] & 1u) ? 0x8000u : 0u;
            if (is_zero16(mn[e])) mn[e] = zs;
            if (is_zero16(mx[e])) mx[e] = zs;
        }
    }
    constexpr int qmax = (1 << BITS) - 1;
    Quantizer qz[4];
    uint32_t s16[4], z16[4];
    bool in_range = true;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float fmn = widen<DT>(static_cast<uint16_t>(mn[e])), fmx = widen<DT>(static_cast<uint16_t>(mx[e]));
        const GroupParams gp = group_params(fmn, fmx, qmax);
        s16[e] = gp.s16;
        z16[e] = gp.z16;
        qz[e] = make_quantizer(gp);
        in_range &= codes_in_range<BITS>(fmn, fmx, qz[e]);
    }
    if (j == 0) {
        *reinterpret_cast<uint2*>(scale + 4 * cq) = make_uint2(s16[0] | (s16[1] << 16), s16[2] | (s16[3] << 16));
        *reinterpret_cast<uint2*>(zero + 4 * cq) = make_uint2(z16[0] | (z16[1] << 16), z16[2] | (z16[3] << 16));
    }
    uint32_t tie_rows = in_range ? 0u : 0xffffffffu >> (32 - NT);   // rows to redo with the exact division
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        uint32_t mark = 0u;
        uint32_t acc = magic_offset(4, BITS);
        acc += code_bits<BITS>(half_at<DT>(x.w[2 * i], 0), qz[0], mark);
        acc += code_bits<BITS>(half_at<DT>(x.w[2 * i], 1), qz[1], mark) << BITS;
        acc += code_bits<BITS>(half_at<DT>(x.w[2 * i + 1], 0), qz[2], mark) << (2 * BITS);
        acc += code_bits<BITS>(half_at<DT>(x.w[2 * i + 1], 1), qz[3], mark) << (3 * BITS);
        tie_rows |= static_cast<uint32_t>(mark != 0u) << i;
        uint8_t* dst = codes + static_cast<int64_t>(i * TS + j) * code_ld;
        if constexpr (BITS == 2) dst[cq] = static_cast<uint8_t>(acc);
        else reinterpret_cast<uint16_t*>(dst)[cq] = static_cast<uint16_t>(acc);
    }
#pragma unroll 1
    while (tie_rows != 0) {
        const int i = __ffs(tie_rows) - 1;
        tie_rows &= tie_rows - 1;
        const uint32_t acc = keys_exact4<BITS, DT>(row(i * TS + j) + 4 * cq, qz[0].z, qz[1].z, qz[2].z, qz[3].z, qz[0].s,
                                                   qz[1].s, qz[2].s, qz[3].s);
        uint8_t* dst = codes + static_cast<int64_t>(i * TS + j) * code_ld;
        if constexpr (BITS == 2) dst[cq] = static_cast<uint8_t>(acc);
        else reinterpret_cast<uint16_t*>(dst)[cq] = static_cast<uint16_t>(acc);
    }
}

// Loads one lane's value row: src is the token's row at the slice's first channel
// (null: this lane has no token).
template <int DS>
__device__ __forceinline__ void values_load(const uint16_t* src, Tile<DS, 32>& x) {
    if (src == nullptr) return;
#pragma unroll
    for (int c = 0; c < DS / 8; ++c) {
        const uint4 v = ld_nc_u4(src + 8 * c);
        x.w[4 * c] = v.x;
        x.w[4 * c + 1] = v.y;
        x.w[4 * c + 2] = v.z;
        x.w[4 * c + 3] = v.w;
    }
}

// Values of one token over one DS-channel slice (DS / G channel groups), by one lane,
// from the row values_load() read from src (null: no token for this lane); codes, scale
// and zero point at the slice's first code byte and first group of the token's rows.
// Packed min/max over channel pairs, then the pair's two halves; a zero minimum or
// maximum takes the sign of the first zero in channel order. Every lane of the warp
// calls it: the exact redo at the end is done by the warp together.
template <int BITS, int DT, int DS, int G>
__device__ __forceinline__ void values_compute(const Tile<DS, 32>& x, const uint16_t* src, uint8_t* codes,
                                               uint16_t* scale, uint16_t* zero) {
    static_assert(DS % G == 0, "a slice holds whole channel groups");
    constexpr int NKG = DS / G, qmax = (1 << BITS) - 1;
    constexpr int WPG = G * BITS / 32;        // code words per channel group
    constexpr int CPW = 32 / BITS;            // codes per word
    float zq[NKG], sq[NKG];   // fp32 zero and scale per group, for the exact redo
    uint32_t tie_groups = 0;  // groups to redo with the exact division
    if (src != nullptr) {
        uint32_t code_w[NKG][WPG];
        uint32_t s16[NKG], z16[NKG];
#pragma unroll
        for (int k = 0; k < NKG; ++k) {
            const uint32_t* w = x.w + (G / 2) * k;
            uint32_t mn2 = w[0], mx2 = w[0];
#pragma unroll
            for (int c = 1; c < G / 2; ++c) {
                mn2 = hmin2<DT>(mn2, w[c]);
                mx2 = hmax2<DT>(mx2, w[c]);
            }
            uint32_t mn = pick_min<DT>(lo16(mn2), hi16(mn2));
            uint32_t mx = pick_max<DT>(lo16(mx2), hi16(mx2));
            if (is_zero16(mn) || is_zero16(mx)) {   // sign of the first zero in channel order
                uint32_t zs = 0;
#pragma unroll 1
                for (int c = G - 1; c >= 0; --c) {
                    const uint32_t hv = src[k * G + c];
                    zs = is_zero16(hv) ? hv & 0x8000u : zs;
                }
                if (is_zero16(mn)) mn = zs;
                if (is_zero16(mx)) mx = zs;
            }
            const float fmn = widen<DT>(static_cast<uint16_t>(mn)), fmx = widen<DT>(static_cast<uint16_t>(mx));
            const GroupParams gp = group_params(fmn, fmx, qmax);
            s16[k] = gp.s16;
            z16[k] = gp.z16;
            const Quantizer q = make_quantizer(gp);
            zq[k] = q.z;
            sq[k] = q.s;
            uint32_t mark = codes_in_range<BITS>(fmn, fmx, q) ? 0u : 1u;
#pragma unroll
            for (int ww = 0; ww < WPG; ++ww) {
                uint32_t acc = magic_offset(CPW, BITS);
#pragma unroll
                for (int e = 0; e < CPW; ++e) {
                    const int c = ww * CPW + e;
                    acc += code_bits<BITS>(half_at<DT>(w[c >> 1], c & 1), q, mark) << (e * BITS);
                }
                code_w[k][ww] = acc;
            }
            tie_groups |= static_cast<uint32_t>(mark != 0u) << k;
        }
        // code row: NKG * WPG words (8 bytes per 32 channels at 2 bits, 16 at 4 bits)
        uint32_t* cw = reinterpret_cast<uint32_t*>(codes);
        if constexpr (NKG * WPG % 4 == 0) {
#pragma unroll
            for (int i = 0; i < NKG * WPG / 4; ++i)
                reinterpret_cast<uint4*>(cw)[i] = make_uint4(code_w[(4 * i) / WPG][(4 * i) % WPG], code_w[(4 * i + 1) / WPG][(4 * i + 1) % WPG],
                                                             code_w[(4 * i + 2) / WPG][(4 * i + 2) % WPG], code_w[(4 * i + 3) / WPG][(4 * i + 3) % WPG]);
        } else {
            reinterpret_cast<uint2*>(cw)[0] = make_uint2(code_w[0][0], code_w[0][1]);   // NKG * WPG == 2
        }
#pragma unroll
        for (int k = 0; k < NKG; ++k) {
            scale[k] = static_cast<uint16_t>(s16[k]);
            zero[k] = static_cast<uint16_t>(z16[k]);
        }
    }
    // Exact redo, by the whole warp: one flagged (token, group) at a time, each lane
    // encoding G / 32 of its elements with the IEEE division, the words packed by an OR
    // reduction. (A lane redoing its own group alone would run G divisions while the
    // others wait.) Every lane of the warp runs this loop.
    const int lane = threadIdx.x & 31;
    uint32_t pending = tie_groups;
    while (true) {
        const uint32_t ball = __ballot_sync(0xffffffffu, pending != 0);
        if (ball == 0) break;
        const int leader = __ffs(ball) - 1;
        const int k = __ffs(__shfl_sync(0xffffffffu, pending, leader)) - 1;
        float zk = zq[0], sk = sq[0];
#pragma unroll
        for (int i = 1; i < NKG; ++i) {
            zk = k == i ? zq[i] : zk;
            sk = k == i ? sq[i] : sk;
        }
        zk = __shfl_sync(0xffffffffu, zk, leader);
        sk = __shfl_sync(0xffffffffu, sk, leader);
        const uint16_t* gsrc = reinterpret_cast<const uint16_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src), leader)) + k * G;
        uint32_t* gdst = reinterpret_cast<uint32_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(codes), leader)) + k * WPG;
        uint32_t code[G / 32];
#pragma unroll
        for (int e = 0; e < G / 32; ++e) code[e] = encode(widen<DT>(gsrc[32 * e + lane]), zk, sk, qmax);
#pragma unroll
        for (int ww = 0; ww < WPG; ++ww) {
            uint32_t part = 0u;
#pragma unroll
            for (int e = 0; e < G / 32; ++e) {
                const int c = 32 * e + lane;
                part |= c / CPW == ww ? code[e] << ((c % CPW) * BITS) : 0u;
            }
            const uint32_t word = __reduce_or_sync(0xffffffffu, part);
            if (lane == ww) gdst[ww] = word;
        }
        if (lane == leader) pending &= pending - 1;
    }
}

// ---------------------------------------------------------------- standalone codec

// One warp per (stream, G-token group, channel slice).
template <int BITS, int DT, int DS, int G>
__global__ void __launch_bounds__(kThreads, CtasPerSm<DS, G>::kValue) quant_keys_kernel(CodecArgs a) {
    const int D = a.D, nsl = D / DS, groups = a.n_tokens / G;
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (unit >= static_cast<int64_t>(a.n_streams) * groups * nsl) return;
    const int sl = static_cast<int>(unit % nsl);
    const int64_t g = unit / nsl;   // stream * groups + group
    const int64_t tok0 = g * G;
    const uint16_t* x = static_cast<const uint16_t*>(a.x) + tok0 * D + sl * DS;
    const int row_bytes = D * BITS / 8;
    auto row = [&](int t) { return x + static_cast<int64_t>(t) * D; };
    Tile<DS, G> tile;
    keys_load<DS, G>(row, true, D, tile);
    keys_compute<BITS, DT, DS, G>(tile, row, a.codes + tok0 * row_bytes + sl * (DS * BITS / 8), row_bytes,
                               a.scale + g * D + sl * DS, a.zero + g * D + sl * DS);
}

// One warp per (stream, run of 32 tokens, channel slice); lane t takes token t.
template <int BITS, int DT, int DS, int G>
__global__ void __launch_bounds__(kThreads, CtasPerSm<DS, 32, BITS, DT>::kValue) quant_values_kernel(CodecArgs a) {
    const int D = a.D, nsl = D / DS, runs = (a.n_tokens + kTile - 1) / kTile;
    const int64_t unit = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (unit >= static_cast<int64_t>(a.n_streams) * runs * nsl) return;
    const int sl = static_cast<int>(unit % nsl);
    const int64_t sr = unit / nsl;
    const int st = static_cast<int>(sr / runs);
    const int t = static_cast<int>(sr % runs) * kTile + (threadIdx.x & 31);
    const int64_t tok = static_cast<int64_t>(st) * a.n_tokens + t;
    const uint16_t* src = t < a.n_tokens ? static_cast<const uint16_t*>(a.x) + tok * D + sl * DS : nullptr;
    Tile<DS, 32> tile;
    values_load<DS>(src, tile);
    values_compute<BITS, DT, DS, G>(tile, src, a.codes + tok * (D * BITS / 8) + sl * (DS * BITS / 8),
                                    a.scale + tok * (D / G) + sl * (DS / G), a.zero + tok * (D / G) + sl * (DS / G));
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
    s.np0 = n_packed(s.L, a.R, a.G);
    s.np1 = n_packed(s.L1, a.R, a.G);
    s.ok = s.L >= 0 && n >= 0 && n <= a.max_new && s.np1 <= cap;
    return s;
}

// Work units of append_pack_kernel: keys (SIDE 0) take (group that this append makes
// leave the residual window, channel slice), values (SIDE 1) take (32-token run of those
// groups, channel slice), one lane per token. One launch per side, so that each launch
// keeps one code path in the instruction cache (measured: 29 % faster than one launch
// doing both); grid (warp runs, kv head, sequence), each warp taking every
// (gridDim.x * kWarps)-th unit of its (head, sequence). Tokens older than kv_len come
// from the ring, newer ones straight from the caller's buffers.
constexpr int kUnitsPerWarp = 32;

template <int BITS, int DT, int DS, int G, int SIDE>
__global__ void __launch_bounds__(kThreads, CtasPerSm<DS, SIDE == 0 ? G : 32, SIDE == 0 ? 2 : BITS, DT>::kValue)
    append_pack_kernel(AppendArgs a) {
    constexpr int TOK = SIDE == 0 ? G : kTile;   // tokens of one unit
    const int h = blockIdx.y, b = blockIdx.z, D = a.D, nsl = D / DS;
    const kivi_seq& sq = a.seqs[b];
    const int cap = sq.cap_tokens;
    const SeqState st = seq_state(a, b, cap);
    if (!st.ok) {
        if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) {
            const bool len_bad = st.L < 0 || st.L1 < st.L || st.L1 - st.L > a.max_new;
            set_status(a.status, len_bad ? KIVI_ERR_LENGTH : KIVI_ERR_CAPACITY);
        }
        return;
    }
    const int64_t n_units = (st.np1 - st.np0) / TOK * nsl;   // (group or run, slice) of this side
    const int ring = a.R + G;
    const int64_t n = st.L1 - st.L;
    const int row_bytes = D * BITS / 8;
    const int lane = threadIdx.x & 31;
    // unit -> (first token, slice)
    auto slice_of = [&](int64_t unit) { return static_cast<int>(unit % nsl); };
    auto unit_pos = [&](int64_t unit) { return st.np0 + (unit / nsl) * TOK; };
    // row of position p0 + t at the slice's first channel
    auto row_at = [&](const void* res, const void* nw, int64_t p0, int sl, int t) -> const uint16_t* {
        const int64_t p = p0 + t;
        if (p < st.L) {
            int slot = static_cast<int>(p0 % ring) + t;
            slot = slot >= ring ? slot - ring : slot;
            return static_cast<const uint16_t*>(res) + (static_cast<int64_t>(h) * ring + slot) * D + sl * DS;
        }
        return static_cast<const uint16_t*>(nw) + (static_cast<int64_t>(h) * n + (p - st.L)) * D + sl * DS;
    };
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
    int64_t unit = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (unit >= n_units) return;
    for (; unit < n_units; unit += stride) {
        const int sl = slice_of(unit);
        const int64_t p0 = unit_pos(unit), j = p0 / G;
        Tile<DS, TOK> tile;
        if constexpr (SIDE == 0) {
            auto row = [&](int t) { return row_at(sq.k_res, a.k_new[b], p0, sl, t); };
            keys_load<DS, G>(row, p0 >= st.L, D, tile);
            const GroupAddr ga = group_addr(sq, a.H, h, j, group_page(sq, j), D, BITS, BITS, G);
            keys_compute<BITS, DT, DS, G>(tile, row, ga.kc + sl * (DS * BITS / 8), row_bytes, ga.ks + sl * DS,
                                          ga.kz + sl * DS);
        } else {
            const int r = static_cast<int>(p0 - j * G) + lane;   // row within the group
            const uint16_t* src = row_at(sq.v_res, a.v_new[b], p0, sl, lane);
            values_load<DS>(src, tile);
            const GroupAddr ga = group_addr(sq, a.H, h, j, group_page(sq, j), D, BITS, BITS, G);
            values_compute<BITS, DT, DS, G>(tile, src, ga.vc + r * row_bytes + sl * (DS * BITS / 8),
                                            ga.vs + r * (D / G) + sl * (DS / G), ga.vz + r * (D / G) + sl * (DS / G));
        }
    }
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
    const int ring = a.R + a.G;
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

// Appends of at most G tokens per sequence (decode steps, a few draft tokens) in ONE launch
// at head_dim 128: such an append flushes at most one group per (sequence, kv head), so one
// CTA per sequence does all of it. Its warps take the flush units of every kv head (the key
// slices of the group, then the value slices of its 32-token runs) with the same warp
// routines as append_pack_kernel, reading the group from the ring (or from the new tokens);
// after a CTA barrier, every thread writes the new tokens that stay in the window into their
// ring slots, and thread 0 advances kv_len. The barrier orders the flush's ring reads before
// the ring writes of the same sequence.
template <int KB, int VB, int DT, int G>
__global__ void __launch_bounds__(kThreads, 1) append_step_kernel(AppendArgs a) {
    constexpr int D = 128;
    constexpr int DSK = key_slice_width(D, G), DSV = slice_width(D);
    constexpr int KU = D / DSK;                    // key units per (kv head, group)
    constexpr int VU = (G / kTile) * (D / DSV);    // value units per (kv head, group)
    const int b = blockIdx.x, H = a.H;
    const kivi_seq& sq = a.seqs[b];
    const int cap = sq.cap_tokens;
    const SeqState st = seq_state(a, b, cap);
    if (!st.ok) {
        if (threadIdx.x == 0) {
            const bool len_bad = st.L < 0 || st.L1 < st.L || st.L1 - st.L > a.max_new;
            set_status(a.status, len_bad ? KIVI_ERR_LENGTH : KIVI_ERR_CAPACITY);
        }
        return;
    }
    const int ring = a.R + G;
    const int64_t n = st.L1 - st.L;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (st.np1 > st.np0) {                         // exactly one group leaves the window
        const int64_t p0g = st.np0, j = p0g / G;
        const int32_t page = group_page(sq, j);
        auto row_at = [&](const void* res, const void* nw, int h, int64_t p0, int sl, int ds, int t) -> const uint16_t* {
            const int64_t p = p0 + t;
            if (p < st.L) {
                int slot = static_cast<int>(p0 % ring) + t;
                slot = slot >= ring ? slot - ring : slot;
                return static_cast<const uint16_t*>(res) + (static_cast<int64_t>(h) * ring + slot) * D + sl * ds;
            }
            return static_cast<const uint16_t*>(nw) + (static_cast<int64_t>(h) * n + (p - st.L)) * D + sl * ds;
        };
        for (int u = warp; u < H * (KU + VU); u += kWarps) {
            if (u < H * KU) {
                const int h = u / KU, sl = u % KU;
                auto row = [&](int t) { return row_at(sq.k_res, a.k_new[b], h, p0g, sl, DSK, t); };
                Tile<DSK, G> tile;
                keys_load<DSK, G>(row, p0g >= st.L, D, tile);
                const GroupAddr ga = group_addr(sq, H, h, j, page, D, KB, KB, G);
                keys_compute<KB, DT, DSK, G>(tile, row, ga.kc + sl * (DSK * KB / 8), D * KB / 8, ga.ks + sl * DSK,
                                             ga.kz + sl * DSK);
            } else {
                const int v = u - H * KU, h = v / VU, rest = v % VU;
                const int run = rest / (D / DSV), sl = rest % (D / DSV);
                const int64_t p0 = p0g + run * kTile;
                const int r = run * kTile + lane;      // row within the group
                const uint16_t* src = row_at(sq.v_res, a.v_new[b], h, p0, sl, DSV, lane);
                Tile<DSV, kTile> tile;
                values_load<DSV>(src, tile);
                const GroupAddr ga = group_addr(sq, H, h, j, page, D, VB, VB, G);
                values_compute<VB, DT, DSV, G>(tile, src, ga.vc + r * (D * VB / 8) + sl * (DSV * VB / 8),
                                               ga.vs + r * (D / G) + sl * (DSV / G), ga.vz + r * (D / G) + sl * (DSV / G));
            }
        }
    }
    __syncthreads();
    const int64_t first = st.L > st.np1 ? st.L : st.np1;  // first position that stays in the ring
    const int64_t count = st.L1 - first;
    if (count > 0) {
        const uint16_t* knew = static_cast<const uint16_t*>(a.k_new[b]);
        const uint16_t* vnew = static_cast<const uint16_t*>(a.v_new[b]);
        uint16_t* kres = static_cast<uint16_t*>(sq.k_res);
        uint16_t* vres = static_cast<uint16_t*>(sq.v_res);
        constexpr int cpr = D / 8;  // 16-byte chunks per row
        const int64_t total = count * H * cpr;
        for (int64_t c = threadIdx.x; c < total; c += kThreads) {
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

// Calls f.template operator()<BITS, DT, DS, G>() for the runtime bit width, input type,
// slice width ds (32, 64 or 128) and group size g (32 or 64).
template <typename F>
cudaError_t dispatch(int bits, int dtype, int ds, int g, F f) {
#define KIVI_DS(B, T, G)                                                                             \
    return ds == 128 ? f.template operator()<B, T, 128, G>()                                        \
         : ds == 64  ? f.template operator()<B, T, 64, G>() : f.template operator()<B, T, 32, G>();
#define KIVI_G(B, T) \
    if (g == 64) { KIVI_DS(B, T, 64) } \
    KIVI_DS(B, T, 32)
    if (bits == 2 && dtype == KIVI_F16) { KIVI_G(2, KIVI_F16) }
    if (bits == 2) { KIVI_G(2, KIVI_BF16) }
    if (dtype == KIVI_F16) { KIVI_G(4, KIVI_F16) }
    KIVI_G(4, KIVI_BF16)
#undef KIVI_G
#undef KIVI_DS
}

// Slice widths instantiated: keys (G = 32) 32, 64, 128; keys (G = 64) and values 32, 64
// where they hold whole channel groups.
template <int DS, int G>
constexpr bool key_slice_ok() { return G == 32 || DS == 64; }
template <int DS, int G>
constexpr bool value_slice_ok() { return DS != 128 && DS % G == 0; }

int64_t blocks_for(int64_t warps) { return (warps + kWarps - 1) / kWarps; }

}  // namespace

cudaError_t launch_quant_keys(const CodecArgs& a, cudaStream_t stream) {
    if (a.n_streams == 0 || a.n_tokens == 0) return cudaSuccess;
    const int ds = key_slice_width(a.D, a.G);
    const int64_t units = static_cast<int64_t>(a.n_streams) * (a.n_tokens / a.G) * (a.D / ds);
    return dispatch(a.bits, a.dtype, ds, a.G, [&]<int B, int T, int DS, int G>() {
        if constexpr (key_slice_ok<DS, G>()) {
            quant_keys_kernel<B, T, DS, G><<<static_cast<unsigned>(blocks_for(units)), kThreads, 0, stream>>>(a);
        }
        return cudaGetLastError();
    });
}

cudaError_t launch_quant_values(const CodecArgs& a, cudaStream_t stream) {
    if (a.n_streams == 0 || a.n_tokens == 0) return cudaSuccess;
    const int ds = slice_width(a.D);
    const int64_t runs = (a.n_tokens + kTile - 1) / kTile;
    const int64_t units = static_cast<int64_t>(a.n_streams) * runs * (a.D / ds);
    return dispatch(a.bits, a.dtype, ds, a.G, [&]<int B, int T, int DS, int G>() {
        if constexpr (value_slice_ok<DS, G>()) {
            quant_values_kernel<B, T, DS, G><<<static_cast<unsigned>(blocks_for(units)), kThreads, 0, stream>>>(a);
        }
        return cudaGetLastError();
    });
}

// The fused one-launch append for head_dim 128 and at most G new tokens per sequence.
template <int G>
cudaError_t launch_append_step(const AppendArgs& a, cudaStream_t stream) {
    auto go = [&]<int KB, int VB>() {
        if (a.dtype == KIVI_F16) append_step_kernel<KB, VB, KIVI_F16, G><<<a.nseq, kThreads, 0, stream>>>(a);
        else append_step_kernel<KB, VB, KIVI_BF16, G><<<a.nseq, kThreads, 0, stream>>>(a);
        return cudaGetLastError();
    };
    if (a.kb == 2) return a.vb == 2 ? go.template operator()<2, 2>() : go.template operator()<2, 4>();
    return a.vb == 2 ? go.template operator()<4, 2>() : go.template operator()<4, 4>();
}

cudaError_t launch_append_flush(const AppendArgs& a, cudaStream_t stream) {
    if (a.nseq == 0) return cudaSuccess;
    if (a.D == 128 && a.max_new <= a.G)
        return a.G == 64 ? launch_append_step<64>(a, stream) : launch_append_step<32>(a, stream);
    const int max_groups = (a.max_new + a.G - 1) / a.G;
    if (max_groups > 0) {
        // keys and values in two launches, so that each keeps one code path in the
        // instruction cache; one warp per unit, kUnitsPerWarp of them per warp
        auto grid_for = [&](int64_t per_seq_units) {
            return dim3(static_cast<unsigned>(blocks_for((per_seq_units + kUnitsPerWarp - 1) / kUnitsPerWarp)), a.H,
                        a.nseq);
        };
        const int dk = key_slice_width(a.D, a.G), dv = slice_width(a.D);
        cudaError_t e = dispatch(a.kb, a.dtype, dk, a.G, [&]<int B, int T, int DS, int G>() {
            if constexpr (key_slice_ok<DS, G>()) {
                append_pack_kernel<B, T, DS, G, 0><<<grid_for(static_cast<int64_t>(max_groups) * (a.D / DS)), kThreads, 0,
                                                     stream>>>(a);
            }
            return cudaGetLastError();
        });
        if (e != cudaSuccess) return e;
        e = dispatch(a.vb, a.dtype, dv, a.G, [&]<int B, int T, int DS, int G>() {
            if constexpr (value_slice_ok<DS, G>()) {
                append_pack_kernel<B, T, DS, G, 1><<<grid_for(static_cast<int64_t>(max_groups) * (G / kTile) * (a.D / DS)),
                                                     kThreads, 0, stream>>>(a);
            }
            return cudaGetLastError();
        });
        if (e != cudaSuccess) return e;
    }
    append_ring_kernel<<<a.nseq, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kivi
