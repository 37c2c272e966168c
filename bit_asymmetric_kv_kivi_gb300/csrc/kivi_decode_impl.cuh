// Split-K decode attention over the KIVI packed cache (sm_103a).
//
// One query token per sequence attends to every cached token: packed tokens
// are dequantized on the fly as c*s + z (keys: scale/zero per (group of G
// tokens, channel); values: per (token, group of G channels)), residual
// tokens are read as stored. "KIVI: Asymmetric 2-Bit KV Cache Quantization
// Guide", sections "Step 2" (dequantize during attention) and "Production
// Serving and vLLM Deployment Trade-offs in 2026" (on-the-fly dequantization
// in SRAM); "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache",
// abstract (decode is bound by loading the cache).
//
//  * decode_mma_kernel (Hq/Hkv = 1, 2, 4, 8): the dot products run on the tensor
//    cores (mma.sync m16n8k16, f16 operands, fp32 accumulation). A CTA owns a
//    range of 32-token tiles of the packed tokens of one (sequence, kv head)
//    (a key group of G = 64 is two tiles), or residual tokens of it. Each of its four warps
//    streams its groups through a private cp.async ring of shared-memory
//    stages and keeps its own online-softmax state.
//      - Scores: S[token][head] = sum_d c[token][d] * Q[d][head] + bias[head],
//        Q = q * s_k (softmax scale and log2(e) folded into q). Codes are the
//        A operand, unpacked to exact f16 integers (one lop3 + one fma per
//        pair; 4-bit keys: one lop3 + two e4m3 converts per four codes, as
//        c * 2^-9). Q is the B operand as an f16 hi + lo pair (two columns per
//        head), built with an exact-error product in f16, so the sum carries
//        about 22 bits; bias = sum_d q z_k is an MMA over 16 groups at once
//        (groups as rows).
//      - Values: O[d][head] += sum_t c[t][d] * P'[t][head] with
//        P' = p * s_v[t][group(d)] (hi + lo again), channels as M; the
//        sum_t p z_v term is a small MMA of its own.
//    q is rescaled by a power of two so that max|q| lies in (1/2, 1]; with
//    |x| <= 65504 no f16 operand can overflow.
//    Hq/Hkv = 8 runs as one stream of eight query heads per kv head
//    (group_segment8: the hi and lo parts of each product are two MMAs over
//    the same unpacked codes), so every tile is read from DRAM once. Several
//    queries (multi-query attention at Hq/Hkv = 4 or 8, and two queries at 1
//    or 2) run as one stream per query and kv head, the count set at run time.
//  * other query groups (up to 32) run on decode_multi_kernel (kivi_multi_impl.cuh)
//    with one query: its CTAs share each unpacked tile between warps of four heads.
//
// Every segment writes (m, l, acc[128]) for its query heads to the workspace, or its
// output when it holds the whole stream; decode_merge_kernel, launched behind the
// decode kernel as a programmatic dependent, merges the records of every stream split
// over several CTAs with the log-sum-exp rescaling and writes the fp32 output.
//
// This header holds the kernels as templates over the key and value code widths
// (KB, VB), the input type, the query group and G; each translation unit that
// includes it instantiates one (KB, VB) pair (launch_decode_kv), so that the
// instantiations compile in parallel.
#pragma once
#include <math_constants.h>

#include <atomic>

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

// 2^x for the softmax weights and rescale factors (x <= 0): the ex2 approximation, results
// below 2^-126 flushed to zero (such a weight adds nothing to an fp32 sum of weights >= 1)
__device__ __forceinline__ float exp2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

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

// 4-bit codes as e4m3 bytes: a byte holding b <= 15 reads as exactly b * 2^-9 (the
// subnormals and the first binade share one step), so one mask leaves four codes in bytes
// and two converts widen them to two exact f16 pairs, 0.75 instructions per code against
// one for code_pair. The convert issues at a quarter of the rate of lop3 and hfma2; it
// measured faster for 4-bit keys only (2-bit fields need more masks and shifts per byte).
__device__ __forceinline__ void e4m3_pairs(uint32_t y, uint32_t& lo, uint32_t& hi) {
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; cvt.rn.f16x2.e4m3x2 %0, l; cvt.rn.f16x2.e4m3x2 %1, h; }"
        : "=r"(lo), "=r"(hi) : "r"(y));
}
constexpr float kE4m3Unit = 512.0f;   // 2^9: a code c widened through e4m3 reads c / 512

// Key slot s (0..15) of a thread's 32-channel span: channel offsets of its pair, (off, off +
// gap). With code_pair (CVT false) slot s of word s / NSLOT pairs the fields at bits KB i
// and 16 + KB i, i = s % NSLOT. With the convert (CVT, 4-bit) the slots 2i and 2i + 1 are
// the halves of one convert of word i / 2: codes (m, m + 2) and (m + 4, m + 6) of the word's
// eight, m = i % 2.
template <int KB, bool CVT>
__host__ __device__ constexpr int kslot_off(int s) {
    return CVT ? (s / 4) * 8 + ((s % 4) >> 1) + (s & 1) * 4 : (s / (16 / KB)) * 2 * (16 / KB) + s % (16 / KB);
}
template <int KB, bool CVT>
__host__ __device__ constexpr int kslot_gap() { return CVT ? 2 : 16 / KB; }
// A slot map must cover the span's 32 channels once, pair channels of equal parity (one prmt
// selector per pair) and keep slots 8h .. 8h + 7 in channels 16h .. 16h + 15 (the bias
// batch reads the key zeros in those halves).
template <int KB, bool CVT>
constexpr bool kslot_map_ok() {
    bool seen[32] = {};
    for (int s = 0; s < 16; ++s) {
        const int c0 = kslot_off<KB, CVT>(s), c1 = c0 + kslot_gap<KB, CVT>();
        if (c0 < 0 || c1 >= 32 || seen[c0] || seen[c1] || ((c0 ^ c1) & 1)) return false;
        if (c0 / 16 != s / 8 || c1 / 16 != s / 8) return false;
        seen[c0] = seen[c1] = true;
    }
    return true;
}
static_assert(kslot_map_ok<2, false>() && kslot_map_ok<4, false>() && kslot_map_ok<4, true>(),
              "key slot maps");

template <int BITS>
struct CodeShift {
    static constexpr int kValue = ((10 - BITS) / BITS + 1) * BITS;   // 10 (2-bit), 8 (4-bit)
};

// ---------------------------------------------------------------- lane-layout pieces

// One 32-token tile of residual tokens [ts, min(ts+32, t1)) for one warp, lane = token:
// scores against the widened stored keys, online-softmax update and value accumulation
// into the lane-layout state (lane owns channels [4 lane, 4 lane + 4)). Every global
// load of the tile (the key row, then the lane's value slices of all 32 tokens) is issued
// before the first use of any, so a tile waits for memory once (for up to four heads; with
// eight, the value loads follow the scores).
template <int DT, int GQ>
__device__ __forceinline__ void residual_tile(const uint16_t* kres, const uint16_t* vres, int ring, int64_t ts,
                                              int64_t t1, const float* qs, int lane, float (&m)[GQ], float (&l)[GQ],
                                              float (&acc)[GQ][kCpl]) {
    const int64_t p = ts + lane;
    const bool valid = p < t1;
    const int ntok = static_cast<int>(t1 - ts < 32 ? t1 - ts : 32);
    const int slot0 = static_cast<int>(ts % ring);
    float sc[GQ];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) sc[hh] = 0.0f;
    uint4 kr[kD / 8];
    {
        const int slot = slot0 + lane >= ring ? slot0 + lane - ring : slot0 + lane;
        const uint4* krow = reinterpret_cast<const uint4*>(kres + static_cast<int64_t>(slot) * kD);
#pragma unroll
        for (int w = 0; w < kD / 8; ++w) kr[w] = valid ? __ldg(krow + w) : make_uint4(0, 0, 0, 0);
    }
    uint2 vr[32];
    auto load_values = [&]() {
#pragma unroll
        for (int tau = 0; tau < 32; ++tau) {
            const int slot = slot0 + tau >= ring ? slot0 + tau - ring : slot0 + tau;
            vr[tau] = tau < ntok ? __ldg(reinterpret_cast<const uint2*>(vres + static_cast<int64_t>(slot) * kD + lane * kCpl))
                                 : make_uint2(0, 0);
        }
    };
    if constexpr (GQ <= 4) load_values();   // at eight heads the lane state leaves no room to hold them early
#pragma unroll
    for (int w = 0; w < kD / 8; ++w) {
        const uint32_t words[4] = {kr[w].x, kr[w].y, kr[w].z, kr[w].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float k0 = widen<DT>(static_cast<uint16_t>(words[e] & 0xffffu));
            const float k1 = widen<DT>(static_cast<uint16_t>(words[e] >> 16));
            const int d = 8 * w + 2 * e;
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) sc[hh] = fmaf(qs[hh * kD + d + 1], k1, fmaf(qs[hh * kD + d], k0, sc[hh]));
        }
    }
    if constexpr (GQ > 4) load_values();
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
#pragma unroll
    for (int tau = 0; tau < 32; ++tau) {
        const float v[kCpl] = {widen<DT>(static_cast<uint16_t>(vr[tau].x & 0xffffu)),
                               widen<DT>(static_cast<uint16_t>(vr[tau].x >> 16)),
                               widen<DT>(static_cast<uint16_t>(vr[tau].y & 0xffffu)),
                               widen<DT>(static_cast<uint16_t>(vr[tau].y >> 16))};
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
            const float pt = __shfl_sync(kFull, pr[hh], tau);   // 0 for tokens past t1
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

// ---------------------------------------------------------------- persistent schedule

// decode_mma_kernel runs one CTA per resident slot. The work of all (sequence, kv head)
// streams, sequence-major, is a row of units: a stream's packed tokens in 32-token tiles
// (one unit each) then its residual tokens in 32-token tiles (kResidualWeight units each,
// about their cost relative to a packed tile). CTA c takes units [c U / Ceff, (c+1) U / Ceff), which
// may span streams; each stream is charged stream_overhead units ahead of its packed tiles
// for its setup and merge, which no segment holds. The part of a stream's packed tiles (or
// of its residual tiles) that one CTA holds is a segment; its partial record sits at index
// 2 s + part + c (s the stream, part 0 for packed and 1 for residual tiles), unique because each step to the next segment raises the
// stream, the part or the CTA, and below 2 S + Ceff. The last CTA to finish a segment of
// a stream (an atomic ticket, no waiting) merges the stream's records.
constexpr int kResidualWeight = 4;
constexpr int kStreamOverhead = 32;      // units charged per stream for its setup and merge
constexpr int kStreamOverheadMha = 16;   // the same at a query group of 1
// Units charged per stream. A stream of one query head (query group 1) loads one head's q
// and writes and merges one head's records, so its setup and merge cost less than a grouped
// stream's; measured, the smaller charge balanced the CTAs better on many short MHA streams
// (8 x 32 streams of 4096 tokens: 3 % faster, long streams unchanged).
__device__ __forceinline__ int64_t stream_overhead(const DecodeArgs& a) {
    return a.Hq == a.H ? kStreamOverheadMha : kStreamOverhead;
}
constexpr int kMinUnitsPerCta = 8;
constexpr int kMaxCtas = kDecodeMaxCtas;
constexpr int kMaxDevices = 64;     // devices whose launch sizes are cached

struct SeqWork {
    int64_t L, np, ng, rt, u;   // tokens, packed tokens, packed tiles, residual tiles, units
    bool bad;
};

template <int G>
__device__ __forceinline__ SeqWork seq_work(const DecodeArgs& a, int b) {
    SeqWork w;
    w.L = a.kv_len[b];
    // a.n_query is 0 for decode (an empty sequence gives zeros) and 1 for multi-query
    // attention with one query (kv_len below n_query is a length error)
    w.bad = w.L < a.n_query || w.L > a.max_kv_len || n_packed(w.L, a.R, G) > a.seqs[b].cap_tokens;
    w.np = w.ng = w.rt = w.u = 0;
    if (w.bad || w.L == 0) return w;
    w.np = n_packed(w.L, a.R, G);
    w.ng = w.np / kTile;
    w.rt = (w.L - w.np + kTile - 1) / kTile;
    w.u = stream_overhead(a) + w.ng + kResidualWeight * w.rt;
    return w;
}

// The CTA whose range holds unit x: the largest c with c U / Ceff <= x.
__device__ __forceinline__ int64_t owner(int64_t x, int64_t U, int64_t Ceff) { return ((x + 1) * Ceff - 1) / U; }

// The segments of one stream: CTAs [cg0, cg1] hold its packed tiles, [cr0, cr1] its residual tiles
// (empty ranges when first > last).
struct StreamSegs {
    int64_t s, cg0, cg1, cr0, cr1;
    int nseg;
};

// The segments of stream s whose units start at Ps (w: its sequence's work), under the split
// of U units over Ceff CTAs.
__device__ __forceinline__ StreamSegs stream_segs(int64_t s, int64_t Ps, const SeqWork& w, int64_t U, int64_t Ceff,
                                                  int64_t overhead) {
    StreamSegs ss;
    const int64_t Ws = Ps + overhead;
    ss.s = s;
    ss.cg0 = owner(Ws, U, Ceff);
    ss.cg1 = w.ng > 0 ? owner(Ws + w.ng - 1, U, Ceff) : ss.cg0 - 1;
    ss.cr0 = owner(Ws + w.ng, U, Ceff);
    ss.cr1 = w.rt > 0 ? owner(Ps + w.u - 1, U, Ceff) : ss.cr0 - 1;
    ss.nseg = static_cast<int>((ss.cg1 - ss.cg0 + 1) + (ss.cr1 - ss.cr0 + 1));
    return ss;
}

// Merges the four warps' states of one segment (red_* in shared memory, filled and
// synchronized by the caller), then writes the output (the stream's only segment) or the
// segment's partial record (m, l, acc[kD]) per head at index seg; decode_merge_kernel merges
// the records of streams with several segments. An empty state (m = -inf, l = 0)
// contributes nothing.
template <int GQ>
__device__ __forceinline__ void write_segment(const DecodeArgs& a, int nseg, int64_t seg, float* out_s,
                                              const float* red_m, const float* red_l, const float* red_acc) {
    const int tid = threadIdx.x;
    constexpr int64_t rec = kD + 4;
    for (int i = tid; i < GQ * kD; i += kThreads) {
        const int hh = i / kD, d = i - hh * kD;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * GQ + hh]);
        float den = 0.0f, num = 0.0f;
        if (M != -CUDART_INF_F) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = exp2f(red_m[w * GQ + hh] - M);
                den = fmaf(red_l[w * GQ + hh], f, den);
                num = fmaf(red_acc[(w * GQ + hh) * kD + d], f, num);
            }
        }
        if (nseg == 1) {
            out_s[i] = num / den;
        } else {
            float* r = a.partials + (seg * GQ + hh) * rec;
            r[d] = num;
            if (d == 0) {
                r[kD] = M;
                r[kD + 1] = den;
            }
        }
    }
}

// The record of the k-th segment of stream ss (its packed segments first), head hh.
template <int GQ>
__device__ __forceinline__ float* segment_record(const DecodeArgs& a, const StreamSegs& ss, int k, int hh) {
    const int ng_cnt = static_cast<int>(ss.cg1 - ss.cg0 + 1);
    const int64_t idx = k < ng_cnt ? 2 * ss.s + ss.cg0 + k : 2 * ss.s + 1 + ss.cr0 + (k - ng_cnt);
    return a.partials + (idx * GQ + hh) * (kD + 4);
}

// Merges the records of a stream with several segments into its output, then sets them back
// to zero (every call leaves the workspace as it found it, whatever plan the next call has).
// Thread d owns channel d of every head and folds the records in one pass with the
// log-sum-exp rescaling (a record with a larger max rescales what came before), so the loads
// of all records are independent of one another.
template <int GQ>
__device__ __forceinline__ void merge_stream(const DecodeArgs& a, const StreamSegs& ss, float* out_s) {
    static_assert(kThreads == kD, "one thread per channel");
    const int d = threadIdx.x;
    float M[GQ], den[GQ], num[GQ];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        M[hh] = -CUDART_INF_F;
        den[hh] = 0.0f;
        num[hh] = 0.0f;
    }
#pragma unroll 4
    for (int k = 0; k < ss.nseg; ++k) {
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
            const float* r = segment_record<GQ>(a, ss, k, hh);
            const float mk = __ldcg(r + kD), lk = __ldcg(r + kD + 1), xk = __ldcg(r + d);
            if (mk == -CUDART_INF_F) continue;   // an empty segment adds nothing
            const float Mn = fmaxf(M[hh], mk);
            const float f = exp2f(M[hh] - Mn), w = exp2f(mk - Mn);   // f = 0 while M is -inf
            den[hh] = fmaf(den[hh], f, lk * w);
            num[hh] = fmaf(num[hh], f, xk * w);
            M[hh] = Mn;
        }
    }
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) out_s[hh * kD + d] = num[hh] / den[hh];
    // the stream's records back to zero (each segment's GQ records are contiguous) once every
    // thread has read them
    __syncthreads();
    for (int k = 0; k < ss.nseg; ++k) {
        float4* z = reinterpret_cast<float4*>(segment_record<GQ>(a, ss, k, 0));
        for (int i = d; i < GQ * (kD + 4) / 4; i += kThreads) z[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
}

// Units of the streams of sequences [b_lo, b_hi) (this thread's run), the units before them
// (an exclusive scan over the CTA's threads) and the total U. sched: shared memory for
// kThreads + 1 + kWarps int64. Contains barriers: every thread of the CTA calls it.
struct UnitScan {
    int b_lo, b_hi;
    int64_t mine, start, U;
};
template <int G>
__device__ __forceinline__ UnitScan scan_units(const DecodeArgs& a, int H, int64_t* sched) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    UnitScan us;
    const int per = (a.nseq + kThreads - 1) / kThreads;
    us.b_lo = tid * per < a.nseq ? tid * per : a.nseq;
    us.b_hi = us.b_lo + per < a.nseq ? us.b_lo + per : a.nseq;
    us.mine = 0;
    for (int b = us.b_lo; b < us.b_hi; ++b) us.mine += static_cast<int64_t>(H) * seq_work<G>(a, b).u;
    // within each warp by shuffles, then the four warp totals (a serial scan by one thread
    // cost ~2 us at the start of every launch)
    int64_t incl = us.mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sched[kThreads + 1 + warp] = incl;
    __syncthreads();
    int64_t before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const int64_t x = sched[kThreads + 1 + w];
        before += w < warp ? x : 0;
        total += x;
    }
    __syncthreads();   // every thread has read the warp totals
    us.start = before + incl - us.mine;
    us.U = total;
    return us;
}

// The number of CTAs the units are split over: the grid, or fewer when there are fewer
// than kMinUnitsPerCta units per CTA.
__device__ __forceinline__ int64_t effective_ctas(int64_t U, int64_t C) {
    const int64_t by_size = U / kMinUnitsPerCta > 1 ? U / kMinUnitsPerCta : 1;
    return C < by_size ? C : by_size;
}

// ---------------------------------------------------------------- tensor-core kernel

// Key zeros for the bias term: a warp computes sum_d q[d] z_k[group][d] for kZB of its tiles
// at once (one m16 tile of MMAs, rows = tiles), from a private buffer of their key-zero rows
// (256 bytes each), filled kZB tiles ahead. The 16-byte chunk c of row r sits at position
// zpos(c, r), so that the reads (thread t: chunks 4t .. 4t + 3 of rows gid and gid + 8, one
// chunk per instruction) fall on distinct shared-memory banks.
constexpr int kZB = 16;
constexpr int kZRow = 256;
__device__ __forceinline__ int zpos(int c, int r) { return (c & ~3) | ((c + (c >> 2) + r) & 3); }

template <int KB, int VB>
struct MmaLayout {
    static constexpr int kKRowBytes = kD * KB / 8;                       // packed key row: 32 or 64 bytes
    static constexpr int kVRowBytes = kD * VB / 8;                       // and value row
    // kc, vc, ks, vs, vz; each 64-byte channel span of ks is padded to 80 bytes so that the
    // four spans read together fall on distinct shared-memory banks; vs and vz take 256 bytes
    // each (128 used when G = 64)
    static constexpr int kMetaPad = 320;
    static constexpr int kCodeBytes = kTile * (kKRowBytes + kVRowBytes);
    static constexpr int kStage = kCodeBytes + kMetaPad + 2 * 256;
    static constexpr int kNslot = 16 / KB;                               // key code pairs per 32-bit word
    static constexpr int kStageBytes = kWarps * kStages * kStage;
    static constexpr int kZBytes = kWarps * kZB * kZRow;                 // the warps' key-zero buffers
    static constexpr int kPtRows(int gq) { return gq > 4 ? gq : 4; }   // probability rows per warp
    static constexpr int kSmemBytes(int gq) {
        return kStageBytes + kZBytes + (gq * kD + kWarps * kPtRows(gq) * kPtLd + 2 * kWarps * gq + 8) * 4;
    }
};

// Thread (gid = lane / 4, t = lane % 4) follows the mma.sync
// m16n8k16 fragment layout. Logical k index 2t+8e+{0,1} of key k-step ks maps to
// the code pair of slot s = 2 ks + e in thread t's 32-channel span of the row:
// channels 32t + m*2*NSLOT + i and + NSLOT, with m = s / NSLOT, i = s % NSLOT.
struct MmaSmem {
    unsigned char* stages;   // [warp][stage][STAGE]
    unsigned char* zbuf;     // [warp][kZB][kZRow]
    float* qs;               // [GQ][kD]
    float* pt_all;           // [warp][max(4, GQ)][kPtLd]
    float* red_m;            // [warp][GQ]
    float* red_l;            // [warp][GQ]
    int* s_misc;             // [8]
    float* red_acc;          // [warp][GQ][kD], aliases the stages once they are drained
    __device__ MmaSmem(unsigned char* smem, int stage_bytes, int gq) {
        stages = smem;
        zbuf = smem + stage_bytes;
        qs = reinterpret_cast<float*>(zbuf + kWarps * kZB * kZRow);
        pt_all = qs + gq * kD;
        red_m = pt_all + kWarps * (gq > 4 ? gq : 4) * kPtLd;
        red_l = red_m + kWarps * gq;
        s_misc = reinterpret_cast<int*>(red_l + kWarps * gq);
        red_acc = reinterpret_cast<float*>(smem);
    }
};

// Streams of sequence b: h = 0 .. QS Hkv - 1, kv head h / QS. For decode (MQ = 0) QS = 1
// and a stream holds the GQ = Hq / Hkv query heads of its kv head. With several queries
// (MQ = 1) QS = n_query and stream h holds the GQ = Hq / Hkv heads of query h % QS. stream_row
// is the row of the stream's first query head in q and out ([nseq][nq][Hq][D], nq = 1 for
// decode); stream_query is its query.
template <int GQ, int MQ>
__device__ __forceinline__ int64_t stream_row(const DecodeArgs& a, int b, int h) {
    if constexpr (!MQ) return static_cast<int64_t>(b) * a.Hq + h * GQ;
    const int nq = a.n_query;
    return (static_cast<int64_t>(b) * nq + h % nq) * a.Hq + (h / nq) * GQ;
}
template <int MQ>
__device__ __forceinline__ int stream_query(const DecodeArgs& a, int h) {
    if constexpr (!MQ) return 0;
    return h % a.n_query;
}

// q rows [row, row + GQ) into shared memory, scaled by softmax_scale * log2(e); the
// caller's earlier use of qs must be over (a CTA barrier) before this runs.
template <int DT, int GQ>
__device__ __forceinline__ void load_q(const DecodeArgs& a, float* qs, int64_t row) {
    const uint16_t* q = static_cast<const uint16_t*>(a.q) + row * kD;
    for (int i = threadIdx.x; i < GQ * kD; i += kThreads) qs[i] = widen<DT>(q[i]) * a.scale_log2;
}

// Residual tiles [t0, t1) of sequence b, kv head hk (tile i = tokens np + 32 i ..), lane-layout
// CUDA-core path, over the tokens below lend (w.L, or the causal end of a stream's query);
// leaves the merged warp states in red_* (synchronized).
template <int DT, int GQ, int G>
__device__ __forceinline__ void residual_segment(const DecodeArgs& a, const MmaSmem& sm, int b, int hk,
                                                 const SeqWork& w, int64_t lend, int64_t t0, int64_t t1) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, ring = a.R + G;
    const kivi_seq& sq = a.seqs[b];
    float m[GQ], l[GQ], acc[GQ][kCpl];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
        m[hh] = -CUDART_INF_F;
        l[hh] = 0.0f;
#pragma unroll
        for (int c = 0; c < kCpl; ++c) acc[hh][c] = 0.0f;
    }
    const uint16_t* kres = static_cast<const uint16_t*>(sq.k_res) + static_cast<int64_t>(hk) * ring * kD;
    const uint16_t* vres = static_cast<const uint16_t*>(sq.v_res) + static_cast<int64_t>(hk) * ring * kD;
    const int64_t tv = (lend - w.np + kTile - 1) / kTile;   // tiles holding visible tokens
    const int64_t te = t1 < tv ? t1 : tv;
    for (int64_t i = t0 + warp; i < te; i += kWarps) {
        residual_tile<DT, GQ>(kres, vres, ring, w.np + kTile * i, lend, sm.qs, lane, m, l, acc);
        __syncwarp();
    }
    store_lane_state<GQ>(warp, lane, m, l, acc, sm.red_m, sm.red_l, sm.red_acc);
    __syncthreads();
}

// Bias term of kZB tiles of a warp, sum_d q[d] z_k[tile][d] per B column, from the key zeros
// in zb (row r = the tile r places after the batch's first): A = the zeros (row = tile), each
// register the channel pair of key-score slot s under the caller's slot map CVT (so the B
// constants of the scores serve as they are); B = bh, then bl when NB == 2 (two MMAs into
// one C). c = the C rows gid and gid + 8, columns 2t and 2t + 1.
template <int NSLOT, int NB, bool CVT = false>
__device__ __forceinline__ void bias_batch(const unsigned char* zb, int gid, int t, const uint32_t (&bh)[16],
                                           const uint32_t (&bl)[16], float (&c)[4]) {
    float c2[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // a second accumulator halves the dependent chain
    c[0] = c[1] = c[2] = c[3] = 0.0f;
    // two halves: chunks 2h, 2h + 1 of the thread's span (its words 8h .. 8h + 7) hold the
    // channel pairs of slots 8h .. 8h + 7, i.e. of k-steps 4h .. 4h + 3
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t Z0[8], Z1[8];   // rows gid and gid + 8
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int ch = 4 * t + 2 * h + j;
            const uint4 u0 = *reinterpret_cast<const uint4*>(zb + gid * kZRow + 16 * zpos(ch, gid));
            const uint4 u1 = *reinterpret_cast<const uint4*>(zb + (gid + 8) * kZRow + 16 * zpos(ch, gid + 8));
            Z0[4 * j] = u0.x; Z0[4 * j + 1] = u0.y; Z0[4 * j + 2] = u0.z; Z0[4 * j + 3] = u0.w;
            Z1[4 * j] = u1.x; Z1[4 * j + 1] = u1.y; Z1[4 * j + 2] = u1.z; Z1[4 * j + 3] = u1.w;
        }
#pragma unroll
        for (int ks = 4 * h; ks < 4 * h + 4; ++ks) {
            uint32_t za[4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int sl = 2 * ks + e;
                const int rel = kslot_off<16 / NSLOT, CVT>(sl) - 16 * h;   // channel in the half
                const int rel1 = rel + kslot_gap<16 / NSLOT, CVT>();
                const uint32_t sel = (rel & 1) ? 0x7632u : 0x5410u;
                za[2 * e] = prmt(Z0[rel >> 1], Z0[rel1 >> 1], sel);
                za[2 * e + 1] = prmt(Z1[rel >> 1], Z1[rel1 >> 1], sel);
            }
            if constexpr (NB == 2) {
                mma_f16(c, za[0], za[1], za[2], za[3], bh[2 * ks], bh[2 * ks + 1]);
                mma_f16(c2, za[0], za[1], za[2], za[3], bl[2 * ks], bl[2 * ks + 1]);
            } else if (ks & 1) {
                mma_f16(c2, za[0], za[1], za[2], za[3], bh[2 * ks], bh[2 * ks + 1]);
            } else {
                mma_f16(c, za[0], za[1], za[2], za[3], bh[2 * ks], bh[2 * ks + 1]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] += c2[i];
}

// Packed tiles [ga, gb) of sequence b, kv head hk, for the GQ query heads at q row qrow, on
// the tensor cores; leaves the merged warp states
// in red_* (synchronized). Issues its first stages, then loads the stream's q into qs.
template <int KB, int VB, int DT, int GQ, int G>
__device__ __forceinline__ void group_segment(const DecodeArgs& a, const MmaSmem& sm, int b, int64_t qrow, int hk, int64_t ga,
                                              int64_t gb) {
    using Lay = MmaLayout<KB, VB>;
    constexpr int RBK = Lay::kKRowBytes, RBV = Lay::kVRowBytes;
    constexpr int STAGE = Lay::kStage;
    constexpr int NSLOT = Lay::kNslot;
    constexpr int SHIFTK = CodeShift<KB>::kValue, SHIFTV = CodeShift<VB>::kValue;
    constexpr int TPG = G / kTile;            // tiles per key group
    constexpr int NVG = kD / G;               // value channel groups per token
    constexpr int VMETA = kTile * NVG * 2;    // bytes of value scales (or zeros) of one tile
    // 4-bit key codes are widened through e4m3 (e4m3_pairs): the scores then come out in
    // units of 2^-9, undone inside the exponent, with the key bias scaled to match. (Value
    // codes keep code_pair: through e4m3 they measured slower, their words needing a shift
    // and a byte interleave of two tokens first.)
    constexpr bool kCvtK = KB == 4;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const kivi_seq& sq = a.seqs[b];
    const int cap = sq.cap_tokens;
    unsigned char* stages = sm.stages;
    float* qs = sm.qs;
    float* pt_all = sm.pt_all;
    float* red_m = sm.red_m;
    float* red_l = sm.red_l;
    int* s_misc = sm.s_misc;
    float* red_acc = sm.red_acc;
    const int gid = lane >> 2, t = lane & 3;
    const int hh = gid >> 1, part = gid & 1;     // B column gid = (head hh, hi/lo part)
    const bool hv = GQ >= 4 || hh < GQ;   // this thread's B column belongs to a real head

    const int64_t g0 = ga, g1 = gb;
    const int64_t gfirst = g0 + warp;
    const int n_my = gfirst < g1 ? static_cast<int>((g1 - gfirst + kWarps - 1) / kWarps) : 0;
    unsigned char* my_st = stages + warp * kStages * STAGE;
    float* pt = pt_all + warp * 4 * kPtLd;

    // Tile j's code rows and value metadata sit at row-tile index rt of (32 code rows,
    // VMETA bytes of each kind of value metadata), its key scales and zeros at group index
    // kg of (256 bytes of each) from these bases: rt = j, kg = j / TPG in a contiguous
    // sequence (bases at head hk); rt = (page * H + hk) * TPG + j mod TPG, kg = page * H + hk
    // in a paged one (bases at the pools; see group_addr), page = block_table[j / TPG].
    const bool paged = seq_paged(sq);
    const int64_t hc = paged ? 0 : static_cast<int64_t>(hk) * cap;   // head offset in tokens
    const unsigned char* kc_base = sq.k_codes + hc * RBK;
    const unsigned char* vc_base = sq.v_codes + hc * RBV;
    const unsigned char* ks_base = reinterpret_cast<const unsigned char*>(sq.k_scale + hc / G * kD);
    const unsigned char* kz_base = reinterpret_cast<const unsigned char*>(sq.k_zero + hc / G * kD);
    const unsigned char* vs_base = reinterpret_cast<const unsigned char*>(sq.v_scale + hc * NVG);
    const unsigned char* vz_base = reinterpret_cast<const unsigned char*>(sq.v_zero + hc * NVG);

    // Per-lane cp.async plan of one tile: code rows as 16-byte chunks (lane + 32k), then one
    // chunk of key scales (lanes 0-15) and of value scale / zero (lanes 0-15 / 16-31 for
    // G = 32; lanes 0-7 / 8-15 for G = 64). Key zeros travel apart, kZB tiles at a time.
    constexpr int kKChunks = RBK / 16, kVChunks = RBV / 16;   // per lane, per code block
    constexpr int VL = VMETA / 16;                             // lanes per kind of value metadata
    const int half = lane >> 4, off16 = (lane & 15) * 16;
    const int vhalf = (lane / VL) & 1, voff16 = (lane % VL) * 16;
    const bool v_issue = lane < 2 * VL;
    const unsigned char* kc_lane = kc_base + lane * 16;
    const unsigned char* vc_lane = vc_base + lane * 16;
    const unsigned char* km_lane = ks_base + off16;
    const unsigned char* vm_lane = (vhalf ? vz_base : vs_base) + voff16;
    const int km_dst = Lay::kCodeBytes + (off16 >> 6) * 80 + (off16 & 63);
    const int vm_dst = Lay::kCodeBytes + Lay::kMetaPad + vhalf * 256 + voff16;
    // Tile and group indices are 32-bit (a stream has fewer than 2^32 tiles, a page pool fewer
    // than 2^32 / (H TPG) pages), so each address is one 32 x 32 -> 64-bit multiply-add.
    auto issue = [&](int slot, uint32_t j, int32_t page) {
        unsigned char* dst = my_st + slot * STAGE;
        uint32_t rt, kg;
        if (paged) {
            kg = static_cast<uint32_t>(page) * static_cast<uint32_t>(a.H) + static_cast<uint32_t>(hk);
            rt = kg * TPG + (TPG > 1 ? j % TPG : 0u);
        } else {
            rt = j;
            kg = TPG > 1 ? j / TPG : j;
        }
        const unsigned char* kc = kc_lane + static_cast<uint64_t>(rt) * (kTile * RBK);
        const unsigned char* vc = vc_lane + static_cast<uint64_t>(rt) * (kTile * RBV);
#pragma unroll
        for (int k = 0; k < kKChunks; ++k) cp_async16(dst + lane * 16 + 512 * k, kc + 512 * k);
#pragma unroll
        for (int k = 0; k < kVChunks; ++k) cp_async16(dst + kTile * RBK + lane * 16 + 512 * k, vc + 512 * k);
        if (half == 0) cp_async16(dst + km_dst, km_lane + static_cast<uint64_t>(kg) * 256);
        if (v_issue) cp_async16(dst + vm_dst, vm_lane + static_cast<uint64_t>(rt) * VMETA);
    };

    // page of this warp's i-th tile (paged sequences); the in-loop issue uses an entry
    // loaded one iteration earlier, so the table read stays off the critical path
    const uint32_t gfirst32 = static_cast<uint32_t>(gfirst);
    auto page_of = [&](int i) -> int32_t {
        return paged ? sq.block_table[(gfirst32 + kWarps * static_cast<uint32_t>(i)) / TPG] : 0;
    };
    // key zeros of this warp's tiles [i0, i0 + kZB) (those below n_my) into its buffer: lane L
    // copies chunk L % 16 of rows L / 16, L / 16 + 2, ...
    unsigned char* zb = sm.zbuf + warp * kZB * kZRow;
    auto issue_z = [&](int i0) {
        const int zc = lane & 15;
#pragma unroll
        for (int m = 0; m < kZB / 2; ++m) {
            const int r = (lane >> 4) + 2 * m, i = i0 + r;
            if (i < n_my) {
                const uint32_t j = gfirst32 + kWarps * static_cast<uint32_t>(i);
                const uint32_t kg = paged ? static_cast<uint32_t>(sq.block_table[j / TPG]) * static_cast<uint32_t>(a.H) +
                                                static_cast<uint32_t>(hk)
                                          : j / TPG;
                cp_async16(zb + r * kZRow + 16 * zpos(zc, r), kz_base + static_cast<uint64_t>(kg) * 256 + zc * 16);
            }
        }
    };
    issue_z(0);   // joins the first stage's group
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) {
        if (i < n_my) issue(i, gfirst32 + kWarps * i, page_of(i));
        cp_async_commit();
    }
    int32_t pg_ahead = kStages - 1 < n_my ? page_of(kStages - 1) : 0;

    // q of the stream, loaded while the first stages are in flight (the caller's barrier
    // has ended the previous segment's use of qs and of the stages)
    load_q<DT, GQ>(a, qs, qrow);
    __syncthreads();

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
    // B = hfma2(cX, s, hfma2(cY, s, -RN(q_hi s) or 0)): q_hi s rounded in the hi columns, its
    // exact rounding error plus q_lo s in the lo columns. The negated product comes from a
    // constant cZ = -q_hi (lo columns) or 0; with 2-bit keys it is formed from the product
    // itself instead (one more instruction per slot, sixteen fewer live registers, which
    // measured faster there and slower with 4-bit keys).
    constexpr bool kKeepZ = KB != 2;
    uint32_t cY[16], cX[16], cZ[kKeepZ ? 16 : 1];
    const uint32_t pmask = part ? 0xffffffffu : 0u;
#pragma unroll
    for (int s = 0; s < 16; ++s) {
        const int c0 = 32 * t + kslot_off<KB, kCvtK>(s), c1 = c0 + kslot_gap<KB, kCvtK>();
        const float v0 = hv ? qs[(hv ? hh : 0) * kD + c0] * qpre : 0.0f;
        const float v1 = hv ? qs[(hv ? hh : 0) * kD + c1] * qpre : 0.0f;
        const uint32_t qh = pack_h2(v0, v1);
        const uint32_t ql = pack_h2(v0 - h2_lo(qh), v1 - h2_hi(qh));
        cY[s] = qh;
        cX[s] = part ? ql : 0u;
        if constexpr (kKeepZ) cZ[s] = (qh ^ 0x80008000u) & pmask;
    }
    auto bkey = [&](const uint32_t (&sp)[16], int sl) -> uint32_t {
        uint32_t neg;
        if constexpr (kKeepZ) neg = hmul2(cZ[sl], sp[sl]);
        else neg = (hmul2(cY[sl], sp[sl]) ^ 0x80008000u) & pmask;
        return hfma2(cX[sl], sp[sl], hfma2(cY[sl], sp[sl], neg));
    };
    // value side: byte / half-word selectors of this thread's four channels per channel group
    const uint32_t g3 = static_cast<uint32_t>(gid & 3);
    const uint32_t sel_v = VB == 2 ? (g3 | (g3 << 4) | ((4 + g3) << 8) | ((4 + g3) << 12))
                                   : ((gid & 1) ? 0x7632u : 0x5410u);
    const int vbyte = VB == 2 ? 4 * (gid >> 2) : 4 * (gid >> 1);   // byte offset of the word in a 32-channel block
    const uint32_t sel_z = (gid & 1) ? 0x7632u : 0x5410u;

    float m_run = -CUDART_INF_F, l_run = 0.0f;
    float cv[8][4], cz[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) cv[i][0] = cv[i][1] = cv[i][2] = cv[i][3] = 0.0f;
    cz[0] = cz[1] = cz[2] = cz[3] = 0.0f;
    float bz_lo = 0.0f, bz_hi = 0.0f;   // the current bias batch: tiles gid and gid + 8, head t

    for (int it = 0; it < n_my; ++it) {
        {
            const int nxt = it + kStages - 1;
            if (nxt < n_my) {
                issue(nxt % kStages, gfirst32 + kWarps * static_cast<uint32_t>(nxt), pg_ahead);
                pg_ahead = nxt + 1 < n_my ? page_of(nxt + 1) : 0;
            }
            cp_async_commit();
        }
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const unsigned char* st = my_st + (it % kStages) * STAGE;
        const unsigned char* kc = st;
        const unsigned char* vc = st + kTile * RBK;
        const unsigned char* ksm = st + Lay::kCodeBytes;
        const unsigned char* vsm = ksm + Lay::kMetaPad;    // [32 tokens][NVG] fp16
        const unsigned char* vzm = vsm + 256;

        // ---- bias of this tile for head t: computed for kZB tiles at the first of them (their
        // zeros landed with this tile's stage), after which the buffer takes the next batch
        const int zr = it & (kZB - 1);
        if (zr == 0) {
            uint32_t cB[16];   // B of the bias: q hi or lo of column gid, by the column's part
#pragma unroll
            for (int sl = 0; sl < 16; ++sl) cB[sl] = part ? cX[sl] : cY[sl];
            float bz[4];
            bias_batch<NSLOT, 1, kCvtK>(zb, gid, t, cB, cB, bz);
            constexpr float kBiasUnit = kCvtK ? 1.0f / kE4m3Unit : 1.0f;   // to the scores' unit
            bz_lo = (bz[0] + bz[1]) * kBiasUnit;      // tile it + gid, head t (hi and lo columns)
            bz_hi = (bz[2] + bz[3]) * kBiasUnit;      // tile it + gid + 8
            __syncwarp();
            if (it + kZB < n_my) issue_z(it + kZB);
        }
        const float bias = __shfl_sync(kFull, zr < 8 ? bz_lo : bz_hi, 4 * (zr & 7) + t);

        // ---- key scale pairs of this thread's span
        uint32_t sp[16];
        {
            uint32_t R[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 r4 = *reinterpret_cast<const uint4*>(ksm + 80 * t + 16 * i);
                R[4 * i] = r4.x; R[4 * i + 1] = r4.y; R[4 * i + 2] = r4.z; R[4 * i + 3] = r4.w;
            }
#pragma unroll
            for (int s = 0; s < 16; ++s) {
                const int rel = kslot_off<KB, kCvtK>(s);
                const uint32_t sel = (rel & 1) ? 0x7632u : 0x5410u;
                sp[s] = prmt(R[rel >> 1], R[(rel + kslot_gap<KB, kCvtK>()) >> 1], sel);
            }
        }

        // ---- scores: A = key codes (tokens gid + 8r), B = (q * s_k) hi / lo; the bias enters
        // through the hi column
        float c0[4] = {bias, 0.0f, bias, 0.0f}, c1[4] = {bias, 0.0f, bias, 0.0f};
        {
            uint32_t cw[4][KB], cws[4][KB];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const unsigned char* row = kc + (gid + 8 * r) * RBK;
                if constexpr (KB == 2) {
                    const uint2 v = *reinterpret_cast<const uint2*>(row + 8 * t);
                    cw[r][0] = v.x; cw[r][1] = v.y;
                } else {
                    const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * t);
                    cw[r][0] = v.x; cw[r][1] = v.y; cw[r][2] = v.z; cw[r][3] = v.w;
                }
#pragma unroll
                for (int w = 0; w < KB; ++w) cws[r][w] = cw[r][w] >> (kCvtK ? 4 : SHIFTK);
            }
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int s0 = 2 * ks, s1 = 2 * ks + 1;
                const uint32_t b0 = bkey(sp, s0), b1 = bkey(sp, s1);
                const int w0 = s0 / NSLOT, w1 = s1 / NSLOT;
                uint32_t a0, a1, a2, a3;
                if constexpr (kCvtK) {
                    // k-step ks: word ks / 2, codes at the low nibble of each byte of the word
                    // (ks even) or of the word shifted by 4
                    uint32_t ak[4][2];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        e4m3_pairs(((ks & 1) ? cws[r][ks >> 1] : cw[r][ks >> 1]) & 0x0F0F0F0Fu, ak[r][0], ak[r][1]);
                    mma_f16(c0, ak[0][0], ak[1][0], ak[0][1], ak[1][1], b0, b1);
                    mma_f16(c1, ak[2][0], ak[3][0], ak[2][1], ak[3][1], b0, b1);
                    continue;
                }
                a0 = code_slot<KB>(cw[0][w0], cws[0][w0], s0);
                a1 = code_slot<KB>(cw[1][w0], cws[1][w0], s0);
                a2 = code_slot<KB>(cw[0][w1], cws[0][w1], s1);
                a3 = code_slot<KB>(cw[1][w1], cws[1][w1], s1);
                mma_f16(c0, a0, a1, a2, a3, b0, b1);
                a0 = code_slot<KB>(cw[2][w0], cws[2][w0], s0);
                a1 = code_slot<KB>(cw[3][w0], cws[3][w0], s0);
                a2 = code_slot<KB>(cw[2][w1], cws[2][w1], s1);
                a3 = code_slot<KB>(cw[3][w1], cws[3][w1], s1);
                mma_f16(c1, a0, a1, a2, a3, b0, b1);
            }
        }

        // ---- online softmax for head t over tokens gid, gid+8, gid+16, gid+24; the scores are
        // in units of the prescaled q, and qpost (a power of two) scales them exactly inside
        // the max and the exponent
        const float S[4] = {c0[0] + c0[1], c0[2] + c0[3], c1[0] + c1[1], c1[2] + c1[3]};
        float tmax = fmaxf(fmaxf(S[0], S[1]), fmaxf(S[2], S[3]));
        const float spost = kCvtK ? qpost * kE4m3Unit : qpost;   // exact: both powers of two
        // the head's max over the tile's 32 tokens (a reduction over the lanes of head t) is
        // needed only when some lane's own four tokens pass its running max; otherwise it
        // could not pass either and the state stays as it is
        if (__any_sync(kFull, tmax * spost > m_run)) {
            tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 4));
            tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
            tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
            const float mnew = fmaxf(m_run, tmax * spost);
            const float alpha = exp2_ftz(m_run - mnew);
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
        for (int r = 0; r < 4; ++r) p[r] = (GQ >= 4 || t < GQ) ? exp2_ftz(fmaf(S[r], spost, -m_run)) : 0.0f;
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
                // scales of tokens tau0 and tau0 + 4 for each 32-channel block kg (its
                // channel group is kg / TPG)
                uint32_t s0w[NVG / 2 > 0 ? NVG / 2 : 1], s1w[NVG / 2 > 0 ? NVG / 2 : 1];
                if constexpr (NVG == 4) {
                    const uint2 x0 = *reinterpret_cast<const uint2*>(vsm + tau0 * 8);
                    const uint2 x1 = *reinterpret_cast<const uint2*>(vsm + (tau0 + 4) * 8);
                    s0w[0] = x0.x; s0w[1] = x0.y; s1w[0] = x1.x; s1w[1] = x1.y;
                } else {
                    s0w[0] = *reinterpret_cast<const uint32_t*>(vsm + tau0 * 4);
                    s1w[0] = *reinterpret_cast<const uint32_t*>(vsm + (tau0 + 4) * 4);
                }
#pragma unroll
                for (int kg = 0; kg < 4; ++kg) {
                    const int vg = kg / TPG;
                    const uint32_t svp = prmt(s0w[vg >> 1], s1w[vg >> 1], (vg & 1) ? 0x7632u : 0x5410u);
                    vb[k2][e][kg] = hfma2(xp, svp, hfma2(ph, svp, hmul2(zn, svp)));
                }
                // rows of the zero-point MMA: channel group gid (gid < NVG)
                const uint32_t zw0 = *reinterpret_cast<const uint32_t*>(vzm + tau0 * (2 * NVG) + 4 * ((gid & 3) >> 1));
                const uint32_t zw1 = *reinterpret_cast<const uint32_t*>(vzm + (tau0 + 4) * (2 * NVG) + 4 * ((gid & 3) >> 1));
                za[k2][e] = gid < NVG ? prmt(zw0, zw1, sel_z) : 0u;
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
                    const int off = kg * (RBV / 4) + vbyte;
                    const uint32_t x0 = *reinterpret_cast<const uint32_t*>(vc + tau0 * RBV + off);
                    const uint32_t x1 = *reinterpret_cast<const uint32_t*>(vc + (tau0 + 4) * RBV + off);
                    wv[e] = prmt(x0, x1, sel_v);
                    wvs[e] = wv[e] >> SHIFTV;
                }
                // m-tile 2kg + u: rows gid (slot 2u) and gid + 8 (slot 2u + 1)
                mma_f16(cv[2 * kg], code_pair<VB, 0>(wv[0], wvs[0]), code_pair<VB, 1>(wv[0], wvs[0]),
                        code_pair<VB, 0>(wv[1], wvs[1]), code_pair<VB, 1>(wv[1], wvs[1]), vb[k2][0][kg],
                        vb[k2][1][kg]);
                mma_f16(cv[2 * kg + 1], code_pair<VB, 2>(wv[0], wvs[0]), code_pair<VB, 3>(wv[0], wvs[0]),
                        code_pair<VB, 2>(wv[1], wvs[1]), code_pair<VB, 3>(wv[1], wvs[1]), vb[k2][0][kg],
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
    const float zmine = cz[0] + cz[1];     // (channel group gid, head t) for gid < NVG
#pragma unroll
    for (int kg = 0; kg < 4; ++kg) zk[kg] = __shfl_sync(kFull, zmine, 4 * (kg / TPG) + t);
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
}

// Packed tiles [ga, gb) of sequence b, kv head hk, for EIGHT query heads (a query group of
// 8) at q row qrow: the same walk as group_segment, but one n8 tile holds eight heads and the
// hi and lo parts of every product go to two MMAs over the same A fragments (accumulating
// into one C), instead of two columns of one MMA. Each thread then owns one head's column
// (gid) of both parts and builds them together: hi = q_h s, lo = (q_h s - hi) + q_l s, four
// instructions for two registers. The kv head's tiles are read once for all eight heads.
// C columns 2t and 2t + 1 are heads 2t and 2t + 1, so each thread keeps the online softmax
// of two heads.
template <int KB, int VB, int DT, int G>
__device__ __forceinline__ void group_segment8(const DecodeArgs& a, const MmaSmem& sm, int b, int64_t qrow, int hk,
                                               int64_t ga, int64_t gb) {
    constexpr int GQ = 8;
    using Lay = MmaLayout<KB, VB>;
    constexpr int RBK = Lay::kKRowBytes, RBV = Lay::kVRowBytes;
    constexpr int STAGE = Lay::kStage;
    constexpr int NSLOT = Lay::kNslot;
    constexpr int SHIFTK = CodeShift<KB>::kValue, SHIFTV = CodeShift<VB>::kValue;
    constexpr int TPG = G / kTile;
    constexpr int NVG = kD / G;
    constexpr int VMETA = kTile * NVG * 2;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const kivi_seq& sq = a.seqs[b];
    const int cap = sq.cap_tokens;
    unsigned char* stages = sm.stages;
    float* qs = sm.qs;
    float* red_m = sm.red_m;
    float* red_l = sm.red_l;
    int* s_misc = sm.s_misc;
    float* red_acc = sm.red_acc;
    const int gid = lane >> 2, t = lane & 3;          // B column gid = head gid; C columns 2t, 2t+1 = heads

    const int64_t gfirst = ga + warp;
    const int n_my = gfirst < gb ? static_cast<int>((gb - gfirst + kWarps - 1) / kWarps) : 0;
    unsigned char* my_st = stages + warp * kStages * STAGE;
    float* pt = sm.pt_all + warp * GQ * kPtLd;

    const bool paged = seq_paged(sq);
    const int64_t hc = paged ? 0 : static_cast<int64_t>(hk) * cap;
    const unsigned char* kc_base = sq.k_codes + hc * RBK;
    const unsigned char* vc_base = sq.v_codes + hc * RBV;
    const unsigned char* ks_base = reinterpret_cast<const unsigned char*>(sq.k_scale + hc / G * kD);
    const unsigned char* kz_base = reinterpret_cast<const unsigned char*>(sq.k_zero + hc / G * kD);
    const unsigned char* vs_base = reinterpret_cast<const unsigned char*>(sq.v_scale + hc * NVG);
    const unsigned char* vz_base = reinterpret_cast<const unsigned char*>(sq.v_zero + hc * NVG);
    constexpr int kKChunks = RBK / 16, kVChunks = RBV / 16;
    constexpr int VL = VMETA / 16;
    const int half = lane >> 4, off16 = (lane & 15) * 16;
    const int vhalf = (lane / VL) & 1, voff16 = (lane % VL) * 16;
    const bool v_issue = lane < 2 * VL;
    const unsigned char* kc_lane = kc_base + lane * 16;
    const unsigned char* vc_lane = vc_base + lane * 16;
    const unsigned char* km_lane = ks_base + off16;
    const unsigned char* vm_lane = (vhalf ? vz_base : vs_base) + voff16;
    const int km_dst = Lay::kCodeBytes + (off16 >> 6) * 80 + (off16 & 63);
    const int vm_dst = Lay::kCodeBytes + Lay::kMetaPad + vhalf * 256 + voff16;
    // Tile and group indices are 32-bit (a stream has fewer than 2^32 tiles, a page pool fewer
    // than 2^32 / (H TPG) pages), so each address is one 32 x 32 -> 64-bit multiply-add.
    auto issue = [&](int slot, uint32_t j, int32_t page) {
        unsigned char* dst = my_st + slot * STAGE;
        uint32_t rt, kg;
        if (paged) {
            kg = static_cast<uint32_t>(page) * static_cast<uint32_t>(a.H) + static_cast<uint32_t>(hk);
            rt = kg * TPG + (TPG > 1 ? j % TPG : 0u);
        } else {
            rt = j;
            kg = TPG > 1 ? j / TPG : j;
        }
        const unsigned char* kc = kc_lane + static_cast<uint64_t>(rt) * (kTile * RBK);
        const unsigned char* vc = vc_lane + static_cast<uint64_t>(rt) * (kTile * RBV);
#pragma unroll
        for (int k = 0; k < kKChunks; ++k) cp_async16(dst + lane * 16 + 512 * k, kc + 512 * k);
#pragma unroll
        for (int k = 0; k < kVChunks; ++k) cp_async16(dst + kTile * RBK + lane * 16 + 512 * k, vc + 512 * k);
        if (half == 0) cp_async16(dst + km_dst, km_lane + static_cast<uint64_t>(kg) * 256);
        if (v_issue) cp_async16(dst + vm_dst, vm_lane + static_cast<uint64_t>(rt) * VMETA);
    };
    const uint32_t gfirst32 = static_cast<uint32_t>(gfirst);
    auto page_of = [&](int i) -> int32_t {
        return paged ? sq.block_table[(gfirst32 + kWarps * static_cast<uint32_t>(i)) / TPG] : 0;
    };
    // key zeros of this warp's tiles [i0, i0 + kZB) (those below n_my) into its buffer: lane L
    // copies chunk L % 16 of rows L / 16, L / 16 + 2, ...
    unsigned char* zb = sm.zbuf + warp * kZB * kZRow;
    auto issue_z = [&](int i0) {
        const int zc = lane & 15;
#pragma unroll
        for (int m = 0; m < kZB / 2; ++m) {
            const int r = (lane >> 4) + 2 * m, i = i0 + r;
            if (i < n_my) {
                const uint32_t j = gfirst32 + kWarps * static_cast<uint32_t>(i);
                const uint32_t kg = paged ? static_cast<uint32_t>(sq.block_table[j / TPG]) * static_cast<uint32_t>(a.H) +
                                                static_cast<uint32_t>(hk)
                                          : j / TPG;
                cp_async16(zb + r * kZRow + 16 * zpos(zc, r), kz_base + static_cast<uint64_t>(kg) * 256 + zc * 16);
            }
        }
    };
    issue_z(0);   // joins the first stage's group
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) {
        if (i < n_my) issue(i, gfirst32 + kWarps * i, page_of(i));
        cp_async_commit();
    }
    int32_t pg_ahead = kStages - 1 < n_my ? page_of(kStages - 1) : 0;

    load_q<DT, GQ>(a, qs, qrow);
    __syncthreads();
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

    // q of head gid, hi and lo, in B-fragment order (slot s: channels c0 and c0 + NSLOT of t's span)
    uint32_t qh[16], ql[16];
#pragma unroll
    for (int sl = 0; sl < 16; ++sl) {
        const int c0 = 32 * t + (sl / NSLOT) * 2 * NSLOT + (sl % NSLOT), c1 = c0 + NSLOT;
        const float v0 = qs[gid * kD + c0] * qpre, v1 = qs[gid * kD + c1] * qpre;
        qh[sl] = pack_h2(v0, v1);
        ql[sl] = pack_h2(v0 - h2_lo(qh[sl]), v1 - h2_hi(qh[sl]));
    }
    const uint32_t g3 = static_cast<uint32_t>(gid & 3);
    const uint32_t sel_v = VB == 2 ? (g3 | (g3 << 4) | ((4 + g3) << 8) | ((4 + g3) << 12))
                                   : ((gid & 1) ? 0x7632u : 0x5410u);
    const int vbyte = VB == 2 ? 4 * (gid >> 2) : 4 * (gid >> 1);
    const uint32_t sel_z = (gid & 1) ? 0x7632u : 0x5410u;

    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F}, l_run[2] = {0.0f, 0.0f};   // heads 2t, 2t + 1
    float cv[8][4], cz[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) cv[i][0] = cv[i][1] = cv[i][2] = cv[i][3] = 0.0f;
    cz[0] = cz[1] = cz[2] = cz[3] = 0.0f;
    float bz[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // the current bias batch (C rows gid, gid + 8)

    for (int it = 0; it < n_my; ++it) {
        {
            const int nxt = it + kStages - 1;
            if (nxt < n_my) {
                issue(nxt % kStages, gfirst32 + kWarps * static_cast<uint32_t>(nxt), pg_ahead);
                pg_ahead = nxt + 1 < n_my ? page_of(nxt + 1) : 0;
            }
            cp_async_commit();
        }
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const unsigned char* st = my_st + (it % kStages) * STAGE;
        const unsigned char* kc = st;
        const unsigned char* vc = st + kTile * RBK;
        const unsigned char* ksm = st + Lay::kCodeBytes;
        const unsigned char* vsm = ksm + Lay::kMetaPad;
        const unsigned char* vzm = vsm + 256;

        // bias of this tile for heads 2t and 2t + 1 (batched as in group_segment)
        const int zr = it & (kZB - 1);
        if (zr == 0) {
            bias_batch<NSLOT, 2>(zb, gid, t, qh, ql, bz);
            __syncwarp();
            if (it + kZB < n_my) issue_z(it + kZB);
        }
        const int zsrc = 4 * (zr & 7) + t;
        const float bias0 = __shfl_sync(kFull, zr < 8 ? bz[0] : bz[2], zsrc);
        const float bias1 = __shfl_sync(kFull, zr < 8 ? bz[1] : bz[3], zsrc);

        uint32_t sp[16];
        {
            uint32_t R[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 r4 = *reinterpret_cast<const uint4*>(ksm + 80 * t + 16 * i);
                R[4 * i] = r4.x; R[4 * i + 1] = r4.y; R[4 * i + 2] = r4.z; R[4 * i + 3] = r4.w;
            }
#pragma unroll
            for (int sl = 0; sl < 16; ++sl) {
                const int rel = (sl / NSLOT) * 2 * NSLOT + (sl % NSLOT);
                const uint32_t sel = (rel & 1) ? 0x7632u : 0x5410u;
                sp[sl] = prmt(R[rel >> 1], R[(rel + NSLOT) >> 1], sel);
            }
        }

        // scores: A = key codes, B = (q s_k) hi into c*, then lo into c*o
        float c0[4] = {bias0, bias1, bias0, bias1}, c1[4] = {bias0, bias1, bias0, bias1};
        float c0o[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c1o[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        {
            uint32_t cw[4][KB], cws[4][KB];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const unsigned char* row = kc + (gid + 8 * r) * RBK;
                if constexpr (KB == 2) {
                    const uint2 v = *reinterpret_cast<const uint2*>(row + 8 * t);
                    cw[r][0] = v.x; cw[r][1] = v.y;
                } else {
                    const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * t);
                    cw[r][0] = v.x; cw[r][1] = v.y; cw[r][2] = v.z; cw[r][3] = v.w;
                }
#pragma unroll
                for (int w = 0; w < KB; ++w) cws[r][w] = cw[r][w] >> SHIFTK;
            }
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int s0 = 2 * ks, s1 = 2 * ks + 1;
                const uint32_t h0 = hmul2(qh[s0], sp[s0]), h1 = hmul2(qh[s1], sp[s1]);
                const uint32_t l0 = hfma2(ql[s0], sp[s0], hfma2(qh[s0], sp[s0], h0 ^ 0x80008000u));
                const uint32_t l1 = hfma2(ql[s1], sp[s1], hfma2(qh[s1], sp[s1], h1 ^ 0x80008000u));
                const int w0 = s0 / NSLOT, w1 = s1 / NSLOT;
                uint32_t a0 = code_slot<KB>(cw[0][w0], cws[0][w0], s0), a1 = code_slot<KB>(cw[1][w0], cws[1][w0], s0);
                uint32_t a2 = code_slot<KB>(cw[0][w1], cws[0][w1], s1), a3 = code_slot<KB>(cw[1][w1], cws[1][w1], s1);
                mma_f16(c0, a0, a1, a2, a3, h0, h1);
                mma_f16(c0o, a0, a1, a2, a3, l0, l1);
                a0 = code_slot<KB>(cw[2][w0], cws[2][w0], s0); a1 = code_slot<KB>(cw[3][w0], cws[3][w0], s0);
                a2 = code_slot<KB>(cw[2][w1], cws[2][w1], s1); a3 = code_slot<KB>(cw[3][w1], cws[3][w1], s1);
                mma_f16(c1, a0, a1, a2, a3, h0, h1);
                mma_f16(c1o, a0, a1, a2, a3, l0, l1);
            }
        }

        // online softmax of heads 2t (e = 0) and 2t + 1 (e = 1) over tokens gid, gid+8, gid+16, gid+24
        // (scores in units of the prescaled q; qpost applied exactly inside the max and the exponent)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            c0[i] += c0o[i];
            c1[i] += c1o[i];
        }
        float p[2][4];
        bool grow = false;
        float mnew[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float tmax = fmaxf(fmaxf(c0[e], c0[2 + e]), fmaxf(c1[e], c1[2 + e]));
            tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 4));
            tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 8));
            tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, 16));
            mnew[e] = fmaxf(m_run[e], tmax * qpost);
            grow |= mnew[e] > m_run[e];
        }
        if (__any_sync(kFull, grow)) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float alpha = exp2_ftz(m_run[e] - mnew[e]);
                l_run[e] *= alpha;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    cv[i][e] *= alpha;
                    cv[i][2 + e] *= alpha;
                }
                cz[e] *= alpha;
                cz[2 + e] *= alpha;
                m_run[e] = mnew[e];
            }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            p[e][0] = exp2_ftz(fmaf(c0[e], qpost, -m_run[e]));
            p[e][1] = exp2_ftz(fmaf(c0[2 + e], qpost, -m_run[e]));
            p[e][2] = exp2_ftz(fmaf(c1[e], qpost, -m_run[e]));
            p[e][3] = exp2_ftz(fmaf(c1[2 + e], qpost, -m_run[e]));
            l_run[e] += (p[e][0] + p[e][1]) + (p[e][2] + p[e][3]);
        }
        // token 8r + j to column 8r + 2 (j % 4) + j / 4, as in group_segment
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int r = 0; r < 4; ++r) pt[(2 * t + e) * kPtLd + 8 * r + 2 * (gid & 3) + (gid >> 2)] = p[e][r];
        __syncwarp();

        // value side B operands of head gid: P' = p s_v hi and lo, and p hi and lo (z_v term)
        uint32_t vbh[2][2][4], vbl[2][2][4], bph[2][2], bpl[2][2], za[2][2];
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tau0 = 16 * k2 + 8 * e + t;
                const float2 pp = *reinterpret_cast<const float2*>(pt + gid * kPtLd + 16 * k2 + 8 * e + 2 * t);
                const uint32_t ph = pack_h2(pp.x, pp.y);
                const uint32_t pl = pack_h2(pp.x - h2_lo(ph), pp.y - h2_hi(ph));
                bph[k2][e] = ph;
                bpl[k2][e] = pl;
                uint32_t s0w[NVG / 2 > 0 ? NVG / 2 : 1], s1w[NVG / 2 > 0 ? NVG / 2 : 1];
                if constexpr (NVG == 4) {
                    const uint2 x0 = *reinterpret_cast<const uint2*>(vsm + tau0 * 8);
                    const uint2 x1 = *reinterpret_cast<const uint2*>(vsm + (tau0 + 4) * 8);
                    s0w[0] = x0.x; s0w[1] = x0.y; s1w[0] = x1.x; s1w[1] = x1.y;
                } else {
                    s0w[0] = *reinterpret_cast<const uint32_t*>(vsm + tau0 * 4);
                    s1w[0] = *reinterpret_cast<const uint32_t*>(vsm + (tau0 + 4) * 4);
                }
#pragma unroll
                for (int kg = 0; kg < 4; ++kg) {
                    const int vg = kg / TPG;
                    const uint32_t svp = prmt(s0w[vg >> 1], s1w[vg >> 1], (vg & 1) ? 0x7632u : 0x5410u);
                    const uint32_t hv = hmul2(ph, svp);
                    vbh[k2][e][kg] = hv;
                    vbl[k2][e][kg] = hfma2(pl, svp, hfma2(ph, svp, hv ^ 0x80008000u));
                }
                const uint32_t zw0 = *reinterpret_cast<const uint32_t*>(vzm + tau0 * (2 * NVG) + 4 * ((gid & 3) >> 1));
                const uint32_t zw1 = *reinterpret_cast<const uint32_t*>(vzm + (tau0 + 4) * (2 * NVG) + 4 * ((gid & 3) >> 1));
                za[k2][e] = gid < NVG ? prmt(zw0, zw1, sel_z) : 0u;
            }
        }
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
            mma_f16(cz, za[k2][0], 0u, za[k2][1], 0u, bph[k2][0], bph[k2][1]);
            mma_f16(cz, za[k2][0], 0u, za[k2][1], 0u, bpl[k2][0], bpl[k2][1]);
        }

        // value codes (A = codes^T, rows = channels) against hi, then lo
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
#pragma unroll
            for (int kg = 0; kg < 4; ++kg) {
                uint32_t wv[2], wvs[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tau0 = 16 * k2 + 8 * e + t;
                    const int off = kg * (RBV / 4) + vbyte;
                    const uint32_t x0 = *reinterpret_cast<const uint32_t*>(vc + tau0 * RBV + off);
                    const uint32_t x1 = *reinterpret_cast<const uint32_t*>(vc + (tau0 + 4) * RBV + off);
                    wv[e] = prmt(x0, x1, sel_v);
                    wvs[e] = wv[e] >> SHIFTV;
                }
                const uint32_t a00 = code_pair<VB, 0>(wv[0], wvs[0]), a01 = code_pair<VB, 1>(wv[0], wvs[0]);
                const uint32_t a02 = code_pair<VB, 0>(wv[1], wvs[1]), a03 = code_pair<VB, 1>(wv[1], wvs[1]);
                const uint32_t a10 = code_pair<VB, 2>(wv[0], wvs[0]), a11 = code_pair<VB, 3>(wv[0], wvs[0]);
                const uint32_t a12 = code_pair<VB, 2>(wv[1], wvs[1]), a13 = code_pair<VB, 3>(wv[1], wvs[1]);
                mma_f16(cv[2 * kg], a00, a01, a02, a03, vbh[k2][0][kg], vbh[k2][1][kg]);
                mma_f16(cv[2 * kg + 1], a10, a11, a12, a13, vbh[k2][0][kg], vbh[k2][1][kg]);
                mma_f16(cv[2 * kg], a00, a01, a02, a03, vbl[k2][0][kg], vbl[k2][1][kg]);
                mma_f16(cv[2 * kg + 1], a10, a11, a12, a13, vbl[k2][0][kg], vbl[k2][1][kg]);
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();

    // warp state -> merge arrays (red_acc aliases the stages: wait for every warp)
    float l_tot[2];
    float zk[2][4];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        float x = l_run[e];
        x += __shfl_xor_sync(kFull, x, 4);
        x += __shfl_xor_sync(kFull, x, 8);
        x += __shfl_xor_sync(kFull, x, 16);
        l_tot[e] = x;
#pragma unroll
        for (int kg = 0; kg < 4; ++kg) zk[e][kg] = __shfl_sync(kFull, cz[e], 4 * (kg / TPG) + t);  // (group, head 2t + e)
    }
    __syncthreads();
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int kg = mt >> 1;
        const int ch = 32 * kg + 4 * gid + 2 * (mt & 1);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            red_acc[(warp * GQ + 2 * t + e) * kD + ch] = cv[mt][e] + zk[e][kg];
            red_acc[(warp * GQ + 2 * t + e) * kD + ch + 1] = cv[mt][2 + e] + zk[e][kg];
        }
    }
    if (gid == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            red_m[warp * GQ + 2 * t + e] = m_run[e];
            red_l[warp * GQ + 2 * t + e] = l_tot[e];
        }
    }
    __syncthreads();
}

template <int KB, int VB, int DT, int GQ, int G, int MQ>
__global__ void __launch_bounds__(kThreads, KB + VB <= 6 ? 3 : 2) decode_mma_kernel(DecodeArgs a) {
    static_assert(GQ == 1 || GQ == 2 || GQ == 4 || GQ == 8, "one n8 tile: hi and lo of up to four heads, or eight heads");
    static_assert(MQ == 0 || GQ == 1 || GQ == 2 || GQ == 4 || GQ == 8, "one n8 tile per stream");
    extern __shared__ __align__(16) unsigned char smem[];
    const MmaSmem sm(smem, MmaLayout<KB, VB>::kStageBytes, GQ);
    int64_t* sched = reinterpret_cast<int64_t*>(smem);   // scan scratch: the stages are idle until the walk
    const int tid = threadIdx.x;
    // the merge kernel behind this one may be scheduled from now on (it waits for this grid's
    // completion before it reads anything this grid writes)
    asm volatile("griddepcontrol.launch_dependents;");
    // streams: (sequence, h), kv head h / QS: decode has one per kv head (its GQ query heads);
    // several queries (MQ) have one per query and kv head, each reading the kv head
    const int QS = MQ ? a.n_query : 1;   // streams per kv head
    const int C = gridDim.x, c = blockIdx.x, H = a.H * QS;

    // sequences without work: zeros for an empty one, NaN and a status for a bad length
    for (int b = c; b < a.nseq; b += C) {
        const SeqWork w = seq_work<G>(a, b);
        if (w.u != 0) continue;
        const int rows = a.Hq * QS;
        float* o = a.out + static_cast<int64_t>(b) * rows * kD;
        for (int i = tid; i < rows * kD; i += kThreads) o[i] = w.bad ? CUDART_NAN_F : 0.0f;
        if (w.bad && tid == 0) set_status(a.status, KIVI_ERR_LENGTH);
    }

    // the walk state lives in shared memory and is read back (volatile) around each
    // segment, so that the hot loops do not hold it in registers: lo, hi, U, Ceff, the
    // first unit of sequence b, b, h (b = nseq ends the walk)
    __shared__ int64_t walk[7];
    volatile int64_t* vw = walk;
    if (tid == 0) vw[5] = a.nseq;
    // units before each thread's run of sequences (exclusive scan), the total U, and this
    // CTA's range [lo, hi)
    const UnitScan us = scan_units<G>(a, H, sched);
    const int b_lo = us.b_lo, b_hi = us.b_hi;
    const int64_t mine = us.mine, U = us.U;
    const int64_t Ceff = effective_ctas(U, C);
    if (U == 0 || c >= Ceff) return;
    const int64_t lo = c * U / Ceff, hi = (c + 1) * U / Ceff;
    const int64_t start = us.start;
    if (mine > 0 && lo >= start && lo < start + mine) {
        int64_t p = start;
        for (int b = b_lo; b < b_hi; ++b) {
            const int64_t us = seq_work<G>(a, b).u, ub = static_cast<int64_t>(H) * us;
            if (lo < p + ub) {
                vw[0] = lo;
                vw[1] = hi;
                vw[2] = U;
                vw[3] = Ceff;
                vw[4] = p;
                vw[5] = b;
                vw[6] = (lo - p) / us;   // the stream holding lo (the walk need not visit those before it)
                break;
            }
            p += ub;
        }
    }
    __syncthreads();

    // stream (vw[5], vw[6]) and the part of it this CTA holds: [x0, x1) in its units
    // (x0, x1 count from the stream's first group; x1 <= x0: no work here)
    struct Cur {
        int b, h;
        int64_t Ps, Ws, x0, x1;   // first unit of the stream and of its groups
        SeqWork w;
    };
    auto current = [&]() {
        Cur k;
        k.b = static_cast<int>(vw[5]);
        k.h = static_cast<int>(vw[6]);
        k.w = seq_work<G>(a, k.b);
        k.Ps = vw[4] + k.h * k.w.u;
        k.Ws = k.Ps + stream_overhead(a);
        const int64_t lo_ = vw[0], hi_ = vw[1];
        k.x0 = (lo_ > k.Ws ? lo_ : k.Ws) - k.Ws;
        k.x1 = (hi_ < k.Ps + k.w.u ? hi_ : k.Ps + k.w.u) - k.Ws;
        return k;
    };
    // the segment's output (the stream's only segment) or its partial record at 2 s + part + c,
    // which is unique (each step to the next segment raises the stream, the part or the CTA)
    // and below 2 S + Ceff
    auto finish = [&](int part) {
        const Cur k = current();
        const int64_t s_ = static_cast<int64_t>(k.b) * H + k.h;
        const StreamSegs ss = stream_segs(s_, k.Ps, k.w, vw[2], vw[3], stream_overhead(a));
        float* out_s = a.out + stream_row<GQ, MQ>(a, k.b, k.h) * kD;
        write_segment<GQ>(a, ss.nseg, 2 * s_ + part + c, out_s, sm.red_m, sm.red_l, sm.red_acc);
    };

    while (true) {
        {
            const int b = static_cast<int>(vw[5]);
            if (b >= a.nseq || vw[4] >= vw[1]) break;
        }
        Cur k = current();
        if (k.Ps >= vw[1]) break;
        if (k.w.u != 0 && k.x1 > k.x0) {
            bool q_ready = false;   // qs holds this stream's q (loaded by its group segment here)
            if (k.x0 < k.w.ng) {
                __syncthreads();   // the previous segment is done with qs and the shared arrays
                if constexpr (GQ == 8)
                    group_segment8<KB, VB, DT, G>(a, sm, k.b, stream_row<GQ, MQ>(a, k.b, k.h), k.h / QS, k.x0,
                                                  k.x1 < k.w.ng ? k.x1 : k.w.ng);
                else
                    group_segment<KB, VB, DT, GQ, G>(a, sm, k.b, stream_row<GQ, MQ>(a, k.b, k.h), k.h / QS, k.x0,
                                                     k.x1 < k.w.ng ? k.x1 : k.w.ng);
                finish(0);
                k = current();
                q_ready = true;
            }
            if (k.x1 > k.w.ng) {
                const int64_t u0 = (k.x0 > k.w.ng ? k.x0 : k.w.ng) - k.w.ng, u1 = k.x1 - k.w.ng;
                __syncthreads();   // the merge arrays and qs are free
                if (!q_ready) {
                    load_q<DT, GQ>(a, sm.qs, stream_row<GQ, MQ>(a, k.b, k.h));
                    __syncthreads();
                }
                // the stream's query i sees tokens below L - n_query + 1 + i (L for decode)
                const int64_t lend = k.w.L - (QS - 1 - stream_query<MQ>(a, k.h));
                residual_segment<DT, GQ, G>(a, sm, k.b, k.h / QS, k.w, lend, (u0 + kResidualWeight - 1) / kResidualWeight,
                                         (u1 + kResidualWeight - 1) / kResidualWeight);
                finish(1);
            }
        }
        __syncthreads();   // every thread has read the walk state of this stream
        if (tid == 0) {
            const int b = static_cast<int>(vw[5]), h = static_cast<int>(vw[6]);
            if (h + 1 < H) {
                vw[6] = h + 1;
            } else {
                vw[4] = vw[4] + static_cast<int64_t>(H) * seq_work<G>(a, b).u;
                vw[5] = b + 1;
                vw[6] = 0;
            }
        }
        __syncthreads();
    }
}

// Resident CTAs of a kernel on the current device (SM count x blocks per SM), at most
// kMaxCtas. The first launch of an instantiation on a device raises its dynamic shared
// memory limit, asks the occupancy calculator and caches the count in an atomic per-device
// slot; later launches read the slot. Host threads that race on a first launch compute and
// store the same value.
template <typename K>
int resident_ctas(K kernel, int smem, std::atomic<int>* cache) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    const int have = cache[dev].load(std::memory_order_relaxed);
    if (have > 0) return have;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) != cudaSuccess) return 0;
    int n = sms * (per_sm > 0 ? per_sm : 1);
    n = n > kMaxCtas ? kMaxCtas : n;
    cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Merges the streams that the C CTAs of decode_mma_kernel split into several segments: it
// recomputes the same plan (the row of units, its split over effective_ctas(U, C) CTAs), and
// each of its CTAs merges the records of a stride of streams (merge_stream). Launched right
// behind the decode kernel as a programmatic dependent: its launch and its plan (which reads
// only kv_len and the sequence table) overlap the decode tail, and griddepcontrol.wait holds
// every thread until the decode grid has completed and its records are visible.
constexpr int kMergeCtas = 1024;   // grid bound (a grid-stride loop covers more streams)
template <int GQ, int G, int MQ>
__global__ void __launch_bounds__(kThreads) decode_merge_kernel(DecodeArgs a, int C) {
    __shared__ int64_t sched[kThreads + 1 + kWarps];
    __shared__ int64_t stream_at[2];   // first unit of the stream, units of one of its sequence's streams
    const int H = a.H * (MQ ? a.n_query : 1);
    const UnitScan us = scan_units<G>(a, H, sched);
    const int64_t Ceff = effective_ctas(us.U, C);
    const int64_t S = us.U == 0 ? 0 : static_cast<int64_t>(a.nseq) * H;
    for (int64_t s = blockIdx.x; s < S; s += gridDim.x) {
        const int b = static_cast<int>(s / H), h = static_cast<int>(s % H);
        if (b >= us.b_lo && b < us.b_hi) {   // the thread whose run holds sequence b
            int64_t p = us.start;
            for (int bb = us.b_lo; bb < b; ++bb) p += static_cast<int64_t>(H) * seq_work<G>(a, bb).u;
            const int64_t u = seq_work<G>(a, b).u;
            stream_at[0] = p + h * u;
            stream_at[1] = u;
        }
        __syncthreads();
        const int64_t Ps = stream_at[0], u = stream_at[1];
        __syncthreads();   // every thread has read stream_at
        if (u == 0) continue;
        const StreamSegs ss = stream_segs(s, Ps, seq_work<G>(a, b), us.U, Ceff, stream_overhead(a));
        if (ss.nseg < 2) continue;
        asm volatile("griddepcontrol.wait;" ::: "memory");   // returns at once after the first time
        merge_stream<GQ>(a, ss, a.out + stream_row<GQ, MQ>(a, b, h) * kD);
    }
}

template <int KB, int VB, int DT, int GQ, int G, int MQ = 0>
cudaError_t launch_mma(const DecodeArgs& a, cudaStream_t stream) {
    constexpr int smem = MmaLayout<KB, VB>::kSmemBytes(GQ);
    static std::atomic<int> ctas[kMaxDevices];
    const int n = resident_ctas(decode_mma_kernel<KB, VB, DT, GQ, G, MQ>, smem, ctas);
    if (n <= 0) return cudaErrorInvalidValue;
    decode_mma_kernel<KB, VB, DT, GQ, G, MQ><<<n, kThreads, smem, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t S = static_cast<int64_t>(a.nseq) * a.H * (MQ ? a.n_query : 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(S < kMergeCtas ? S : kMergeCtas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel<GQ, G, MQ>, a, n);
}

template <int KB, int VB, int DT, int G>
cudaError_t launch_gq(const DecodeArgs& a, cudaStream_t stream) {
    const int g = a.Hq / a.H;
    if (a.n_query > 1) {   // several queries: one stream of the g heads of each query per kv head
        switch (g) {
            case 1: return launch_mma<KB, VB, DT, 1, G, 1>(a, stream);
            case 2: return launch_mma<KB, VB, DT, 2, G, 1>(a, stream);
            case 4: return launch_mma<KB, VB, DT, 4, G, 1>(a, stream);
            case 8: return launch_mma<KB, VB, DT, 8, G, 1>(a, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (g) {
        case 1: return launch_mma<KB, VB, DT, 1, G>(a, stream);
        case 2: return launch_mma<KB, VB, DT, 2, G>(a, stream);
        case 4: return launch_mma<KB, VB, DT, 4, G>(a, stream);
        case 8: return launch_mma<KB, VB, DT, 8, G>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

// Decode for one pair of code widths: dispatches the input type and G.
template <int KB, int VB>
cudaError_t launch_kv(const DecodeArgs& a, cudaStream_t stream) {
    if (a.nseq == 0) return cudaSuccess;
    if (a.G == 64) {
        return a.dtype == KIVI_F16 ? launch_gq<KB, VB, KIVI_F16, 64>(a, stream)
                                   : launch_gq<KB, VB, KIVI_BF16, 64>(a, stream);
    }
    return a.dtype == KIVI_F16 ? launch_gq<KB, VB, KIVI_F16, 32>(a, stream) : launch_gq<KB, VB, KIVI_BF16, 32>(a, stream);
}

}  // namespace
}  // namespace kivi
