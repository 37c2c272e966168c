// Multi-query attention over the KIVI packed cache (sm_103a): the n_query newest
// tokens of each sequence attend causally to the cache (query i at position
// L - n_query + i sees positions [0, L - n_query + i]), as in speculative-decoding
// verification and chunked prefill. Dequantization on the fly follows "KIVI:
// Asymmetric 2-Bit KV Cache Quantization Guide", section "Step 2"; the pages do not
// describe several queries per step, so the causal reading is this library's.
//
// decode_multi_kernel. The V = n_query * Hq/Hkv (query, head) pairs of one kv head
// ("virtual heads", query-major: v = i * g + hh) share every byte of the cache they
// read, so one CTA serves all of them: W = ceil(V / 4) warps, warp w owning virtual
// heads 4w .. 4w + 3 (one n8 tile of hi / lo B columns, as in decode_mma_kernel).
// Per 32-token packed tile the CTA
//   1. streams the packed tile (codes and metadata) into a ring of shared-memory
//      stages with cp.async (all threads);
//   2. dequantizes it once into two f16 tiles of exact code values (keys and values,
//      [token][position], position p of a row holding channel P(p): the two codes of
//      one unpacked pair side by side), and gathers the key scale / zero pairs in the
//      order of the B fragments;
//   3. lets every warp load its A fragments with ldmatrix (keys: rows = tokens;
//      values: ldmatrix.trans, rows = positions) and run the same tensor-core
//      arithmetic as decode_mma_kernel for its four virtual heads.
// The unpack cost is paid once per tile instead of once per warp. The causal mask
// only touches the residual window (n_query <= 32 <= R), which a split of its own
// reads on the CUDA cores with a per-head visible length. Splits are fixed token
// ranges of packed tiles plus that residual split; the last CTA of a (sequence, kv
// head) to finish (an atomic ticket, no waiting) merges the splits' records.
#pragma once
#include "kivi_decode_impl.cuh"

namespace kivi {
namespace {

constexpr int kF16Pitch = 272;           // bytes per token row of the f16 tiles (256 + 16: no bank conflicts)

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const unsigned char* p) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const unsigned char* p) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s)
                 : "memory");
}

// Channel held at position p (0..127) of an f16 row: the unpack of a 32-bit word of
// B-bit codes gives pairs (c, c + 16 / B) side by side (code_pair), so positions
// 2s, 2s + 1 of the word's block hold channels s and s + 16 / B of it.
template <int B>
__host__ __device__ constexpr int pos_channel(int p) {
    if (B == 2) return 16 * (p / 16) + (p % 16) / 2 + 8 * (p % 2);
    return 8 * (p / 8) + (p % 8) / 2 + 4 * (p % 2);
}

template <int KB, int VB, int W>
struct MultiLayout {
    static constexpr int kStages = 4;                                  // cp.async ring depth (CTA-wide)
    static constexpr int kKRow = kD * KB / 8, kVRow = kD * VB / 8;
    static constexpr int kKMeta = kTile * kKRow + kTile * kVRow;      // stage: key scale, key zero (256 B each)
    static constexpr int kVMeta = kKMeta + 512;                        // value scale, value zero (256 B each)
    static constexpr int kStage = kVMeta + 512;
    static constexpr int kF16 = kStages * kStage;                      // two buffers of (f16 key tile, value tile)
    static constexpr int kF16Buf = 2 * kTile * kF16Pitch;
    static constexpr int kPerm = kF16 + 2 * kF16Buf;                   // two of key scale / zero pairs [2][8][4][2] u32
    static constexpr int kQs = kPerm + 2 * 2 * 8 * 4 * 2 * 4;          // [4W][kD] f32
    static constexpr int kPt = kQs + 4 * W * kD * 4;                   // [W][4][kPtLd] f32
    static constexpr int kMisc = kPt + W * 4 * kPtLd * 4;              // [8] ints
    static constexpr int kBytes = kMisc + 8 * 4;
};

// The residual tokens [ts, ts + 32) of stream (b, h) for one warp's four virtual heads,
// lane = token, each head seeing the tokens below its own end t1[hh]: scores against
// the stored keys, online softmax, value accumulation in the lane layout.
template <int DT>
__device__ __forceinline__ void residual_tile_masked(const uint16_t* kres, const uint16_t* vres, int ring, int64_t ts,
                                                     const int64_t (&t1)[4], const float* qs, int lane, float (&m)[4],
                                                     float (&l)[4], float (&acc)[4][kCpl]) {
    const int64_t p = ts + lane;
    const int64_t tmax_end = max(max(t1[0], t1[1]), max(t1[2], t1[3]));
    const int ntok = static_cast<int>(tmax_end - ts < 32 ? (tmax_end > ts ? tmax_end - ts : 0) : 32);
    const int slot0 = static_cast<int>(ts % ring);
    // keys in two halves of the row and values in runs of eight tokens, every load of a
    // part issued before its first use (this path shares the kernel's register budget
    // with the tensor-core path)
    float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int kslot = slot0 + lane >= ring ? slot0 + lane - ring : slot0 + lane;
    const uint4* krow = reinterpret_cast<const uint4*>(kres + static_cast<int64_t>(kslot) * kD);
    const bool any = lane < ntok;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint4 kr[kD / 16];
#pragma unroll
        for (int w = 0; w < kD / 16; ++w) kr[w] = any ? __ldg(krow + half * (kD / 16) + w) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int w = 0; w < kD / 16; ++w) {
            const uint32_t words[4] = {kr[w].x, kr[w].y, kr[w].z, kr[w].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float k0 = widen<DT>(static_cast<uint16_t>(words[e] & 0xffffu));
                const float k1 = widen<DT>(static_cast<uint16_t>(words[e] >> 16));
                const int d = 8 * (half * (kD / 16) + w) + 2 * e;
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) sc[hh] = fmaf(qs[hh * kD + d + 1], k1, fmaf(qs[hh * kD + d], k0, sc[hh]));
            }
        }
    }
    float pr[4];
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
        const bool valid = p < t1[hh];
        const float tmax = warp_max(valid ? sc[hh] : -CUDART_INF_F);
        const float mnew = fmaxf(m[hh], tmax);
        // a head with nothing visible so far keeps m = -inf and l = 0
        const float alpha = mnew == -CUDART_INF_F ? 1.0f : exp2f(m[hh] - mnew);
        pr[hh] = valid ? exp2f(sc[hh] - mnew) : 0.0f;
        l[hh] = l[hh] * alpha + warp_sum(pr[hh]);
#pragma unroll
        for (int c = 0; c < kCpl; ++c) acc[hh][c] *= alpha;
        m[hh] = mnew;
    }
#pragma unroll
    for (int run = 0; run < 4; ++run) {
        uint2 vr[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int tau = 8 * run + j;
            const int slot = slot0 + tau >= ring ? slot0 + tau - ring : slot0 + tau;
            vr[j] = tau < ntok ? __ldg(reinterpret_cast<const uint2*>(vres + static_cast<int64_t>(slot) * kD + lane * kCpl))
                               : make_uint2(0, 0);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float v[kCpl] = {widen<DT>(static_cast<uint16_t>(vr[j].x & 0xffffu)),
                                   widen<DT>(static_cast<uint16_t>(vr[j].x >> 16)),
                                   widen<DT>(static_cast<uint16_t>(vr[j].y & 0xffffu)),
                                   widen<DT>(static_cast<uint16_t>(vr[j].y >> 16))};
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                const float pt = __shfl_sync(kFull, pr[hh], 8 * run + j);   // 0 for tokens a head does not see
#pragma unroll
                for (int c = 0; c < kCpl; ++c) acc[hh][c] = fmaf(pt, v[c], acc[hh][c]);
            }
        }
    }
}

// Grid (split, kv head, sequence); W warps. Splits 0 .. nsp - 1 take a.chunk tokens of
// packed tiles each; split nsp (when the sequence has residual tokens) takes the
// residual window. a.max_splits bounds the splits per stream (workspace records).
template <int KB, int VB, int DT, int W, int G>
__global__ void __launch_bounds__(32 * W, W >= 4 ? 12 / W : (W == 2 ? 5 : 8)) decode_multi_kernel(DecodeArgs a) {
    using Lay = MultiLayout<KB, VB, W>;
    constexpr int RBK = Lay::kKRow, RBV = Lay::kVRow;
    constexpr int NT = 32 * W;                 // threads
    constexpr int TPG = G / kTile;             // tiles per key group
    constexpr int NVG = kD / G;                // value channel groups per token
    constexpr int VMETA = kTile * NVG * 2;     // bytes of value scales (or zeros) of one tile
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* stages = smem;
    constexpr int S = Lay::kStages;
    unsigned char* kf = smem + Lay::kF16;                      // [buf][key, value][32][kF16Pitch] f16 codes
    uint32_t* perm = reinterpret_cast<uint32_t*>(smem + Lay::kPerm);   // [buf][scale / zero][ks][t][e]
    float* qs_all = reinterpret_cast<float*>(smem + Lay::kQs);
    float* pt_all = reinterpret_cast<float*>(smem + Lay::kPt);
    int* s_misc = reinterpret_cast<int*>(smem + Lay::kMisc);

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // n_query == 0: decode attention (one query, an empty sequence gives zeros)
    const int nq = a.n_query > 0 ? a.n_query : 1;
    const int g = a.Hq / a.H, V = nq * g;
    const kivi_seq& sq = a.seqs[b];
    const int64_t L = a.kv_len[b];
    const bool empty = a.n_query == 0 && L == 0;
    const bool bad = (L < nq && !empty) || L > a.max_kv_len || n_packed(L, a.R, G) > sq.cap_tokens;
    // out[b][i][hq][d]; virtual head v = i * g + hh -> row (b * nq + i) * Hq + h * g + hh
    auto out_row = [&](int v) {
        const int i = v / g, hh = v - i * g;
        return a.out + ((static_cast<int64_t>(b) * nq + i) * a.Hq + static_cast<int64_t>(h) * g + hh) * kD;
    };
    if (bad || empty) {
        if (split == 0) {
            for (int i = tid; i < V * kD; i += NT) out_row(i / kD)[i % kD] = bad ? CUDART_NAN_F : 0.0f;
            if (bad && h == 0 && tid == 0) set_status(a.status, KIVI_ERR_LENGTH);
        }
        return;
    }
    const int64_t np = n_packed(L, a.R, G);
    const int64_t ntiles = np / kTile;
    const int64_t tps = a.chunk / kTile;                       // packed tiles per split
    const int nsp = static_cast<int>((ntiles + tps - 1) / tps);
    const int nsplit = nsp + (L > np ? 1 : 0);
    if (split >= nsplit) return;

    // q of the warp's virtual heads, times softmax_scale * log2(e); zero for padding heads
    const int v0 = 4 * warp;
    float* qs = qs_all + v0 * kD;
    for (int i = lane; i < 4 * kD; i += 32) {
        const int v = v0 + i / kD, d = i % kD;
        float x = 0.0f;
        if (v < V) {
            const int qi = v / g, hh = v - qi * g;
            const uint16_t* q = static_cast<const uint16_t*>(a.q) +
                                ((static_cast<int64_t>(b) * nq + qi) * a.Hq + static_cast<int64_t>(h) * g + hh) * kD;
            x = widen<DT>(q[d]) * a.scale_log2;
        }
        qs[i] = x;
    }
    __syncwarp();

    const int rec_stride = kD + 4;
    const int64_t rec_base = (static_cast<int64_t>(b) * a.H + h) * a.max_splits;
    auto record = [&](int v) { return a.partials + ((rec_base + split) * (4 * W) + v) * rec_stride; };

    if (split == nsp) {
        // ---- residual split: lane = token, every head up to its own visible end
        const int ring = a.R + G;
        const uint16_t* kres = static_cast<const uint16_t*>(sq.k_res) + static_cast<int64_t>(h) * ring * kD;
        const uint16_t* vres = static_cast<const uint16_t*>(sq.v_res) + static_cast<int64_t>(h) * ring * kD;
        float m[4], l[4], acc[4][kCpl];
        int64_t t1[4];
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
            m[hh] = -CUDART_INF_F;
            l[hh] = 0.0f;
#pragma unroll
            for (int c = 0; c < kCpl; ++c) acc[hh][c] = 0.0f;
            const int v = v0 + hh;
            t1[hh] = v < V ? L - nq + 1 + v / g : np;      // padding heads see nothing
        }
#pragma unroll 1
        for (int64_t ts = np; ts < L; ts += kTile) residual_tile_masked<DT>(kres, vres, ring, ts, t1, qs, lane, m, l, acc);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
            float* r = record(v0 + hh);
#pragma unroll
            for (int c = 0; c < kCpl; ++c) r[lane * kCpl + c] = acc[hh][c];
            if (lane == 0) {
                r[kD] = m[hh];
                r[kD + 1] = l[hh];
            }
        }
    } else {
        // ---- packed split: tiles [j0, j1) on the tensor cores
        const int64_t j0 = static_cast<int64_t>(split) * tps;
        const int64_t j1 = j0 + tps < ntiles ? j0 + tps : ntiles;
        const int n_my = static_cast<int>(j1 - j0);
        const int gid = lane >> 2, t = lane & 3;
        const int hh = gid >> 1, part = gid & 1;     // B column gid = (virtual head v0 + hh, hi/lo part)

        // q prescale of this warp: a power of two putting max |q| in (1/2, 1]
        float qmax_abs = 0.0f;
        for (int i = lane; i < 4 * kD; i += 32) qmax_abs = fmaxf(qmax_abs, fabsf(qs[i]));
        qmax_abs = warp_max(qmax_abs);
        int qexp = 0;
        if (qmax_abs > 0.0f) frexpf(qmax_abs, &qexp);
        const float qpre = ldexpf(1.0f, -qexp), qpost = ldexpf(1.0f, qexp);

        // key-side B constants: slot s = 2 ks + e holds k rows 2t + 8e, 2t + 8e + 1 of k-step ks
        uint32_t cY[16], cX[16], cZ[16], cB[16];
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            const int p0 = 16 * (s / 2) + 2 * t + 8 * (s % 2);
            const float q0 = qs[hh * kD + pos_channel<KB>(p0)] * qpre;
            const float q1 = qs[hh * kD + pos_channel<KB>(p0 + 1)] * qpre;
            const uint32_t qh = pack_h2(q0, q1);
            const uint32_t ql = pack_h2(q0 - h2_lo(qh), q1 - h2_hi(qh));
            cY[s] = qh;
            cX[s] = part ? ql : 0u;
            cZ[s] = part ? (qh ^ 0x80008000u) : 0u;
            cB[s] = part ? ql : qh;
        }

        // stream bases (see group_segment for the index arithmetic of either layout)
        const bool paged = seq_paged(sq);
        const int64_t hc = paged ? 0 : static_cast<int64_t>(h) * sq.cap_tokens;
        const unsigned char* kc_base = sq.k_codes + hc * RBK;
        const unsigned char* vc_base = sq.v_codes + hc * RBV;
        const unsigned char* ks_base = reinterpret_cast<const unsigned char*>(sq.k_scale + hc / G * kD);
        const unsigned char* kz_base = reinterpret_cast<const unsigned char*>(sq.k_zero + hc / G * kD);
        const unsigned char* vs_base = reinterpret_cast<const unsigned char*>(sq.v_scale + hc * NVG);
        const unsigned char* vz_base = reinterpret_cast<const unsigned char*>(sq.v_zero + hc * NVG);
        constexpr int CK = kTile * RBK / 16, CV = kTile * RBV / 16, CM = VMETA / 16;
        constexpr int CTOT = CK + CV + 32 + 2 * CM;            // 16-byte chunks of one stage
        auto issue = [&](int slot, int64_t j) {
            unsigned char* dst = stages + slot * Lay::kStage;
            int64_t rt, kg;
            if (paged) {
                kg = static_cast<int64_t>(sq.block_table[j / TPG]) * a.H + h;
                rt = kg * TPG + (TPG > 1 ? j % TPG : 0);
            } else {
                rt = j;
                kg = TPG > 1 ? j / TPG : j;
            }
#pragma unroll 1
            for (int c = tid; c < CTOT; c += NT) {
                const unsigned char* src;
                unsigned char* d;
                if (c < CK) {
                    src = kc_base + rt * (kTile * RBK) + 16 * c;
                    d = dst + 16 * c;
                } else if (c < CK + CV) {
                    src = vc_base + rt * (kTile * RBV) + 16 * (c - CK);
                    d = dst + kTile * RBK + 16 * (c - CK);
                } else if (c < CK + CV + 32) {
                    const int m = c - CK - CV;     // 0..15 scale, 16..31 zero
                    src = (m < 16 ? ks_base : kz_base) + kg * 256 + 16 * (m & 15);
                    d = dst + Lay::kKMeta + 256 * (m >> 4) + 16 * (m & 15);
                } else {
                    const int m = c - CK - CV - 32;     // 0..CM-1 scale, CM..2CM-1 zero
                    const int z = m >= CM, mm = z ? m - CM : m;
                    src = (z ? vz_base : vs_base) + rt * VMETA + 16 * mm;
                    d = dst + Lay::kVMeta + 256 * z + 16 * mm;
                }
                cp_async16(d, src);
            }
        };

        float m_run = -CUDART_INF_F, l_run = 0.0f;
        float cv[8][4], cz[4];
#pragma unroll
        for (int i = 0; i < 8; ++i) cv[i][0] = cv[i][1] = cv[i][2] = cv[i][3] = 0.0f;
        cz[0] = cz[1] = cz[2] = cz[3] = 0.0f;
        const uint32_t sel_z = (gid & 1) ? 0x7632u : 0x5410u;
        float* pt = pt_all + warp * 4 * kPtLd;

        // unpack stage `slot` into f16 buffer `buf` (keys, values) and its key scale / zero pairs
        auto unpack = [&](int slot, int buf) {
            const unsigned char* st = stages + slot * Lay::kStage;
            // ---- unpack the tile once: (row, 16-channel block) units of keys then values; a
            // thread's UPT units load their words first, then unpack and store. Unit u = tid +
            // k NT is a key unit for k < UPT / 2 and a value unit after (NT divides kTile * 8).
            // Unit uu of a side covers row r, block mblk with r = 4 (uu >> 5) + (uu >> 2 & 3),
            // mblk = (uu & 3) + 4 (uu >> 4 & 1): a warp's 32 loads hit 32 banks, and each
            // quarter-warp's 16-byte stores (rows r, r + 1 x four blocks) hit 8 bank groups.
            constexpr int UPT = 2 * kTile * 8 / NT, HALF = UPT / 2;
            auto unit_rm = [](int uu, int& r, int& mblk) {
                r = 4 * (uu >> 5) + ((uu >> 2) & 3);
                mblk = (uu & 3) + 4 * ((uu >> 4) & 1);
            };
            uint2 wd[UPT];
#pragma unroll
            for (int k = 0; k < UPT; ++k) {
                int r, mblk;
                unit_rm(tid + (k % HALF) * NT, r, mblk);
                const int bits = k < HALF ? KB : VB;
                const unsigned char* row = k < HALF ? st + r * RBK : st + kTile * RBK + r * RBV;
                wd[k] = bits == 2 ? make_uint2(*reinterpret_cast<const uint32_t*>(row + 4 * mblk), 0u)
                                  : *reinterpret_cast<const uint2*>(row + 8 * mblk);
            }
#pragma unroll
            for (int k = 0; k < UPT; ++k) {
                int r, mblk;
                unit_rm(tid + (k % HALF) * NT, r, mblk);
                uint32_t pr[8];
                auto unpack_word = [&]<int B>(uint2 w2) {
                    constexpr int SH = CodeShift<B>::kValue;
                    if constexpr (B == 2) {
                        const uint32_t w = w2.x, ws = w >> SH;
                        pr[0] = code_pair<2, 0>(w, ws); pr[1] = code_pair<2, 1>(w, ws);
                        pr[2] = code_pair<2, 2>(w, ws); pr[3] = code_pair<2, 3>(w, ws);
                        pr[4] = code_pair<2, 4>(w, ws); pr[5] = code_pair<2, 5>(w, ws);
                        pr[6] = code_pair<2, 6>(w, ws); pr[7] = code_pair<2, 7>(w, ws);
                    } else {
                        const uint32_t s0 = w2.x >> SH, s1 = w2.y >> SH;
                        pr[0] = code_pair<4, 0>(w2.x, s0); pr[1] = code_pair<4, 1>(w2.x, s0);
                        pr[2] = code_pair<4, 2>(w2.x, s0); pr[3] = code_pair<4, 3>(w2.x, s0);
                        pr[4] = code_pair<4, 0>(w2.y, s1); pr[5] = code_pair<4, 1>(w2.y, s1);
                        pr[6] = code_pair<4, 2>(w2.y, s1); pr[7] = code_pair<4, 3>(w2.y, s1);
                    }
                };
                if (k < HALF) unpack_word.template operator()<KB>(wd[k]);
                else unpack_word.template operator()<VB>(wd[k]);
                unsigned char* dst =
                    kf + buf * Lay::kF16Buf + (k < HALF ? 0 : kTile * kF16Pitch) + r * kF16Pitch + 32 * mblk;
                *reinterpret_cast<uint4*>(dst) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
                *reinterpret_cast<uint4*>(dst + 16) = make_uint4(pr[4], pr[5], pr[6], pr[7]);
            }
            // key scale / zero pairs in B-fragment order: perm[kind][ks][t][e] holds the
            // pair of positions 16 ks + 2t + 8e, + 1
#pragma unroll 1
            for (int u = tid; u < 2 * 8 * 4 * 2; u += NT) {
                const int e = u & 1, tt = (u >> 1) & 3, ks = (u >> 3) & 7, kind = u >> 6;
                const uint16_t* meta = reinterpret_cast<const uint16_t*>(st + Lay::kKMeta + 256 * kind);
                const int p0 = 16 * ks + 2 * tt + 8 * e;
                perm[buf * 128 + u] = static_cast<uint32_t>(meta[pos_channel<KB>(p0)]) |
                                      (static_cast<uint32_t>(meta[pos_channel<KB>(p0 + 1)]) << 16);
            }
        };

        // Pipeline, one barrier per tile: iteration it unpacks tile it + 1 into the other f16
        // buffer while the warps compute tile it; the barrier at its top makes tile it + 1's
        // stage visible, tile it's unpack visible, and frees the stage and buffer of it - 1.
#pragma unroll
        for (int i = 0; i < S - 1; ++i) {
            if (i < n_my) issue(i, j0 + i);
            cp_async_commit();
        }
        cp_async_wait<S - 2>();
        __syncthreads();
        unpack(0, 0);
        for (int it = 0; it < n_my; ++it) {
            cp_async_wait<S - 3>();
            __syncthreads();
            {
                const int nxt = it + S - 1;
                if (nxt < n_my) issue(nxt % S, j0 + nxt);
                cp_async_commit();
            }
            if (it + 1 < n_my) unpack((it + 1) % S, (it + 1) & 1);
            const unsigned char* st = stages + (it % S) * Lay::kStage;
            const unsigned char* kf_it = kf + (it & 1) * Lay::kF16Buf;
            const unsigned char* vf_it = kf_it + kTile * kF16Pitch;
            const uint32_t* perm_it = perm + (it & 1) * 128;
            const unsigned char* vsm = st + Lay::kVMeta;        // [32 tokens][NVG] fp16
            const unsigned char* vzm = vsm + 256;
            uint32_t sp[16], zp[16];
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint2 s2 = *reinterpret_cast<const uint2*>(perm_it + (ks * 4 + t) * 2);
                const uint2 z2 = *reinterpret_cast<const uint2*>(perm_it + 64 + (ks * 4 + t) * 2);
                sp[2 * ks] = s2.x; sp[2 * ks + 1] = s2.y;
                zp[2 * ks] = z2.x; zp[2 * ks + 1] = z2.y;
            }
            // ---- bias: every row of A is z_k, B = q (hi / lo column)
            float cb[4] = {0.0f, 0.0f, 0.0f, 0.0f}, cb2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int ks = 0; ks < 8; ks += 2) {
                mma_f16(cb, zp[2 * ks], zp[2 * ks], zp[2 * ks + 1], zp[2 * ks + 1], cB[2 * ks], cB[2 * ks + 1]);
                mma_f16(cb2, zp[2 * ks + 2], zp[2 * ks + 2], zp[2 * ks + 3], zp[2 * ks + 3], cB[2 * ks + 2],
                        cB[2 * ks + 3]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) cb[i] += cb2[i];
            // ---- scores: A = key codes (ldmatrix, rows = tokens), B = (q * s_k) hi / lo
            float c0[4] = {cb[0], cb[1], cb[2], cb[3]}, c1[4] = {cb[0], cb[1], cb[2], cb[3]};
            float c0o[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c1o[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const unsigned char* ka = kf_it + (lane & 15) * kF16Pitch + 16 * (lane >> 4);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int s0 = 2 * ks, s1 = 2 * ks + 1;
                const uint32_t b0 = hfma2(cX[s0], sp[s0], hfma2(cY[s0], sp[s0], hmul2(cZ[s0], sp[s0])));
                const uint32_t b1 = hfma2(cX[s1], sp[s1], hfma2(cY[s1], sp[s1], hmul2(cZ[s1], sp[s1])));
                uint32_t a0[4], a1[4];
                ldsm_x4(a0, ka + 32 * ks);
                ldsm_x4(a1, ka + 16 * kF16Pitch + 32 * ks);
                if (ks & 1) {
                    mma_f16(c0o, a0[0], a0[1], a0[2], a0[3], b0, b1);
                    mma_f16(c1o, a1[0], a1[1], a1[2], a1[3], b0, b1);
                } else {
                    mma_f16(c0, a0[0], a0[1], a0[2], a0[3], b0, b1);
                    mma_f16(c1, a1[0], a1[1], a1[2], a1[3], b0, b1);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                c0[i] += c0o[i];
                c1[i] += c1o[i];
            }
            // ---- online softmax for virtual head v0 + t over tokens gid, gid+8, gid+16, gid+24
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
            for (int r = 0; r < 4; ++r) p[r] = exp2f(S[r] - m_run);
            l_run += (p[0] + p[1]) + (p[2] + p[3]);
#pragma unroll
            for (int r = 0; r < 4; ++r) pt[t * kPtLd + gid + 8 * r] = p[r];
            __syncwarp();

            // ---- value side B operands: P' = p * s_v (hi / lo), and p (hi / lo) for the z_v term;
            // k rows 2t + 8e, + 1 of k-step kk are tokens 16 kk + 2t + 8e, + 1
            uint32_t vb[2][2][4], bp[2][2], za[2][2];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tau0 = 16 * kk + 2 * t + 8 * e;
                    const float2 pp = *reinterpret_cast<const float2*>(pt + hh * kPtLd + tau0);
                    const uint32_t ph = pack_h2(pp.x, pp.y);
                    const uint32_t pl = pack_h2(pp.x - h2_lo(ph), pp.y - h2_hi(ph));
                    const uint32_t xp = part ? pl : 0u, zn = part ? (ph ^ 0x80008000u) : 0u;
                    bp[kk][e] = part ? pl : ph;
                    uint32_t s0w[NVG / 2 > 0 ? NVG / 2 : 1], s1w[NVG / 2 > 0 ? NVG / 2 : 1];
                    if constexpr (NVG == 4) {
                        const uint2 x0 = *reinterpret_cast<const uint2*>(vsm + tau0 * 8);
                        const uint2 x1 = *reinterpret_cast<const uint2*>(vsm + (tau0 + 1) * 8);
                        s0w[0] = x0.x; s0w[1] = x0.y; s1w[0] = x1.x; s1w[1] = x1.y;
                    } else {
                        s0w[0] = *reinterpret_cast<const uint32_t*>(vsm + tau0 * 4);
                        s1w[0] = *reinterpret_cast<const uint32_t*>(vsm + (tau0 + 1) * 4);
                    }
#pragma unroll
                    for (int kg = 0; kg < 4; ++kg) {
                        const int vg = kg / TPG;
                        const uint32_t svp = prmt(s0w[vg >> 1], s1w[vg >> 1], (vg & 1) ? 0x7632u : 0x5410u);
                        vb[kk][e][kg] = hfma2(xp, svp, hfma2(ph, svp, hmul2(zn, svp)));
                    }
                    const uint32_t zw0 = *reinterpret_cast<const uint32_t*>(vzm + tau0 * (2 * NVG) + 4 * ((gid & 3) >> 1));
                    const uint32_t zw1 = *reinterpret_cast<const uint32_t*>(vzm + (tau0 + 1) * (2 * NVG) + 4 * ((gid & 3) >> 1));
                    za[kk][e] = gid < NVG ? prmt(zw0, zw1, sel_z) : 0u;
                }
            }
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) mma_f16(cz, za[kk][0], 0u, za[kk][1], 0u, bp[kk][0], bp[kk][1]);
            // ---- values: A = value codes^T (ldmatrix.trans: rows = positions, k = tokens)
            const unsigned char* va = vf_it + (8 * (lane >> 4) + (lane & 7)) * kF16Pitch + 16 * ((lane >> 3) & 1);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    uint32_t av[4];
                    ldsm_x4_t(av, va + 16 * kk * kF16Pitch + 32 * mt);
                    mma_f16(cv[mt], av[0], av[1], av[2], av[3], vb[kk][0][mt >> 1], vb[kk][1][mt >> 1]);
                }
            }
        }
        cp_async_wait<0>();

        // ---- this warp's record for each of its virtual heads (head v0 + t for the C columns)
        float l_tot = l_run;
        l_tot += __shfl_xor_sync(kFull, l_tot, 4);
        l_tot += __shfl_xor_sync(kFull, l_tot, 8);
        l_tot += __shfl_xor_sync(kFull, l_tot, 16);
        float zk[4];
        const float zmine = cz[0] + cz[1];     // (channel group gid, head t) for gid < NVG
#pragma unroll
        for (int kg = 0; kg < 4; ++kg) zk[kg] = __shfl_sync(kFull, zmine, 4 * (kg / TPG) + t);
        float* r = record(v0 + t);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int kg = mt >> 1;
            r[pos_channel<VB>(16 * mt + gid)] = cv[mt][0] + cv[mt][1] + zk[kg];
            r[pos_channel<VB>(16 * mt + gid + 8)] = cv[mt][2] + cv[mt][3] + zk[kg];
        }
        if (gid == 0) {
            r[kD] = m_run;
            r[kD + 1] = l_tot;
        }
    }

    // ---- the last CTA of (b, h) to finish merges the splits' records of every virtual head
    __threadfence();
    __syncthreads();
    if (tid == 0) s_misc[0] = atomicAdd(&a.counters[static_cast<int64_t>(b) * a.H + h], 1) == nsplit - 1;
    __syncthreads();
    if (!s_misc[0]) return;
    __threadfence();
    for (int i = tid; i < V * kD; i += NT) {
        const int v = i / kD, d = i - v * kD;
        float M = -CUDART_INF_F, den = 0.0f, num = 0.0f;
        for (int s = 0; s < nsplit; ++s) {
            const float* rec = a.partials + ((rec_base + s) * (4 * W) + v) * rec_stride;
            const float ms = __ldcg(rec + kD);
            if (ms == -CUDART_INF_F) continue;
            const float Mn = fmaxf(M, ms);
            const float fo = exp2f(M - Mn), fs = exp2f(ms - Mn);
            den = den * fo + __ldcg(rec + kD + 1) * fs;
            num = num * fo + __ldcg(rec + d) * fs;
            M = Mn;
        }
        out_row(v)[d] = num / den;
    }
    // every record of this (sequence, kv head), padding heads included, back to zero: each call
    // leaves the workspace as it found it (all zero), whatever plan the next call has
    __syncthreads();
    {
        float4* z = reinterpret_cast<float4*>(a.partials + rec_base * (4 * W) * rec_stride);
        const int64_t n4 = static_cast<int64_t>(nsplit) * (4 * W) * rec_stride / 4;
        for (int64_t i = tid; i < n4; i += NT) z[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    if (tid == 0) a.counters[static_cast<int64_t>(b) * a.H + h] = 0;
}

template <int KB, int VB, int DT, int W, int G>
cudaError_t launch_multi_w(const DecodeArgs& a, cudaStream_t stream) {
    constexpr int smem = MultiLayout<KB, VB, W>::kBytes;
    // the shared memory limit is raised once per device (an atomic flag per device; racing
    // first launches set the same value)
    static std::atomic<int> raised[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (raised[dev].load(std::memory_order_relaxed) == 0) {
        const cudaError_t e = cudaFuncSetAttribute(decode_multi_kernel<KB, VB, DT, W, G>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        raised[dev].store(1, std::memory_order_relaxed);
    }
    decode_multi_kernel<KB, VB, DT, W, G><<<dim3(a.max_splits, a.H, a.nseq), 32 * W, smem, stream>>>(a);
    return cudaGetLastError();
}

// Multi-query decode for one pair of code widths: dispatches the input type, G and the
// number of warps (ceil(V / 4), rounded up to 1, 2, 4 or 8).
template <int KB, int VB>
cudaError_t launch_multi_kv(const DecodeArgs& a, cudaStream_t stream) {
    if (a.nseq == 0) return cudaSuccess;
    const int V = (a.n_query > 0 ? a.n_query : 1) * (a.Hq / a.H);   // as multi_plan sized the records
    const int w = V <= 4 ? 1 : V <= 8 ? 2 : V <= 16 ? 4 : 8;
    auto by_g = [&]<int DT, int W>() {
        return a.G == 64 ? launch_multi_w<KB, VB, DT, W, 64>(a, stream) : launch_multi_w<KB, VB, DT, W, 32>(a, stream);
    };
    auto by_w = [&]<int DT>() {
        switch (w) {
            case 1: return by_g.template operator()<DT, 1>();
            case 2: return by_g.template operator()<DT, 2>();
            case 4: return by_g.template operator()<DT, 4>();
            default: return by_g.template operator()<DT, 8>();
        }
    };
    return a.dtype == KIVI_F16 ? by_w.template operator()<KIVI_F16>() : by_w.template operator()<KIVI_BF16>();
}

}  // namespace
}  // namespace kivi
