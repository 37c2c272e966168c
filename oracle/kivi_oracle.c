/*
 * KIVI oracle: a plain, slow CPU statement of what the KIVI hot path computes.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header or table with the CUDA
 * path: it has its own fp16/bf16 converters, its own packing and its own
 * attention.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC
 * (no contraction: every fp32 subtraction and division below is one IEEE
 * operation rounded to nearest-even, on x86-64 and on aarch64 alike).
 *
 * What it follows (page titles and sections):
 *  - "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache"
 *    (abstract): keys are quantized per channel, values per token, 2 bits.
 *  - "KIVI: Asymmetric 2-Bit KV Cache Quantization Guide", section "The Three
 *    Structural Innovations of KIVI" (items 1-3: per-channel keys grouped
 *    along tokens, per-token values grouped along channels, an fp16 FIFO
 *    window whose overflow is grouped and packed) and "Step 1"/"Step 2"
 *    (min/max asymmetric quantizer: scale = (max - min) / (2^bits - 1),
 *    round, clamp to [0, 2^bits - 1]; dequantize on the fly).
 *  - "KV cache quantization with KIVI INT2 setup guide 2026", section
 *    "KIVI: Per-Channel Key, Per-Token Value Quantization Explained"
 *    (G = 32, R = 128).
 *  - "KV-Cache Quantization: I Ran the Experiments So You Don't Have To",
 *    "Component 1" and "The memory math (verified)" (KV byte accounting).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - zero point is the fp16-rounded group minimum z, dequant = c*s + z
 *    (the guide's integer zero point is not used);
 *  - s and z are rounded to fp16 first, and codes are computed from the
 *    stored s and z widened to fp32: c = rint((x - z) / s), IEEE fp32
 *    subtraction and division, round-half-even, clamped to [0, qmax];
 *    s == 0 gives all codes 0;
 *  - codes are packed along channels inside one token row, lowest bits first:
 *    channel d sits in byte d*bits/8 at bit (d mod (8/bits))*bits;
 *  - keys: one group per (G consecutive tokens, channel), aligned to absolute
 *    position 0; values: one group per (token, G consecutive channels);
 *    G = 32 by default, 64 in the config example of "KV-Cache Quantization:
 *    I Ran the Experiments So You Don't Have To", section "Component 4"
 *    (which also sets R = 64 and separate key and value widths, k_bits and
 *    v_bits);
 *  - the residual ring has R+G slots and position p lives in slot p mod (R+G);
 *    a group is flushed when the residual reaches R+G tokens;
 *  - query head hq reads kv head hq / (Hq/Hkv); no mask; the decode query
 *    attends to every cached token.
 *
 * Parity pins (tests): converters against numpy/torch; planted-grid known
 * answers; brute-force nearest-grid on tiny inputs; the invariants of the
 * quantizer; attention against torch's scaled_dot_product_attention in fp64;
 * closed forms for the flush schedule and the byte accounting.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F16 0
#define ORC_BF16 1

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_CAPACITY 3

typedef struct {
    int32_t k_bits;      /* key code width: 2 or 4 */
    int32_t v_bits;      /* value code width: 2 or 4 */
    int32_t group;       /* G: tokens per key group, channels per value group */
    int32_t residual;    /* R: fp16 window length, a multiple of G */
    int32_t head_dim;    /* D: a multiple of G */
    int32_t num_q_heads; /* Hq */
    int32_t num_kv_heads;/* Hkv, divides Hq */
    int32_t dtype;       /* ORC_F16 or ORC_BF16: storage type of K, V, q */
} orc_cfg;

/* ------------------------------------------------------------------ */
/* Floating-point formats, written from the IEEE 754 binary16 and the   */
/* bfloat16 definitions (sign, biased exponent, fraction).              */
/* ------------------------------------------------------------------ */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* binary16 -> binary32, exact. */
float orc_f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t e = (h >> 10) & 0x1f;
    uint32_t m = h & 0x3ff;
    if (e == 0x1f) return bits_f32(sign | 0x7f800000u | (m << 13)); /* inf / nan */
    if (e == 0) {
        /* zero or subnormal: value = m * 2^-24, exact in binary32 */
        float v = (float)m * (1.0f / 16777216.0f);
        return sign ? -v : v;
    }
    return bits_f32(sign | ((e + 112u) << 23) | (m << 13));
}

/* binary32 -> binary16, round to nearest, ties to even. */
uint16_t orc_f32_to_f16(float f) {
    uint32_t x = f32_bits(f);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t a = x & 0x7fffffffu;
    uint32_t E = a >> 23;            /* biased binary32 exponent */
    uint32_t frac = a & 0x7fffffu;
    if (E == 0xff) {                 /* inf or nan */
        if (frac == 0) return sign | 0x7c00;
        return sign | 0x7e00 | (uint16_t)(frac >> 13);
    }
    if (E >= 143) return sign | 0x7c00; /* |f| >= 2^16: overflow */
    if (E >= 113) {
        /* normal binary16 range (before rounding): keep 10 fraction bits */
        uint32_t r = ((E - 112) << 10) | (frac >> 13);
        uint32_t rem = frac & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (r & 1u))) r += 1; /* may carry into inf */
        return sign | (uint16_t)r;
    }
    if (E < 102) return sign;        /* |f| < 2^-25: rounds to zero */
    {
        /* binary16 subnormal: value / 2^-24 = m_full * 2^(E - 150 + 24) */
        uint32_t m_full = frac | 0x800000u;
        uint32_t shift = 126 - E;    /* 14 .. 24 */
        uint32_t q = m_full >> shift;
        uint32_t rem = m_full & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        if (rem > half || (rem == half && (q & 1u))) q += 1;
        return sign | (uint16_t)q;
    }
}

/* bfloat16 -> binary32: the upper half of the binary32 pattern, exact. */
float orc_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)b << 16); }

void orc_f32_to_f16_array(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(in[i]);
}
void orc_f16_to_f32_array(const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f32(in[i]);
}

static float widen(uint16_t v, int dtype) {
    return dtype == ORC_BF16 ? orc_bf16_to_f32(v) : orc_f16_to_f32(v);
}

/* ------------------------------------------------------------------ */
/* The asymmetric min/max quantizer of one group                        */
/* ------------------------------------------------------------------ */

/*
 * Quantize n values x[0], x[stride], ... (already widened to fp32, exact).
 * Outputs the fp16 bit patterns of the scale s and zero z, and n codes.
 * Steps, in the order of the guide's "Step 1" (min, max, scale from the
 * range, round, clamp), with the zero point taken as the minimum itself:
 *   mn = min x, mx = max x                      (exact)
 *   s  = fp16( (mx - mn) / qmax )               (fp32 sub, fp32 div, RN)
 *   z  = fp16( mn )
 *   c  = clamp( rint( (x - z) / s ), 0, qmax )  (s, z widened back to fp32)
 *   s == 0  ->  c = 0
 */
static void quant_group(const float* x, int n, int stride, int qmax,
                        uint16_t* s_out, uint16_t* z_out, int* codes) {
    float mn = x[0], mx = x[0];
    for (int i = 1; i < n; ++i) {
        float v = x[(int64_t)i * stride];
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    float range = mx - mn;
    float s32 = range / (float)qmax;
    uint16_t s16 = orc_f32_to_f16(s32);
    uint16_t z16 = orc_f32_to_f16(mn);
    float s = orc_f16_to_f32(s16);
    float z = orc_f16_to_f32(z16);
    for (int i = 0; i < n; ++i) {
        int c = 0;
        if (s != 0.0f) {
            float num = x[(int64_t)i * stride] - z;
            float t = num / s;
            float r = rintf(t);
            if (r < 0.0f) r = 0.0f;
            if (r > (float)qmax) r = (float)qmax;
            c = (int)r;
        }
        codes[i] = c;
    }
    *s_out = s16;
    *z_out = z16;
}

/* Packing rule: channel d of a token row sits in byte d*bits/8 at bit offset
 * (d mod (8/bits))*bits, lowest bits first. */
static void put_code(uint8_t* row, int d, int bits, int c) {
    int per_byte = 8 / bits;
    int byte = d / per_byte;
    int shift = (d % per_byte) * bits;
    uint8_t mask = (uint8_t)(((1 << bits) - 1) << shift);
    row[byte] = (uint8_t)((row[byte] & ~mask) | ((c << shift) & mask));
}

static int get_code(const uint8_t* row, int d, int bits) {
    int per_byte = 8 / bits;
    return (row[d / per_byte] >> ((d % per_byte) * bits)) & ((1 << bits) - 1);
}

int orc_get_code(const uint8_t* row, int d, int bits) { return get_code(row, d, bits); }

/* ------------------------------------------------------------------ */
/* Codec entry points over raw [n_streams][n_tokens][D] tensors          */
/* ------------------------------------------------------------------ */

/*
 * Keys, per channel: for every stream, every group of G consecutive tokens
 * and every channel d, one (s, z) pair and G codes.
 *   x      [n_streams][n_tokens][D]        dtype bit patterns
 *   codes  [n_streams][n_tokens][D*k_bits/8] packed rows
 *   scale, zero [n_streams][n_tokens/G][D] fp16 bit patterns
 */
int orc_quant_keys(const orc_cfg* cfg, int n_streams, int n_tokens, const uint16_t* x,
                   uint8_t* codes, uint16_t* scale, uint16_t* zero) {
    const int D = cfg->head_dim, G = cfg->group, bits = cfg->k_bits;
    const int qmax = (1 << bits) - 1, row_bytes = D * bits / 8;
    if (n_tokens % G != 0) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int st = 0; st < n_streams; ++st) {
        float* col = (float*)malloc(sizeof(float) * G);
        int* c = (int*)malloc(sizeof(int) * G);
        for (int j = 0; j < n_tokens / G; ++j) {
            for (int d = 0; d < D; ++d) {
                for (int t = 0; t < G; ++t)
                    col[t] = widen(x[((int64_t)st * n_tokens + j * G + t) * D + d], cfg->dtype);
                int64_t m = ((int64_t)st * (n_tokens / G) + j) * D + d;
                quant_group(col, G, 1, qmax, &scale[m], &zero[m], c);
                for (int t = 0; t < G; ++t)
                    put_code(codes + ((int64_t)st * n_tokens + j * G + t) * row_bytes, d, bits, c[t]);
            }
        }
        free(col);
        free(c);
    }
    return ORC_OK;
}

/*
 * Values, per token: for every token and every group of G consecutive
 * channels, one (s, z) pair and G codes.
 *   codes  [n_streams][n_tokens][D*v_bits/8]
 *   scale, zero [n_streams][n_tokens][D/G]
 */
int orc_quant_values(const orc_cfg* cfg, int n_streams, int n_tokens, const uint16_t* x,
                     uint8_t* codes, uint16_t* scale, uint16_t* zero) {
    const int D = cfg->head_dim, G = cfg->group, bits = cfg->v_bits;
    const int qmax = (1 << bits) - 1, row_bytes = D * bits / 8;
#pragma omp parallel for schedule(static)
    for (int st = 0; st < n_streams; ++st) {
        float* row = (float*)malloc(sizeof(float) * D);
        int* c = (int*)malloc(sizeof(int) * G);
        for (int t = 0; t < n_tokens; ++t) {
            int64_t tok = (int64_t)st * n_tokens + t;
            for (int d = 0; d < D; ++d) row[d] = widen(x[tok * D + d], cfg->dtype);
            for (int k = 0; k < D / G; ++k) {
                int64_t m = tok * (D / G) + k;
                quant_group(row + k * G, G, 1, qmax, &scale[m], &zero[m], c);
                for (int i = 0; i < G; ++i) put_code(codes + tok * row_bytes, k * G + i, bits, c[i]);
            }
        }
        free(row);
        free(c);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* The cache of one sequence: packed history + fp16 residual ring        */
/* ------------------------------------------------------------------ */

/* Buffers of one sequence, laid out exactly as the library's:
 *   k_codes [Hkv][cap][D*k_bits/8], v_codes [Hkv][cap][D*v_bits/8]
 *   k_scale, k_zero   [Hkv][cap/G][D]
 *   v_scale, v_zero   [Hkv][cap][D/G]
 *   k_res, v_res      [Hkv][R+G][D]  (dtype bit patterns)                */
typedef struct {
    uint8_t* k_codes; uint16_t* k_scale; uint16_t* k_zero;
    uint8_t* v_codes; uint16_t* v_scale; uint16_t* v_zero;
    uint16_t* k_res; uint16_t* v_res;
    int32_t cap;
} orc_seq;

/* Number of packed tokens once the sequence holds L tokens: the residual
 * keeps between R and R+G-1 tokens once L >= R; everything older is packed
 * in whole groups. */
int64_t orc_n_packed(const orc_cfg* cfg, int64_t L) {
    int64_t over = L - cfg->residual;
    if (over <= 0) return 0;
    return (over / cfg->group) * cfg->group;
}

/* Pack group [n0, n0+G) of head h from the ring into the packed buffers. */
static void flush_group(const orc_cfg* cfg, const orc_seq* s, int h, int64_t n0) {
    const int D = cfg->head_dim, G = cfg->group, kb = cfg->k_bits, vb = cfg->v_bits, R = cfg->residual;
    const int kq = (1 << kb) - 1, vq = (1 << vb) - 1, ring = R + G;
    const int krow = D * kb / 8, vrow = D * vb / 8;
    const int64_t cap = s->cap;
    float* tile = (float*)malloc(sizeof(float) * G * D); /* [t][d] */
    float* kcol = (float*)malloc(sizeof(float) * G);
    int* c = (int*)malloc(sizeof(int) * G);
    for (int t = 0; t < G; ++t) {
        int64_t slot = (n0 + t) % ring;
        for (int d = 0; d < D; ++d)
            tile[t * D + d] = widen(s->k_res[((int64_t)h * ring + slot) * D + d], cfg->dtype);
    }
    /* keys: per channel over the G tokens */
    for (int d = 0; d < D; ++d) {
        for (int t = 0; t < G; ++t) kcol[t] = tile[t * D + d];
        int64_t m = ((int64_t)h * (cap / G) + n0 / G) * D + d;
        quant_group(kcol, G, 1, kq, &s->k_scale[m], &s->k_zero[m], c);
        for (int t = 0; t < G; ++t)
            put_code(s->k_codes + ((int64_t)h * cap + n0 + t) * krow, d, kb, c[t]);
    }
    /* values: per token over each group of G channels */
    for (int t = 0; t < G; ++t) {
        int64_t slot = (n0 + t) % ring;
        for (int d = 0; d < D; ++d)
            tile[t * D + d] = widen(s->v_res[((int64_t)h * ring + slot) * D + d], cfg->dtype);
        for (int k = 0; k < D / G; ++k) {
            int64_t m = ((int64_t)h * cap + n0 + t) * (D / G) + k;
            quant_group(tile + t * D + k * G, G, 1, vq, &s->v_scale[m], &s->v_zero[m], c);
            for (int i = 0; i < G; ++i)
                put_code(s->v_codes + ((int64_t)h * cap + n0 + t) * vrow, k * G + i, vb, c[i]);
        }
    }
    free(tile);
    free(kcol);
    free(c);
}

/*
 * Append n_new tokens to one sequence, one token at a time, the way the
 * guide's rolling-window cache manager does it, but flushing one whole group
 * of G tokens (the oldest) when the residual reaches R+G tokens.
 *   k_new, v_new [Hkv][n_new][D] dtype bit patterns
 * On capacity overflow (more than cap packed tokens would be needed) nothing
 * is changed and ORC_ERR_CAPACITY is returned.
 */
int orc_append(const orc_cfg* cfg, const orc_seq* s, int32_t* kv_len,
               const uint16_t* k_new, const uint16_t* v_new, int n_new) {
    const int D = cfg->head_dim, G = cfg->group, R = cfg->residual, H = cfg->num_kv_heads;
    const int ring = R + G;
    int64_t L = *kv_len;
    if (n_new < 0) return ORC_ERR_ARG;
    if (orc_n_packed(cfg, L + n_new) > s->cap) return ORC_ERR_CAPACITY;
    int64_t n_packed = orc_n_packed(cfg, L);
    for (int i = 0; i < n_new; ++i) {
        int64_t p = L + i;
        int64_t slot = p % ring;
        for (int h = 0; h < H; ++h) {
            memcpy(&s->k_res[((int64_t)h * ring + slot) * D], &k_new[((int64_t)h * n_new + i) * D], 2 * D);
            memcpy(&s->v_res[((int64_t)h * ring + slot) * D], &v_new[((int64_t)h * n_new + i) * D], 2 * D);
        }
        if (p + 1 - n_packed == R + G) {
            for (int h = 0; h < H; ++h) flush_group(cfg, s, h, n_packed);
            n_packed += G;
        }
    }
    *kv_len = (int32_t)(L + n_new);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Decode attention over the dequantized cache, fp64                     */
/* ------------------------------------------------------------------ */

/* Dequantized key and value of token p of head h, in fp64. Packed tokens:
 * k = c * s + z (exact in fp64); residual tokens: the stored value. */
static void token_kv(const orc_cfg* cfg, const orc_seq* s, int h, int64_t p, int64_t n_packed,
                     double* k, double* v) {
    const int D = cfg->head_dim, G = cfg->group, kb = cfg->k_bits, vb = cfg->v_bits, R = cfg->residual;
    const int ring = R + G;
    const int64_t cap = s->cap;
    if (p < n_packed) {
        const uint8_t* kr = s->k_codes + ((int64_t)h * cap + p) * (D * kb / 8);
        const uint8_t* vr = s->v_codes + ((int64_t)h * cap + p) * (D * vb / 8);
        for (int d = 0; d < D; ++d) {
            int64_t mk = ((int64_t)h * (cap / G) + p / G) * D + d;
            int64_t mv = ((int64_t)h * cap + p) * (D / G) + d / G;
            k[d] = (double)get_code(kr, d, kb) * (double)orc_f16_to_f32(s->k_scale[mk])
                 + (double)orc_f16_to_f32(s->k_zero[mk]);
            v[d] = (double)get_code(vr, d, vb) * (double)orc_f16_to_f32(s->v_scale[mv])
                 + (double)orc_f16_to_f32(s->v_zero[mv]);
        }
    } else {
        int64_t slot = p % ring;
        for (int d = 0; d < D; ++d) {
            k[d] = (double)widen(s->k_res[((int64_t)h * ring + slot) * D + d], cfg->dtype);
            v[d] = (double)widen(s->v_res[((int64_t)h * ring + slot) * D + d], cfg->dtype);
        }
    }
}

/*
 * Attention of one query over the first Lvis tokens of a sequence that holds
 * L >= Lvis tokens, for the query heads [hq0, hq0 + nhq):
 *   out[hq][d] = sum_{t < Lvis} softmax_t(scale * q.k_t) v_t[d]
 * Tokens are read as the cache holds them at length L (packed below
 * n_packed(L), residual above). Lvis == L is decode attention.
 *   q   [Hq][D] dtype bit patterns
 *   out [Hq][D] fp64 (rows outside [hq0, hq0+nhq) untouched)
 * Lvis == 0 gives zeros.
 */
static void attend_prefix(const orc_cfg* cfg, const orc_seq* s, int64_t L, int64_t Lvis, const uint16_t* q,
                          double scale, double* out, int hq0, int nhq) {
    const int D = cfg->head_dim, Hq = cfg->num_q_heads, H = cfg->num_kv_heads;
    const int g = Hq / H;
    const int64_t n_packed = orc_n_packed(cfg, L);
#pragma omp parallel for schedule(dynamic)
    for (int hq = hq0; hq < hq0 + nhq; ++hq) {
        int h = hq / g;
        double* qd = (double*)malloc(sizeof(double) * D);
        double* k = (double*)malloc(sizeof(double) * D);
        double* v = (double*)malloc(sizeof(double) * D);
        double* score = (double*)malloc(sizeof(double) * (Lvis > 0 ? Lvis : 1));
        for (int d = 0; d < D; ++d) qd[d] = (double)widen(q[(int64_t)hq * D + d], cfg->dtype);
        double m = -INFINITY;
        for (int64_t p = 0; p < Lvis; ++p) {
            token_kv(cfg, s, h, p, n_packed, k, v);
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qd[d] * k[d];
            score[p] = scale * acc;
            if (score[p] > m) m = score[p];
        }
        double denom = 0.0;
        for (int d = 0; d < D; ++d) out[(int64_t)hq * D + d] = 0.0;
        for (int64_t p = 0; p < Lvis; ++p) {
            token_kv(cfg, s, h, p, n_packed, k, v);
            double w = exp(score[p] - m);
            denom += w;
            for (int d = 0; d < D; ++d) out[(int64_t)hq * D + d] += w * v[d];
        }
        if (Lvis > 0)
            for (int d = 0; d < D; ++d) out[(int64_t)hq * D + d] /= denom;
        free(qd); free(k); free(v); free(score);
    }
}

/* Decode attention of one sequence holding L tokens: every query head attends to
 * all L tokens (no mask; the query is the newest token). */
void orc_decode_seq(const orc_cfg* cfg, const orc_seq* s, int64_t L, const uint16_t* q,
                    double scale, double* out, int hq0, int nhq) {
    attend_prefix(cfg, s, L, L, q, scale, out, hq0, nhq);
}

/*
 * Attention of the n_query newest tokens of one sequence holding L >= n_query
 * tokens (speculative verification, chunked prefill): query i sits at position
 * L - n_query + i and attends causally to positions [0, L - n_query + i].
 *   q   [n_query][Hq][D] dtype bit patterns
 *   out [n_query][Hq][D] fp64
 * Returns ORC_ERR_ARG when n_query < 1 or L < n_query.
 */
int orc_decode_multi_seq(const orc_cfg* cfg, const orc_seq* s, int64_t L, int n_query, const uint16_t* q,
                         double scale, double* out) {
    const int64_t row = (int64_t)cfg->num_q_heads * cfg->head_dim;
    if (n_query < 1 || L < n_query) return ORC_ERR_ARG;
    for (int i = 0; i < n_query; ++i)
        attend_prefix(cfg, s, L, L - n_query + 1 + i, q + i * row, scale, out + i * row, 0, cfg->num_q_heads);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Byte accounting                                                       */
/* ------------------------------------------------------------------ */

/* The plain KV-cache size of "The memory math (verified)": K and V, every
 * layer, kv head, channel and token, at `bits` per element, no metadata. */
double orc_kv_bytes_plain(int layers, int kv_heads, int head_dim, double bits, double seq, double batch) {
    return 2.0 * layers * kv_heads * head_dim * (bits / 8.0) * seq * batch;
}

/* Bytes of one sequence's buffers at capacity cap (packed tokens), in the
 * layout above: codes, fp16 scale and zero for keys (per group, per channel)
 * and values (per token, per channel group), and the R+G-slot residual ring. */
int64_t orc_seq_bytes(const orc_cfg* cfg, int64_t cap) {
    const int64_t D = cfg->head_dim, G = cfg->group, H = cfg->num_kv_heads;
    const int64_t codes = cap * D * (cfg->k_bits + cfg->v_bits) / 8;
    const int64_t kmeta = 2 * (cap / G) * D * 2;
    const int64_t vmeta = 2 * cap * (D / G) * 2;
    const int64_t ring = (cfg->residual + G) * D * 2;
    return H * (codes + kmeta + vmeta + 2 * ring);
}
