/*
 * gq_oracle.c -- plain, slow, single-threaded CPU oracle for block-quantized mul_mat.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may include, link or call this
 * file; only the tests, the package smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or constant with the CUDA library: the two meet only
 * in the seeded input generators.
 *
 * What it computes, and where the pages say so:
 *   - Q4_0 block layout: one fp16 scale (2 bytes) followed by 32 4-bit codes (16 bytes),
 *     i.e. 18 bytes per 32 weights ("Development Guide for Small AI Models (TinyLLaMA,
 *     etc.) Using C++", section 6.1).
 *   - Block quantization w_i ~= Delta * q_i with Delta = max_i |w_i| / 7 and 4-bit codes
 *     q_i in [-8, 7] ("A Complete Guide to llama.cpp and Customization with C++",
 *     section 2.2, the two displayed formulas for w_i and Delta). Stored codes carry an
 *     offset of +8 so that they fit an unsigned nibble.
 *   - Q8_0: the pages name 8-bit quantization ("No Python! Building an AI Inference
 *     Engine Exclusively in C++", section 9; "A Complete Guide ...", section 1.1) but lay
 *     out no 8-bit block. This oracle takes the 4-bit rule with signed 8-bit codes:
 *     Delta = max |w| / 127, code = round(w / Delta) in [-127, 127], same fp16 scale.
 *   - Dequantize right after the load, then multiply-accumulate with fp32 activations
 *     ("Development Guide ...", section 6.2, the load / unpack / dequantize / FMA flow;
 *     "No Python! ...", section 9).
 *   - The two adjacent steps of a transformer layer fused with the product: RMSNorm of
 *     the activations ahead of it ("Development Guide ...", section 4.1) and the SwiGLU
 *     of the gate and up projections after it (the same guide, section 4.4).
 *   - The product itself: C_ij = sum_k A_ik B_kj ("No Python! ...", section 6), realised
 *     as Y[n][m] = sum_k What[m][k] * X[n][k] -- the layout of the cuBLAS call in
 *     section 7.2 of the same article (W is M x K row-major, X is N x K row-major,
 *     Y is N x M row-major).
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - round() is C roundf: halves go away from zero.
 *   - the code is computed from the fp32 quotient w / d, with d = amax / 7 in fp32; the
 *     fp16 copy of d is what is stored and what dequantization uses.
 *   - an all-zero block stores d = +0 and the zero-point code (8 for Q4_0, 0 for Q8_0).
 *   - nibble order: byte j holds element j in its low nibble and element j + 16 in its
 *     high nibble.
 *   - fp32 -> fp16 is IEEE 754 round-to-nearest-even with subnormals kept and overflow to
 *     infinity, written here from the IEEE 754 binary16 definition.
 *   - accumulation is in fp64 in increasing k, rounded once to fp32 at the end.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (never -ffast-math: the
 * quantizer must be bit-exact IEEE division and rounding).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_TYPE_Q4_0 2
#define ORACLE_TYPE_Q8_0 8
#define ORACLE_TYPE_Q4_K 12

/* ---------------------------------------------------------------------------------- */
/* IEEE 754 binary32 -> binary16, round to nearest, ties to even.                      */
/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. Normal numbers   */
/* cover 2^-14 .. 65504, subnormals are m * 2^-24 for m in 1..1023.                    */
/* ---------------------------------------------------------------------------------- */
uint16_t oracle_fp16_from_f32(float f)
{
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    const uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    const uint32_t biased = (x >> 23) & 0xFFu;
    const uint32_t frac = x & 0x7FFFFFu;

    if (biased == 0xFFu) {                       /* infinity or NaN */
        if (frac == 0) return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | 0x7E00u | (frac >> 13));   /* quiet NaN */
    }
    if (biased == 0) return sign;                /* |f| < 2^-126: far below 2^-25 */

    const int e = (int)biased - 127;             /* f = sig * 2^(e - 23) */
    const uint32_t sig = frac | 0x800000u;       /* 24-bit significand */

    if (e > 15) return (uint16_t)(sign | 0x7C00u);           /* >= 2^16: overflow */

    if (e >= -14) {                              /* binary16 normal range */
        uint32_t h = sig >> 13;                  /* keep 11 bits */
        const uint32_t rest = sig & 0x1FFFu;     /* 13 dropped bits */
        if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u;
        uint32_t hexp = (uint32_t)(e + 15);
        if (h == 0x800u) { h = 0x400u; hexp += 1u; }         /* carry into exponent */
        if (hexp >= 31u) return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | (hexp << 10) | (h & 0x3FFu));
    }

    /* binary16 subnormal: value = m * 2^-24 with m = sig * 2^(e + 1) */
    const int drop = -(e + 1);                   /* >= 14 */
    if (drop > 24) return sign;                  /* below 2^-25: rounds to zero */
    uint32_t m = sig >> drop;
    const uint32_t rest = sig & ((1u << drop) - 1u);
    const uint32_t half = 1u << (drop - 1);
    if (rest > half || (rest == half && (m & 1u))) m += 1u;
    return (uint16_t)(sign | m);                 /* m == 1024 is the smallest normal */
}

float oracle_f32_from_fp16(uint16_t h)
{
    const int negative = (h & 0x8000u) != 0;
    const int biased = (h >> 10) & 0x1F;
    const int frac = h & 0x3FF;
    double v;
    if (biased == 0) {
        v = ldexp((double)frac, -24);
    } else if (biased == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), biased - 25);
    }
    return (float)(negative ? -v : v);
}

/* Element-wise loops over the two conversions, so that tests can sweep every pattern. */
void oracle_fp16_from_f32_array(const float* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp16_from_f32(x[i]);
}

void oracle_f32_from_fp16_array(const uint16_t* h, int64_t n, float* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_from_fp16(h[i]);
}

/* ---------------------------------------------------------------------------------- */
/* Quantization, one 32-element block at a time, blocks in row-major order.           */
/* ---------------------------------------------------------------------------------- */
static float block_absmax(const float* w)
{
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) {
        const float a = fabsf(w[i]);
        if (a > amax) amax = a;
    }
    return amax;
}

static void put_u16_le(uint8_t* p, uint16_t v)
{
    p[0] = (uint8_t)(v & 0xFFu);
    p[1] = (uint8_t)(v >> 8);
}

static uint16_t get_u16_le(const uint8_t* p)
{
    return (uint16_t)(p[0] | (p[1] << 8));
}

/* Q4_0 block: Delta = amax / 7, code = clamp(round(w / Delta) + 8, 0, 15). */
static void quantize_block_q4_0(const float* w, uint8_t* out)
{
    const float amax = block_absmax(w);
    const float d = amax / 7.0f;
    int code[32];
    for (int i = 0; i < 32; ++i) {
        if (d == 0.0f) {
            code[i] = 8;
        } else {
            int c = (int)roundf(w[i] / d) + 8;
            if (c < 0) c = 0;
            if (c > 15) c = 15;
            code[i] = c;
        }
    }
    put_u16_le(out, oracle_fp16_from_f32(d));
    for (int j = 0; j < 16; ++j)
        out[2 + j] = (uint8_t)(code[j] | (code[j + 16] << 4));
}

/* Q8_0 block: Delta = amax / 127, code = clamp(round(w / Delta), -127, 127). */
static void quantize_block_q8_0(const float* w, uint8_t* out)
{
    const float amax = block_absmax(w);
    const float d = amax / 127.0f;
    put_u16_le(out, oracle_fp16_from_f32(d));
    for (int i = 0; i < 32; ++i) {
        int c = 0;
        if (d != 0.0f) {
            c = (int)roundf(w[i] / d);
            if (c < -127) c = -127;
            if (c > 127) c = 127;
        }
        out[2 + i] = (uint8_t)(int8_t)c;
    }
}

/* ---------------------------------------------------------------------------------- */
/* Q4_K super-blocks. The pages name Q4_K as the 4-bit format behind TinyLLaMA's      */
/* "around 600 MB" ("Development Guide for Small AI Models (TinyLLaMA, etc.) Using    */
/* C++", section 6; "A Complete Guide to llama.cpp and Customization with C++",       */
/* section 2.2) but give no layout. This follows the published GGUF Q4_K block format:*/
/* 256 weights in 8 sub-blocks of 32, 144 bytes:                                       */
/*   bytes 0-1   d    (fp16): scale of the sub-block scales                            */
/*   bytes 2-3   dmin (fp16): scale of the sub-block mins                              */
/*   bytes 4-15  s[0..11]: eight 6-bit scales sc_j and eight 6-bit mins m_j:           */
/*               j < 4:  sc_j = s[j] & 63,  m_j = s[j + 4] & 63                         */
/*               j >= 4: sc_j = (s[j + 4] & 15) | (s[j - 4] >> 6) << 4,                 */
/*                       m_j  = (s[j + 4] >> 4) | (s[j] >> 6) << 4                      */
/*   bytes 16-143 codes: byte 16 + 32 g + l (g = 0..3, l = 0..31) holds weight         */
/*               64 g + l in its low nibble and weight 64 g + 32 + l in its high one  */
/*   What = d sc_j q - dmin m_j for weight with code q in sub-block j: both products  */
/*   are exact in fp32 (11 + 6 + 4 and 11 + 6 bits), one rounding at the subtraction. */
/* The quantizer is this oracle's reading (the format fixes only the dequantization): */
/* per sub-block lo = min(0, min w), hi = max w, step = (hi - lo) / 15, min = -lo;     */
/* d = max step / 63, dmin = max min / 63 (fp32, stored as fp16);                      */
/* sc_j = round(step_j / d), m_j = round(min_j / dmin) (fp32 quotients, halves away   */
/* from zero, clamped to [0, 63]; 0 where d or dmin is 0); codes                       */
/* round((w + M_j) / D_j) in [0, 15] against the dequantization's own                 */
/* D_j = fp16(d) sc_j and M_j = fp16(dmin) m_j (0 where D_j = 0).                     */
/* ---------------------------------------------------------------------------------- */
#define Q4K_WEIGHTS 256
#define Q4K_BYTES 144

static void q4k_get_scale_min(const uint8_t* s, int j, int* sc, int* m)
{
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

static void q4k_put_scale_min(uint8_t* s, const int* sc, const int* m)
{
    for (int j = 0; j < 12; ++j) s[j] = 0;
    for (int j = 0; j < 4; ++j) {
        s[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        s[j + 4] = (uint8_t)((m[j] & 63) | ((m[j + 4] >> 4) << 6));
        s[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
}

static void quantize_superblock_q4_k(const float* w, uint8_t* out)
{
    float step[8], mn[8];
    for (int j = 0; j < 8; ++j) {
        const float* v = w + 32 * j;
        float lo = v[0], hi = v[0];
        for (int i = 1; i < 32; ++i) {
            if (v[i] < lo) lo = v[i];
            if (v[i] > hi) hi = v[i];
        }
        if (lo > 0.0f) lo = 0.0f;
        step[j] = (hi - lo) / 15.0f;
        mn[j] = 0.0f - lo;
    }
    float smax = 0.0f, mmax = 0.0f;
    for (int j = 0; j < 8; ++j) {
        if (step[j] > smax) smax = step[j];
        if (mn[j] > mmax) mmax = mn[j];
    }
    const float d = smax / 63.0f;
    const float dmin = mmax / 63.0f;
    const uint16_t dh = oracle_fp16_from_f32(d);
    const uint16_t dminh = oracle_fp16_from_f32(dmin);
    int sc[8], m[8];
    for (int j = 0; j < 8; ++j) {
        int a = 0, b = 0;
        if (d != 0.0f) {
            a = (int)roundf(step[j] / d);
            if (a < 0) a = 0;
            if (a > 63) a = 63;
        }
        if (dmin != 0.0f) {
            b = (int)roundf(mn[j] / dmin);
            if (b < 0) b = 0;
            if (b > 63) b = 63;
        }
        sc[j] = a;
        m[j] = b;
    }
    put_u16_le(out, dh);
    put_u16_le(out + 2, dminh);
    q4k_put_scale_min(out + 4, sc, m);
    const float df = oracle_f32_from_fp16(dh), dminf = oracle_f32_from_fp16(dminh);
    int code[Q4K_WEIGHTS];
    for (int j = 0; j < 8; ++j) {
        const float D = df * (float)sc[j];
        const float M = dminf * (float)m[j];
        for (int i = 0; i < 32; ++i) {
            int q = 0;
            if (D != 0.0f) {
                q = (int)roundf((w[32 * j + i] + M) / D);
                if (q < 0) q = 0;
                if (q > 15) q = 15;
            }
            code[32 * j + i] = q;
        }
    }
    for (int g = 0; g < 4; ++g)
        for (int l = 0; l < 32; ++l)
            out[16 + 32 * g + l] = (uint8_t)(code[64 * g + l] | (code[64 * g + 32 + l] << 4));
}

static void dequantize_superblock_q4_k(const uint8_t* blk, float* w)
{
    const float d = oracle_f32_from_fp16(get_u16_le(blk));
    const float dmin = oracle_f32_from_fp16(get_u16_le(blk + 2));
    for (int j = 0; j < 8; ++j) {
        int sc, m;
        q4k_get_scale_min(blk + 4, j, &sc, &m);
        const float D = d * (float)sc;         /* exact */
        const float M = dmin * (float)m;       /* exact */
        const int g = j / 2, high = j % 2;
        for (int l = 0; l < 32; ++l) {
            const int byte = blk[16 + 32 * g + l];
            const int q = high ? (byte >> 4) : (byte & 15);
            w[32 * j + l] = D * (float)q - M;  /* D q exact; one rounding */
        }
    }
}

/* Bytes of one block: 18 (Q4_0) and 34 (Q8_0) per 32 weights; 144 (Q4_K) per 256. */
int64_t oracle_block_bytes(int type)
{
    if (type == ORACLE_TYPE_Q4_0) return 2 + 16;
    if (type == ORACLE_TYPE_Q8_0) return 2 + 32;
    if (type == ORACLE_TYPE_Q4_K) return Q4K_BYTES;
    return -1;
}

/* Weights per block: 32, or 256 for Q4_K. */
static int64_t block_weights(int type)
{
    return type == ORACLE_TYPE_Q4_K ? Q4K_WEIGHTS : 32;
}

/* Bytes of one row of K weights (K a multiple of the block's weights), else -1. */
int64_t oracle_row_bytes(int type, int64_t K)
{
    const int64_t bb = oracle_block_bytes(type);
    if (bb < 0 || K < 0 || K % block_weights(type) != 0) return -1;
    return K / block_weights(type) * bb;
}

/* W: M x K fp32 row-major, K a multiple of the block's weights. out: the blocks of each
   row, rows in order. */
int oracle_quantize(int type, const float* W, int64_t M, int64_t K, uint8_t* out)
{
    const int64_t bb = oracle_block_bytes(type);
    if (bb < 0 || M < 0 || oracle_row_bytes(type, K) < 0) return -1;
    const int64_t bw = block_weights(type);
    const int64_t nb = K / bw;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* w = W + m * K + b * bw;
            uint8_t* o = out + (m * nb + b) * bb;
            if (type == ORACLE_TYPE_Q4_0) quantize_block_q4_0(w, o);
            else if (type == ORACLE_TYPE_Q8_0) quantize_block_q8_0(w, o);
            else quantize_superblock_q4_k(w, o);
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------------- */
/* Dequantization: What = (code - 8) * Delta (Q4_0) or code * Delta (Q8_0).            */
/* Both products are exact in fp32 (at most 8 + 11 significant bits).                 */
/* ---------------------------------------------------------------------------------- */
static void dequantize_block(int type, const uint8_t* blk, float* w)
{
    if (type == ORACLE_TYPE_Q4_K) {
        dequantize_superblock_q4_k(blk, w);
        return;
    }
    const float d = oracle_f32_from_fp16(get_u16_le(blk));
    if (type == ORACLE_TYPE_Q4_0) {
        for (int j = 0; j < 16; ++j) {
            const int lo = blk[2 + j] & 0x0F;
            const int hi = blk[2 + j] >> 4;
            w[j] = (float)(lo - 8) * d;
            w[j + 16] = (float)(hi - 8) * d;
        }
    } else {
        for (int i = 0; i < 32; ++i)
            w[i] = (float)(int8_t)blk[2 + i] * d;
    }
}

/* One row of K weights (all its blocks) into w. */
static void dequantize_row(int type, const uint8_t* row, int64_t K, float* w)
{
    const int64_t bb = oracle_block_bytes(type), bw = block_weights(type);
    for (int64_t b = 0; b < K / bw; ++b) dequantize_block(type, row + b * bb, w + b * bw);
}

int oracle_dequantize(int type, const uint8_t* blocks, int64_t M, int64_t K, float* out)
{
    const int64_t rb = oracle_row_bytes(type, K);
    if (rb < 0 || M < 0) return -1;
    for (int64_t m = 0; m < M; ++m) dequantize_row(type, blocks + m * rb, K, out + m * K);
    return 0;
}

/* ---------------------------------------------------------------------------------- */
/* mul_mat: Y[n][m] = (float) sum_k (double) What[m][k] * (double) X[n][k].           */
/* Each product is exact in fp64; the sum runs over k in increasing order and is      */
/* rounded to fp32 once. `wrow` is caller-provided space for one dequantized row (K). */
/* ---------------------------------------------------------------------------------- */
int oracle_mul_mat(int type, const uint8_t* blocks, int64_t M, int64_t K,
                   const float* X, int64_t N, float* Y, float* wrow)
{
    const int64_t rb = oracle_row_bytes(type, K);
    if (rb < 0 || M < 0 || N < 0) return -1;
    for (int64_t m = 0; m < M; ++m) {
        dequantize_row(type, blocks + m * rb, K, wrow);
        for (int64_t n = 0; n < N; ++n) {
            const float* x = X + n * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)wrow[k] * (double)x[k];
            Y[n * M + m] = (float)acc;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------------- */
/* mul_mat with quantized activations ("A Complete Guide to llama.cpp and             */
/* Customization with C++", section 2.2, the last two displayed formulas): when x is  */
/* "similarly quantized", x_i ~= Delta_x * q_x,i, the block dot product becomes       */
/* Delta * Delta_x * sum_i q_i q_x,i with the sum a pure integer operation.           */
/* Reading (the pages give no x bit width or scale rule): every 32-element block of an */
/* activation row is quantized exactly like a Q8_0 weight block (Delta_x = fp16 of    */
/* max |x| / 127, codes round(x / Delta) in [-127, 127]). q_i is the signed weight    */
/* code: c - 8 (Q4_0) or c (Q8_0). Then                                               */
/*     Y[n][m] = (float) sum_b (double) Delta_w[m][b] * (double) Delta_x[n][b] * S_b, */
/* S_b = sum over the block of q_i * q_x,i (an exact integer), b in increasing order. */
/* `xq` is caller-provided space for the quantized X: N * K / 32 blocks of 34 bytes.  */
/* ---------------------------------------------------------------------------------- */
static int weight_code(int type, const uint8_t* blk, int i)
{
    if (type == ORACLE_TYPE_Q4_0) {
        const int byte = blk[2 + (i & 15)];
        return (i < 16 ? (byte & 0x0F) : (byte >> 4)) - 8;
    }
    return (int)(int8_t)blk[2 + i];
}

int oracle_mul_mat_q8x(int type, const uint8_t* blocks, int64_t M, int64_t K,
                       const float* X, int64_t N, float* Y, uint8_t* xq)
{
    const int64_t bb = oracle_block_bytes(type);
    if (type == ORACLE_TYPE_Q4_K) return -1;   /* defined for the 32-weight block types */
    if (bb < 0 || K % 32 != 0 || M < 0 || K < 0 || N < 0) return -1;
    const int64_t nb = K / 32;
    if (oracle_quantize(ORACLE_TYPE_Q8_0, X, N, K, xq) != 0) return -1;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t* wb = blocks + (m * nb + b) * bb;
                const uint8_t* xb = xq + (n * nb + b) * 34;
                int64_t sum = 0;
                for (int i = 0; i < 32; ++i)
                    sum += (int64_t)weight_code(type, wb, i) * (int64_t)(int8_t)xb[2 + i];
                const double dw = (double)oracle_f32_from_fp16(get_u16_le(wb));
                const double dx = (double)oracle_f32_from_fp16(get_u16_le(xb));
                acc += dw * dx * (double)sum;
            }
            Y[n * M + m] = (float)acc;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------------- */
/* mul_mat of the RMS-normalized activations ("Development Guide for Small AI Models   */
/* (TinyLLaMA, etc.) Using C++", section 4.1):                                          */
/*     RMSNorm(x) = x / sqrt((1/d) sum_i x_i^2 + eps) (.) gamma,   d = K,              */
/*     Y[n][m] = (float) sum_k (double) What[m][k] * xhat[n][k],                        */
/* with xhat computed in fp64 (sum of squares in increasing k, then the square root    */
/* and the division) and never rounded; one rounding at the end. `wrow` holds one      */
/* dequantized row (K floats); `xhat` is caller space for one normalized row (K).      */
/* ---------------------------------------------------------------------------------- */
int oracle_mul_mat_rmsnorm(int type, const uint8_t* blocks, int64_t M, int64_t K,
                           const float* X, const float* gamma, double eps, int64_t N,
                           float* Y, float* wrow, double* xhat)
{
    const int64_t rb = oracle_row_bytes(type, K);
    if (rb < 0 || M < 0 || K <= 0 || N < 0) return -1;
    for (int64_t n = 0; n < N; ++n) {
        const float* x = X + n * K;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) ss += (double)x[k] * (double)x[k];
        const double rms = sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; ++k) xhat[k] = (double)x[k] / rms * (double)gamma[k];
        for (int64_t m = 0; m < M; ++m) {
            dequantize_row(type, blocks + m * rb, K, wrow);
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += (double)wrow[k] * xhat[k];
            Y[n * M + m] = (float)acc;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------------- */
/* The gated feed-forward activation ("Development Guide ...", section 4.4):           */
/*     SwiGLU(x) = Swish(x W_gate) (x) (x W_up),   Swish(z) = z / (1 + e^-z),           */
/* in this library's layout H[n][m] = Swish(g) * u with g = sum_k Wgate_hat[m][k] x[k]  */
/* and u = sum_k Wup_hat[m][k] x[k], each an fp64 sum in increasing k; Swish and the    */
/* product in fp64, one rounding at the end. Both weights: M x K blocks of `type`.     */
/* `wrow` is caller space for two dequantized rows (2 K floats).                        */
/* ---------------------------------------------------------------------------------- */
int oracle_mul_mat_swiglu(int type, const uint8_t* gate, const uint8_t* up, int64_t M,
                          int64_t K, const float* X, int64_t N, float* H, float* wrow)
{
    const int64_t rb = oracle_row_bytes(type, K);
    if (rb < 0 || M < 0 || N < 0) return -1;
    float* wg = wrow;
    float* wu = wrow + K;
    for (int64_t m = 0; m < M; ++m) {
        dequantize_row(type, gate + m * rb, K, wg);
        dequantize_row(type, up + m * rb, K, wu);
        for (int64_t n = 0; n < N; ++n) {
            const float* x = X + n * K;
            double g = 0.0, u = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                g += (double)wg[k] * (double)x[k];
                u += (double)wu[k] * (double)x[k];
            }
            H[n * M + m] = (float)(g / (1.0 + exp(-g)) * u);
        }
    }
    return 0;
}
