/*
 * qmm_oracle.c -- plain, slow, CPU reference for the GGML block-quantized
 * linear layer (Q8_0, the K-quants Q2_K to Q6_K, FP8 E4M3).  TEST INFRASTRUCTURE ONLY: the tests, the
 * package's smoke check and the CPU-baseline leg of the benchmark call this
 * library; the product path never does.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Source of the method.  The mistral.rs documentation page "Quantization
 * types" names the two formats and their nominal widths: table "Q*K family"
 * (q4k, 4 bits) and table "Legacy GGML types" (q8_0, 8 bits); its section
 * "Numeric shorthands" maps `--isq 8` to Q8_0 and `--isq 4` to Q4K on CUDA.
 * The same page, in its opening section, defines ISQ as quantizing the
 * unquantized weights at load time.  The pages give no byte layout and no
 * quantizer formula; the ones written here are this library's stated reading:
 *
 *   Q8_0 block (32 weights, 34 bytes):
 *     amax = max |x_i|; d = amax / 127 (fp32 division); d16 = fp16_rne(d);
 *     q_i = clamp(roundf(x_i / float(d16)), -127, 127), or 0 when d16 == 0;
 *     bytes: d16 little-endian, then int8 q[0..31].
 *   Q4_K superblock (256 weights = 8 sub-blocks of 32, 144 bytes):
 *     mn_j = min(0, min_i x_i); mx_j = max_i x_i;
 *     s_j = (mx_j - mn_j) / 15;  m_j = 0 - mn_j;
 *     d16 = fp16_rne(max_j s_j / 63); dmin16 = fp16_rne(max_j m_j / 63);
 *     sc_j = clamp(roundf(s_j / d16), 0, 63)   (0 when d16 == 0);
 *     mc_j = clamp(roundf(m_j / dmin16), 0, 63) (0 when dmin16 == 0);
 *     S_j = d16 * sc_j; Mn_j = dmin16 * mc_j  (both exact in fp32);
 *     q_i = clamp(roundf((x_i + Mn_j) / S_j), 0, 15), or 0 when S_j == 0;
 *     dequantized value: S_j * q - Mn_j.
 *     bytes 0-1 d16, 2-3 dmin16, 4-15 the twelve scale bytes s[]:
 *       j<4: s[j]   = sc_j | (sc_{j+4} >> 4) << 6
 *            s[j+4] = mc_j | (mc_{j+4} >> 4) << 6
 *            s[j+8] = (sc_{j+4} & 15) | (mc_{j+4} & 15) << 4
 *     bytes 16-143: four 32-byte chunks c; byte 32c+l holds weight l of
 *       sub-block 2c in its low nibble and weight l of sub-block 2c+1 in its
 *       high nibble.
 *   Q6_K superblock (256 weights = 16 sub-blocks of 16, 210 bytes): the
 *     page's Q*K table lists q6k at 6 bits, and its "Numeric shorthands"
 *     table maps `--isq 6` to Q6K on CUDA; its "Sensitive tensor precision"
 *     section gives Q6K to the embeddings and output head of a Q4K model.
 *     The reading here (GGUF-shaped bytes, a plain symmetric quantizer):
 *     s_j = max_i |x_i| / 31;  d16 = fp16_rne(max_j s_j / 127);
 *     sc_j = clamp(roundf(s_j / d16), 0, 127)  (0 when d16 == 0);
 *     S_j = d16 * sc_j (exact);  c_i = clamp(roundf(x_i / S_j), -32, 31)
 *     (0 when S_j == 0);  dequantized value: S_j * c_i (exact in fp32).
 *     bytes 0-127 ql, 128-191 qh, 192-207 int8 sc[16], 208-209 d16; with
 *     q = c + 32 in 0..63 and weight w = 128h + 32s + l (h < 2, s < 4,
 *     l < 32): low 4 bits of q in byte 64h + 32(s & 1) + l of ql (low
 *     nibble for s < 2, high nibble for s >= 2), high 2 bits in bits 2s,
 *     2s + 1 of byte 32h + l of qh; weight w uses sc[w / 16].
 *   Q5_K, Q3_K, Q2_K (the page's Q*K table lists q5k, q3k, q2k at 5, 3
 *     and 2 bits; its "Numeric shorthands" table maps `--isq 5 / 3 / 2` to
 *     Q5K / Q3K / Q2K on CUDA).  Readings in the same plain style:
 *   Q5_K superblock (8 sub-blocks of 32, 176 bytes): Q4_K's quantizer with
 *     5-bit codes: s_j = (mx_j - mn_j) / 31, m_j = 0 - mn_j, d16 / dmin16 /
 *     sc_j / mc_j / S_j / Mn_j as for Q4_K, q_i = clamp(roundf((x_i + Mn_j) /
 *     S_j), 0, 31); value S_j * q - Mn_j.  Bytes 0-1 d16, 2-3 dmin16, 4-15
 *     the scale bytes (Q4_K's packing), 16-47 qh, 48-175 qs: byte 48+32c+l
 *     holds the low 4 bits of weight l of sub-block 2c (low nibble) and of
 *     sub-block 2c+1 (high nibble); bit j of qh byte 16+l is bit 4 of weight
 *     l of sub-block j.
 *   Q3_K superblock (16 sub-blocks of 16, 110 bytes), symmetric like Q6_K:
 *     s_j = max_i |x_i| / 3; d16 = fp16_rne(max_j s_j / 31); sc_j =
 *     clamp(roundf(s_j / d16), 0, 31) (0 when d16 == 0); S_j = d16 * sc_j;
 *     c_i = clamp(roundf(x_i / S_j), -4, 3) (0 when S_j == 0); value S_j * c_i
 *     (exact).  Bytes 0-31 hmask, 32-95 qs, 96-107 the sixteen 6-bit scale
 *     fields (each sc_j + 32), 108-109 d16.  With q = c + 4 in 0..7 and weight
 *     w = 128h + 32s + l (h < 2, s < 4, l < 32): bits 0-1 of q in bits 2s,
 *     2s+1 of qs byte 32h + l; bit 2 of q in bit 4h + s of hmask byte l.
 *     Scale field j: low 4 bits in scale byte j mod 8 (low nibble for j < 8,
 *     high nibble for j >= 8), high 2 bits in bits 2(j div 4), 2(j div 4)+1
 *     of scale byte 8 + j mod 4.
 *   Q2_K superblock (16 sub-blocks of 16, 84 bytes), affine like Q4_K:
 *     s_j = (mx_j - mn_j) / 3, m_j = 0 - mn_j; d16 = fp16_rne(max_j s_j / 15),
 *     dmin16 = fp16_rne(max_j m_j / 15); sc_j, mc_j = clamped roundf of
 *     s_j / d16, m_j / dmin16 in 0..15; q_i = clamp(roundf((x_i + Mn_j) /
 *     S_j), 0, 3); value S_j * q - Mn_j.  Bytes 0-15 the scales (byte j: sc_j
 *     in the low nibble, mc_j in the high one), 16-79 qs (weight w = 128h +
 *     32s + l in bits 2s, 2s+1 of byte 16 + 32h + l), 80-81 d16, 82-83 dmin16.
 *   FP8 E4M3 with a scale per row (W8A16): the page's section "FP8" says
 *     E4M3 FP8 can be produced with ISQ and lists symmetric E4M3 W8A16 with
 *     tensor, channel or block weight scales; the reading here is one fp32
 *     scale per output row (channel): s = max_k |x_k| / 448 (448 is E4M3's
 *     largest finite value); code = E4M3(x_k / s), round to nearest even,
 *     saturating at +-448 (all codes 0 when s == 0); dequantized value:
 *     float(E4M3 value) * s, one fp32 rounding.  A packed row is the K codes,
 *     then s (little-endian fp32), then 12 zero bytes: K + 16 bytes.
 *   gather (embedding lookup): out[t][:] = dequantized row ids[t] of the
 *     packed [V x D] table (Q8_0 is the page's common embedding target).
 *   matmul: Y[m][n] = sum_k double(w^[n][k]) * double(x[m][k]) over the exactly
 *     dequantized weights w^ and the bf16 activations, summed in k order in
 *     fp64; A[m][n] = sum_k |w^ x| in fp64 (the scale of the error bound).
 *
 * Build: plain C11, -O2 -ffp-contract=off (no fused multiply-add, IEEE single
 * arithmetic on x86-64 SSE), optionally -fopenmp (rows are independent, so the
 * thread count never changes a result).
 *
 * fp16 encoding is written here from the IEEE 754 binary16 definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits, subnormals,
 * round to nearest, ties to even); the tests pin it against two independent
 * library conversions.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* IEEE 754 binary16 and bfloat16                                      */
/* ------------------------------------------------------------------ */

/* binary16 -> float.  E == 0: subnormal F * 2^-24; E == 31: inf / NaN;
 * otherwise (1024 + F) * 2^(E - 25). */
float orc_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int E = (h >> 10) & 31;
    int F = h & 1023;
    double v;
    if (E == 0)
        v = ldexp((double)F, -24);
    else if (E == 31)
        v = F ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + F), E - 25);
    return (float)(sign ? -v : v);
}

/* float -> binary16, round to nearest, ties to even.
 * For finite |f| with binary exponent e = floor(log2 |f|), clamped below at
 * -14 (the subnormal range shares the exponent of the smallest normal), the
 * representable neighbours are integer multiples of the quantum 2^(e-10).
 * N = rint(|f| / 2^(e-10)) (exact scaling in double, rint rounds ties to
 * even) is the significand; the encoding of N * 2^(e-10) is then
 * (e + 14) * 1024 + N for every case: N < 1024 only happens for e == -14
 * (a subnormal, field E = 0), N == 2048 is a carry into the next binade.
 * A result of 2^16 or more (|f| >= 65520) is an overflow to infinity. */
uint16_t orc_f32_to_f16(float f)
{
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs((double)f);
    if (isnan(f))
        return (uint16_t)(sign | 0x7E00);
    if (a == 0.0)
        return sign;
    if (isinf(f) || a >= 65520.0)
        return (uint16_t)(sign | 0x7C00);
    int ex;
    frexp(a, &ex);          /* a = m * 2^ex, m in [0.5, 1) */
    int e = ex - 1;         /* a in [2^e, 2^(e+1)) */
    if (e < -14)
        e = -14;
    double N = rint(ldexp(a, 10 - e));
    long bits = (long)(e + 14) * 1024 + (long)N;
    return (uint16_t)(sign | (uint16_t)bits);
}

/* Element-wise versions of the two conversions above (for the tests). */
void orc_f32_to_f16_array(const float *x, uint16_t *h, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        h[i] = orc_f32_to_f16(x[i]);
}

void orc_f16_to_f32_array(const uint16_t *h, float *x, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        x[i] = orc_f16_to_f32(h[i]);
}

/* bfloat16 is the upper half of a binary32: widening is exact. */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static float load_src(int src_kind, const void *src, int64_t idx)
{
    if (src_kind == 0)
        return orc_bf16_to_f32(((const uint16_t *)src)[idx]);
    return ((const float *)src)[idx];
}

static float clampf(float v, float lo, float hi)
{
    if (v < lo)
        return lo;
    if (v > hi)
        return hi;
    return v;
}

static void put_u16(uint8_t *p, uint16_t v)
{
    p[0] = (uint8_t)(v & 0xFF);
    p[1] = (uint8_t)(v >> 8);
}

static uint16_t get_u16(const uint8_t *p)
{
    return (uint16_t)(p[0] | (p[1] << 8));
}

/* ------------------------------------------------------------------ */
/* Q8_0: 32 weights, fp16 scale d, int8 codes; 34 bytes                */
/* ------------------------------------------------------------------ */

enum { Q8_0_QK = 32, Q8_0_BYTES = 34, Q4_K_QK = 256, Q4_K_BYTES = 144 };

static void quantize_q8_0_block(const float *x, uint8_t *out)
{
    float amax = 0.0f;
    for (int i = 0; i < Q8_0_QK; i++) {
        float a = fabsf(x[i]);
        if (a > amax)
            amax = a;
    }
    float d = amax / 127.0f;
    uint16_t d16 = orc_f32_to_f16(d);
    float df = orc_f16_to_f32(d16);
    put_u16(out, d16);
    for (int i = 0; i < Q8_0_QK; i++) {
        float q = 0.0f;
        if (df != 0.0f)
            q = clampf(roundf(x[i] / df), -127.0f, 127.0f);
        out[2 + i] = (uint8_t)(int8_t)(int)q;
    }
}

static void dequantize_q8_0_block(const uint8_t *blk, float *y)
{
    float df = orc_f16_to_f32(get_u16(blk));
    for (int i = 0; i < Q8_0_QK; i++)
        y[i] = df * (float)(int8_t)blk[2 + i];
}

/* ------------------------------------------------------------------ */
/* Q4_K: 256-weight superblock, 8 sub-blocks of 32; 144 bytes          */
/* ------------------------------------------------------------------ */

/* Write the eight 6-bit scale codes and eight 6-bit min codes into the
 * twelve scale bytes (layout in the file header). */
static void pack_scales_q4_k(const int sc[8], const int mc[8], uint8_t s[12])
{
    for (int j = 0; j < 4; j++) {
        s[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        s[j + 4] = (uint8_t)((mc[j] & 63) | ((mc[j + 4] >> 4) << 6));
        s[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((mc[j + 4] & 15) << 4));
    }
}

static void unpack_scales_q4_k(const uint8_t s[12], int sc[8], int mc[8])
{
    for (int j = 0; j < 4; j++) {
        sc[j] = s[j] & 63;
        mc[j] = s[j + 4] & 63;
        sc[j + 4] = (s[j + 8] & 15) | ((s[j] >> 6) << 4);
        mc[j + 4] = (s[j + 8] >> 4) | ((s[j + 4] >> 6) << 4);
    }
}

static void quantize_q4_k_superblock(const float *x, uint8_t *out)
{
    float s[8], m[8];
    float smax = 0.0f, mmax = 0.0f;
    for (int j = 0; j < 8; j++) {
        const float *xs = x + 32 * j;
        float mx = xs[0];
        float mn = 0.0f; /* min(0, min_i x_i) */
        for (int i = 0; i < 32; i++) {
            if (xs[i] > mx)
                mx = xs[i];
            if (xs[i] < mn)
                mn = xs[i];
        }
        float range = mx - mn;
        s[j] = range / 15.0f;
        m[j] = 0.0f - mn;
        if (s[j] > smax)
            smax = s[j];
        if (m[j] > mmax)
            mmax = m[j];
    }
    uint16_t d16 = orc_f32_to_f16(smax / 63.0f);
    uint16_t dmin16 = orc_f32_to_f16(mmax / 63.0f);
    float df = orc_f16_to_f32(d16);
    float dminf = orc_f16_to_f32(dmin16);

    int sc[8], mc[8];
    for (int j = 0; j < 8; j++) {
        sc[j] = df > 0.0f ? (int)clampf(roundf(s[j] / df), 0.0f, 63.0f) : 0;
        mc[j] = dminf > 0.0f ? (int)clampf(roundf(m[j] / dminf), 0.0f, 63.0f) : 0;
    }

    put_u16(out, d16);
    put_u16(out + 2, dmin16);
    pack_scales_q4_k(sc, mc, out + 4);

    int q[256];
    for (int j = 0; j < 8; j++) {
        float S = df * (float)sc[j];
        float Mn = dminf * (float)mc[j];
        for (int i = 0; i < 32; i++) {
            float v = 0.0f;
            if (S > 0.0f) {
                float shifted = x[32 * j + i] + Mn;
                v = clampf(roundf(shifted / S), 0.0f, 15.0f);
            }
            q[32 * j + i] = (int)v;
        }
    }
    uint8_t *qs = out + 16;
    for (int c = 0; c < 4; c++)
        for (int l = 0; l < 32; l++)
            qs[32 * c + l] = (uint8_t)(q[32 * (2 * c) + l] | (q[32 * (2 * c + 1) + l] << 4));
}

static void dequantize_q4_k_superblock(const uint8_t *blk, float *y)
{
    float df = orc_f16_to_f32(get_u16(blk));
    float dminf = orc_f16_to_f32(get_u16(blk + 2));
    int sc[8], mc[8];
    unpack_scales_q4_k(blk + 4, sc, mc);
    const uint8_t *qs = blk + 16;
    for (int j = 0; j < 8; j++) {
        float S = df * (float)sc[j];
        float Mn = dminf * (float)mc[j];
        int c = j / 2;
        int hi = j % 2;
        for (int l = 0; l < 32; l++) {
            int q = hi ? (qs[32 * c + l] >> 4) : (qs[32 * c + l] & 15);
            float prod = S * (float)q;
            y[32 * j + l] = prod - Mn;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Q6_K: 256-weight superblock, 16 sub-blocks of 16; 210 bytes          */
/* ------------------------------------------------------------------ */

enum { Q6_K_QK = 256, Q6_K_BYTES = 210 };

/* Byte positions of the 6-bit code of weight w (0..255) of a superblock:
 * its low 4 bits in ql byte *lo_byte (high nibble when *lo_hi), its high 2
 * bits at bit *hi_shift of qh byte *hi_byte (offsets from the block start). */
static void q6_k_position(int w, int *lo_byte, int *lo_hi, int *hi_byte, int *hi_shift)
{
    int h = w / 128, s = (w / 32) % 4, l = w % 32;
    *lo_byte = 64 * h + 32 * (s & 1) + l;
    *lo_hi = s >= 2;
    *hi_byte = 128 + 32 * h + l;
    *hi_shift = 2 * s;
}

static void quantize_q6_k_superblock(const float *x, uint8_t *out)
{
    float s[16], smax = 0.0f;
    for (int j = 0; j < 16; j++) {
        float amax = 0.0f;
        for (int i = 0; i < 16; i++) {
            float a = fabsf(x[16 * j + i]);
            if (a > amax)
                amax = a;
        }
        s[j] = amax / 31.0f;
        if (s[j] > smax)
            smax = s[j];
    }
    uint16_t d16 = orc_f32_to_f16(smax / 127.0f);
    float df = orc_f16_to_f32(d16);
    memset(out, 0, Q6_K_BYTES);
    for (int j = 0; j < 16; j++) {
        int sc = df > 0.0f ? (int)clampf(roundf(s[j] / df), 0.0f, 127.0f) : 0;
        float S = df * (float)sc;
        out[192 + j] = (uint8_t)(int8_t)sc;
        for (int i = 0; i < 16; i++) {
            int w = 16 * j + i;
            int c = S > 0.0f ? (int)clampf(roundf(x[w] / S), -32.0f, 31.0f) : 0;
            int q = c + 32;
            int lo_byte, lo_hi, hi_byte, hi_shift;
            q6_k_position(w, &lo_byte, &lo_hi, &hi_byte, &hi_shift);
            out[lo_byte] |= (uint8_t)((q & 15) << (lo_hi ? 4 : 0));
            out[hi_byte] |= (uint8_t)((q >> 4) << hi_shift);
        }
    }
    put_u16(out + 208, d16);
}

static void dequantize_q6_k_superblock(const uint8_t *blk, float *y)
{
    float df = orc_f16_to_f32(get_u16(blk + 208));
    for (int w = 0; w < 256; w++) {
        int lo_byte, lo_hi, hi_byte, hi_shift;
        q6_k_position(w, &lo_byte, &lo_hi, &hi_byte, &hi_shift);
        int q = ((lo_hi ? blk[lo_byte] >> 4 : blk[lo_byte]) & 15) | (((blk[hi_byte] >> hi_shift) & 3) << 4);
        float S = df * (float)(int8_t)blk[192 + w / 16];
        y[w] = S * (float)(q - 32);
    }
}

/* ------------------------------------------------------------------ */
/* Q5_K: Q4_K with 5-bit codes; 176 bytes                              */
/* ------------------------------------------------------------------ */

enum { Q5_K_QK = 256, Q5_K_BYTES = 176, Q3_K_QK = 256, Q3_K_BYTES = 110, Q2_K_QK = 256, Q2_K_BYTES = 84 };

/* Per-sub-block range statistics of an affine K-quant: s_j = (max - min(0,
 * min)) / levels, m_j = 0 - min(0, min) over sub-blocks of `len` weights. */
static void affine_stats(const float *x, int nsub, int len, float levels, float *s, float *m, float *smax,
                         float *mmax)
{
    *smax = 0.0f;
    *mmax = 0.0f;
    for (int j = 0; j < nsub; j++) {
        const float *xs = x + len * j;
        float mx = xs[0], mn = 0.0f;
        for (int i = 0; i < len; i++) {
            if (xs[i] > mx)
                mx = xs[i];
            if (xs[i] < mn)
                mn = xs[i];
        }
        s[j] = (mx - mn) / levels;
        m[j] = 0.0f - mn;
        if (s[j] > *smax)
            *smax = s[j];
        if (m[j] > *mmax)
            *mmax = m[j];
    }
}

static void quantize_q5_k_superblock(const float *x, uint8_t *out)
{
    float s[8], m[8], smax, mmax;
    affine_stats(x, 8, 32, 31.0f, s, m, &smax, &mmax);
    uint16_t d16 = orc_f32_to_f16(smax / 63.0f);
    uint16_t dmin16 = orc_f32_to_f16(mmax / 63.0f);
    float df = orc_f16_to_f32(d16), dminf = orc_f16_to_f32(dmin16);
    int sc[8], mc[8];
    for (int j = 0; j < 8; j++) {
        sc[j] = df > 0.0f ? (int)clampf(roundf(s[j] / df), 0.0f, 63.0f) : 0;
        mc[j] = dminf > 0.0f ? (int)clampf(roundf(m[j] / dminf), 0.0f, 63.0f) : 0;
    }
    memset(out, 0, Q5_K_BYTES);
    put_u16(out, d16);
    put_u16(out + 2, dmin16);
    pack_scales_q4_k(sc, mc, out + 4);
    for (int j = 0; j < 8; j++) {
        float S = df * (float)sc[j];
        float Mn = dminf * (float)mc[j];
        for (int l = 0; l < 32; l++) {
            int q = 0;
            if (S > 0.0f)
                q = (int)clampf(roundf((x[32 * j + l] + Mn) / S), 0.0f, 31.0f);
            out[48 + 32 * (j / 2) + l] |= (uint8_t)((q & 15) << (4 * (j % 2)));
            out[16 + l] |= (uint8_t)((q >> 4) << j);
        }
    }
}

static void dequantize_q5_k_superblock(const uint8_t *blk, float *y)
{
    float df = orc_f16_to_f32(get_u16(blk));
    float dminf = orc_f16_to_f32(get_u16(blk + 2));
    int sc[8], mc[8];
    unpack_scales_q4_k(blk + 4, sc, mc);
    for (int j = 0; j < 8; j++) {
        float S = df * (float)sc[j];
        float Mn = dminf * (float)mc[j];
        for (int l = 0; l < 32; l++) {
            int q = ((blk[48 + 32 * (j / 2) + l] >> (4 * (j % 2))) & 15) | (((blk[16 + l] >> j) & 1) << 4);
            float prod = S * (float)q;
            y[32 * j + l] = prod - Mn;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Q3_K: 16 sub-blocks of 16, symmetric 3-bit codes; 110 bytes          */
/* ------------------------------------------------------------------ */

/* Scale field j (0..15) of Q3_K: returns the 6-bit field and writes it. */
static int q3_k_get_field(const uint8_t *sb, int j)
{
    int lo = (sb[j % 8] >> (j < 8 ? 0 : 4)) & 15;
    int hi = (sb[8 + j % 4] >> (2 * (j / 4))) & 3;
    return lo | (hi << 4);
}
static void q3_k_put_field(uint8_t *sb, int j, int v)
{
    sb[j % 8] |= (uint8_t)((v & 15) << (j < 8 ? 0 : 4));
    sb[8 + j % 4] |= (uint8_t)(((v >> 4) & 3) << (2 * (j / 4)));
}

/* Positions of the 3-bit code of weight w: bits 0-1 at bit *lo_shift of
 * byte *lo_byte (qs), bit 2 at bit *hi_bit of byte *hi_byte (hmask);
 * offsets from the block start. */
static void q3_k_position(int w, int *lo_byte, int *lo_shift, int *hi_byte, int *hi_bit)
{
    int h = w / 128, s = (w / 32) % 4, l = w % 32;
    *lo_byte = 32 + 32 * h + l;
    *lo_shift = 2 * s;
    *hi_byte = l;
    *hi_bit = 4 * h + s;
}

static void quantize_q3_k_superblock(const float *x, uint8_t *out)
{
    float s[16], smax = 0.0f;
    for (int j = 0; j < 16; j++) {
        float amax = 0.0f;
        for (int i = 0; i < 16; i++) {
            float a = fabsf(x[16 * j + i]);
            if (a > amax)
                amax = a;
        }
        s[j] = amax / 3.0f;
        if (s[j] > smax)
            smax = s[j];
    }
    uint16_t d16 = orc_f32_to_f16(smax / 31.0f);
    float df = orc_f16_to_f32(d16);
    memset(out, 0, Q3_K_BYTES);
    for (int j = 0; j < 16; j++) {
        int sc = df > 0.0f ? (int)clampf(roundf(s[j] / df), 0.0f, 31.0f) : 0;
        float S = df * (float)sc;
        q3_k_put_field(out + 96, j, sc + 32);
        for (int i = 0; i < 16; i++) {
            int w = 16 * j + i;
            int c = S > 0.0f ? (int)clampf(roundf(x[w] / S), -4.0f, 3.0f) : 0;
            int q = c + 4;
            int lo_byte, lo_shift, hi_byte, hi_bit;
            q3_k_position(w, &lo_byte, &lo_shift, &hi_byte, &hi_bit);
            out[lo_byte] |= (uint8_t)((q & 3) << lo_shift);
            out[hi_byte] |= (uint8_t)((q >> 2) << hi_bit);
        }
    }
    put_u16(out + 108, d16);
}

static void dequantize_q3_k_superblock(const uint8_t *blk, float *y)
{
    float df = orc_f16_to_f32(get_u16(blk + 108));
    for (int w = 0; w < 256; w++) {
        int lo_byte, lo_shift, hi_byte, hi_bit;
        q3_k_position(w, &lo_byte, &lo_shift, &hi_byte, &hi_bit);
        int q = ((blk[lo_byte] >> lo_shift) & 3) | (((blk[hi_byte] >> hi_bit) & 1) << 2);
        float S = df * (float)(q3_k_get_field(blk + 96, w / 16) - 32);
        y[w] = S * (float)(q - 4);
    }
}

/* ------------------------------------------------------------------ */
/* Q2_K: 16 sub-blocks of 16, affine 2-bit codes; 84 bytes              */
/* ------------------------------------------------------------------ */

static void quantize_q2_k_superblock(const float *x, uint8_t *out)
{
    float s[16], m[16], smax, mmax;
    affine_stats(x, 16, 16, 3.0f, s, m, &smax, &mmax);
    uint16_t d16 = orc_f32_to_f16(smax / 15.0f);
    uint16_t dmin16 = orc_f32_to_f16(mmax / 15.0f);
    float df = orc_f16_to_f32(d16), dminf = orc_f16_to_f32(dmin16);
    memset(out, 0, Q2_K_BYTES);
    for (int j = 0; j < 16; j++) {
        int sc = df > 0.0f ? (int)clampf(roundf(s[j] / df), 0.0f, 15.0f) : 0;
        int mc = dminf > 0.0f ? (int)clampf(roundf(m[j] / dminf), 0.0f, 15.0f) : 0;
        out[j] = (uint8_t)(sc | (mc << 4));
        float S = df * (float)sc;
        float Mn = dminf * (float)mc;
        for (int i = 0; i < 16; i++) {
            int w = 16 * j + i;
            int q = 0;
            if (S > 0.0f)
                q = (int)clampf(roundf((x[w] + Mn) / S), 0.0f, 3.0f);
            int h = w / 128, sh = (w / 32) % 4, l = w % 32;
            out[16 + 32 * h + l] |= (uint8_t)(q << (2 * sh));
        }
    }
    put_u16(out + 80, d16);
    put_u16(out + 82, dmin16);
}

static void dequantize_q2_k_superblock(const uint8_t *blk, float *y)
{
    float df = orc_f16_to_f32(get_u16(blk + 80));
    float dminf = orc_f16_to_f32(get_u16(blk + 82));
    for (int w = 0; w < 256; w++) {
        int j = w / 16, h = w / 128, sh = (w / 32) % 4, l = w % 32;
        float S = df * (float)(blk[j] & 15);
        float Mn = dminf * (float)(blk[j] >> 4);
        int q = (blk[16 + 32 * h + l] >> (2 * sh)) & 3;
        float prod = S * (float)q;
        y[w] = prod - Mn;
    }
}

/* ------------------------------------------------------------------ */
/* FP8 E4M3 (OCP 8-bit floating point, E4M3: 1 sign, 4 exponent bits with  */
/* bias 7, 3 fraction bits, no infinities, S.1111.111 is NaN)            */
/* ------------------------------------------------------------------ */

enum { FP8_ROW_PAD = 16 };

/* E4M3 -> float.  E == 0: subnormal F * 2^-9; (E, F) == (15, 7): NaN;
 * otherwise (8 + F) * 2^(E - 10). */
float orc_e4m3_to_f32(uint8_t b)
{
    int sign = b >> 7, E = (b >> 3) & 15, F = b & 7;
    double v;
    if (E == 0)
        v = ldexp((double)F, -9);
    else if (E == 15 && F == 7)
        v = NAN;
    else
        v = ldexp((double)(8 + F), E - 10);
    return (float)(sign ? -v : v);
}

/* float (finite) -> E4M3, round to nearest even, saturating at +-448.
 * With e = floor(log2 |f|) clamped below at -6 (subnormals share the
 * exponent of the smallest normal), the grid around |f| has quantum
 * 2^(e-3); N = rint(|f| / 2^(e-3)) (exact scaling in double, ties to
 * even), and N * 2^(e-3) is encoded after clamping to 448. */
uint8_t orc_f32_to_e4m3(float f)
{
    uint8_t sign = signbit(f) ? 0x80 : 0;
    double a = fabs((double)f);
    if (a == 0.0)
        return sign;
    int ex;
    frexp(a, &ex);
    int e = ex - 1;
    if (e < -6)
        e = -6;
    double v = ldexp(rint(ldexp(a, 3 - e)), e - 3);
    if (v > 448.0)
        v = 448.0;
    if (v == 0.0)
        return sign;
    frexp(v, &ex);
    e = ex - 1;
    if (e < -6)
        return (uint8_t)(sign | (int)ldexp(v, 9)); /* subnormal: v = F * 2^-9 */
    int frac = (int)ldexp(v, 3 - e) - 8;          /* v = (8 + F) * 2^(e - 3) */
    return (uint8_t)(sign | ((e + 7) << 3) | frac);
}

static void quantize_fp8_row(const float *x, int64_t K, uint8_t *out)
{
    float amax = 0.0f;
    for (int64_t k = 0; k < K; k++) {
        float a = fabsf(x[k]);
        if (a > amax)
            amax = a;
    }
    float s = amax / 448.0f;
    for (int64_t k = 0; k < K; k++)
        out[k] = s > 0.0f ? orc_f32_to_e4m3(x[k] / s) : 0;
    memcpy(out + K, &s, 4);
    memset(out + K + 4, 0, FP8_ROW_PAD - 4);
}

static void dequantize_fp8_row(const uint8_t *in, int64_t K, float *y)
{
    float s;
    memcpy(&s, in + K, 4);
    for (int64_t k = 0; k < K; k++)
        y[k] = orc_e4m3_to_f32(in[k]) * s;
}

void orc_f32_to_e4m3_array(const float *x, uint8_t *b, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        b[i] = orc_f32_to_e4m3(x[i]);
}

void orc_e4m3_to_f32_array(const uint8_t *b, float *x, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        x[i] = orc_e4m3_to_f32(b[i]);
}

/* ------------------------------------------------------------------ */
/* Exported API                                                        */
/* ------------------------------------------------------------------ */

enum { ORC_Q8_0 = 8, ORC_Q4_K = 4, ORC_Q6_K = 6, ORC_Q5_K = 5, ORC_Q3_K = 3, ORC_Q2_K = 2, ORC_FP8 = 80 };

static int qk_of(int fmt);
static int bytes_of(int fmt);

/* Bytes of one packed row of `cols` weights (0 if cols is not a whole
 * number of blocks). */
static int64_t row_bytes_of(int fmt, int64_t cols)
{
    if (fmt == ORC_FP8)
        return cols % 256 == 0 ? cols + FP8_ROW_PAD : 0;
    int qk = qk_of(fmt);
    if (qk == 0 || cols % qk != 0)
        return 0;
    return (cols / qk) * bytes_of(fmt);
}

static int qk_of(int fmt)
{
    switch (fmt) {
    case ORC_Q8_0: return Q8_0_QK;
    case ORC_Q4_K: return Q4_K_QK;
    case ORC_Q6_K: return Q6_K_QK;
    case ORC_Q5_K: return Q5_K_QK;
    case ORC_Q3_K: return Q3_K_QK;
    case ORC_Q2_K: return Q2_K_QK;
    default: return 0;
    }
}
static int bytes_of(int fmt)
{
    switch (fmt) {
    case ORC_Q8_0: return Q8_0_BYTES;
    case ORC_Q4_K: return Q4_K_BYTES;
    case ORC_Q6_K: return Q6_K_BYTES;
    case ORC_Q5_K: return Q5_K_BYTES;
    case ORC_Q3_K: return Q3_K_BYTES;
    case ORC_Q2_K: return Q2_K_BYTES;
    default: return 0;
    }
}

static void quantize_block(int fmt, const float *x, uint8_t *out)
{
    switch (fmt) {
    case ORC_Q8_0: quantize_q8_0_block(x, out); break;
    case ORC_Q4_K: quantize_q4_k_superblock(x, out); break;
    case ORC_Q6_K: quantize_q6_k_superblock(x, out); break;
    case ORC_Q5_K: quantize_q5_k_superblock(x, out); break;
    case ORC_Q3_K: quantize_q3_k_superblock(x, out); break;
    case ORC_Q2_K: quantize_q2_k_superblock(x, out); break;
    }
}

static void dequantize_block(int fmt, const uint8_t *blk, float *y)
{
    switch (fmt) {
    case ORC_Q8_0: dequantize_q8_0_block(blk, y); break;
    case ORC_Q4_K: dequantize_q4_k_superblock(blk, y); break;
    case ORC_Q6_K: dequantize_q6_k_superblock(blk, y); break;
    case ORC_Q5_K: dequantize_q5_k_superblock(blk, y); break;
    case ORC_Q3_K: dequantize_q3_k_superblock(blk, y); break;
    case ORC_Q2_K: dequantize_q2_k_superblock(blk, y); break;
    }
}

int64_t orc_packed_bytes(int fmt, int64_t rows, int64_t cols)
{
    if (rows < 0 || cols <= 0)
        return -1;
    int64_t rb = row_bytes_of(fmt, cols);
    return rb > 0 ? rows * rb : -1;
}

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* src_kind: 0 = bf16 (raw uint16 bits), 1 = fp32.  Returns 0 on success. */
int orc_quantize(int fmt, int src_kind, const void *src, uint8_t *dst, int64_t rows, int64_t cols)
{
    if (src_kind != 0 && src_kind != 1)
        return -1;
    if (fmt == ORC_FP8) {
        int64_t rb = row_bytes_of(fmt, cols);
        if (rb == 0)
            return -1;
        int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
        for (int64_t r = 0; r < rows; r++) {
            float *x = (float *)malloc((size_t)cols * sizeof(float));
            if (!x) {
                bad |= 1;
                continue;
            }
            for (int64_t k = 0; k < cols; k++)
                x[k] = load_src(src_kind, src, r * cols + k);
            quantize_fp8_row(x, cols, dst + r * rb);
            free(x);
        }
        return bad ? -2 : 0;
    }
    int qk = qk_of(fmt);
    if (qk == 0 || cols % qk != 0)
        return -1;
    int64_t nb = cols / qk;
    int64_t row_bytes = nb * bytes_of(fmt);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        float x[256];
        for (int64_t b = 0; b < nb; b++) {
            for (int i = 0; i < qk; i++)
                x[i] = load_src(src_kind, src, r * cols + b * qk + i);
            quantize_block(fmt, x, dst + r * row_bytes + b * bytes_of(fmt));
        }
    }
    return 0;
}

int orc_dequantize(int fmt, const uint8_t *src, float *dst, int64_t rows, int64_t cols)
{
    if (fmt == ORC_FP8) {
        int64_t rb = row_bytes_of(fmt, cols);
        if (rb == 0)
            return -1;
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; r++)
            dequantize_fp8_row(src + r * rb, cols, dst + r * cols);
        return 0;
    }
    int qk = qk_of(fmt);
    if (qk == 0 || cols % qk != 0)
        return -1;
    int64_t nb = cols / qk;
    int64_t row_bytes = nb * bytes_of(fmt);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < nb; b++) {
            dequantize_block(fmt, src + r * row_bytes + b * bytes_of(fmt), dst + r * cols + b * qk);
        }
    }
    return 0;
}

static void dequantize_row(int fmt, const uint8_t *src, float *dst, int64_t cols)
{
    if (fmt == ORC_FP8) {
        dequantize_fp8_row(src, cols, dst);
        return;
    }
    int qk = qk_of(fmt);
    for (int64_t b = 0; b < cols / qk; b++)
        dequantize_block(fmt, src + b * bytes_of(fmt), dst + b * qk);
}

/* Embedding lookup: out[t][0 .. D) = dequantized row ids[t] of the packed
 * table W[V x D].  Returns -1 (writing nothing) if an id is outside 0 .. V-1
 * or the shape is not a whole number of blocks. */
int orc_gather(int fmt, const uint8_t *W, int64_t V, int64_t D, const int64_t *ids, int64_t T,
               float *out)
{
    int64_t row_bytes = row_bytes_of(fmt, D);
    if (row_bytes == 0 || V < 0 || T < 0)
        return -1;
    for (int64_t t = 0; t < T; t++)
        if (ids[t] < 0 || ids[t] >= V)
            return -1;
    for (int64_t t = 0; t < T; t++)
        dequantize_row(fmt, W + ids[t] * row_bytes, out + t * D, D);
    return 0;
}

/* Y[m][t] and A[m][t] (row-major, M x count) for the output features n = ns[t]
 * of X[M x K] (bf16 bits) times the packed W[N x K]: one weight row is
 * dequantized exactly, then every activation row is dotted with it in k
 * order in fp64.  A may be NULL.  Returns 0 on success. */
int orc_matmul_columns(int fmt, const uint8_t *W, const uint16_t *X, int64_t M, int64_t K,
                       const int64_t *ns, int64_t count, double *Y, double *A)
{
    int64_t row_bytes = row_bytes_of(fmt, K);
    if (row_bytes == 0)
        return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : bad)
    for (int64_t t = 0; t < count; t++) {
        float *w = (float *)malloc((size_t)K * sizeof(float));
        if (!w) {
            bad |= 1;
            continue;
        }
        dequantize_row(fmt, W + ns[t] * row_bytes, w, K);
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0, aacc = 0.0;
            const uint16_t *xm = X + m * K;
            for (int64_t k = 0; k < K; k++) {
                double p = (double)w[k] * (double)orc_bf16_to_f32(xm[k]);
                acc += p;
                aacc += fabs(p);
            }
            Y[m * count + t] = acc;
            if (A)
                A[m * count + t] = aacc;
        }
        free(w);
    }
    return bad ? -2 : 0;
}

/* The full product: Y[M x N], A[M x N] in fp64 (A may be NULL). */
int orc_matmul(int fmt, const uint8_t *W, const uint16_t *X, double *Y, double *A,
               int64_t M, int64_t N, int64_t K)
{
    int64_t *ns = (int64_t *)malloc((size_t)(N > 0 ? N : 1) * sizeof(int64_t));
    if (!ns)
        return -2;
    for (int64_t n = 0; n < N; n++)
        ns[n] = n;
    int rc = orc_matmul_columns(fmt, W, X, M, K, ns, N, Y, A);
    free(ns);
    return rc;
}

/* Debug access to the code positions of Q6_K (used by the layout pins). */
void orc_q6_k_position(int w, int *pos4)
{
    q6_k_position(w, &pos4[0], &pos4[1], &pos4[2], &pos4[3]);
}

/* Debug access to the scale-byte packing of Q4_K (used by the layout pins). */
void orc_q4_k_pack_scales(const int *sc, const int *mc, uint8_t *s12) { pack_scales_q4_k(sc, mc, s12); }
void orc_q4_k_unpack_scales(const uint8_t *s12, int *sc, int *mc) { unpack_scales_q4_k(s12, sc, mc); }

/* Debug access to the code positions of Q3_K and its scale fields (layout pins). */
void orc_q3_k_position(int w, int *pos4)
{
    q3_k_position(w, &pos4[0], &pos4[1], &pos4[2], &pos4[3]);
}
int orc_q3_k_get_field(const uint8_t *sb12, int j) { return q3_k_get_field(sb12, j); }
