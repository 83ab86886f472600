/*
 * qmv_oracle.c -- plain, slow, single-threaded CPU oracle for the weight-only
 * mixed-bit packed matvec with a fused residual-add + RMSNorm prologue.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this file's library.  The GPU library never links,
 * calls or includes it, and it includes nothing from the GPU library.
 *
 * Build: gcc -std=c99 -O2 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (no FMA contraction: every fp32 operation below is one IEEE-754 binary32
 * operation, rounded to nearest-even, in the order written).
 *
 * What it computes, and the passages it follows:
 *   - int2 codes, sixteen per 32-bit word, whose products with fp16
 *     activations are exact, accumulated in fp32 in code order
 *     ("Gemma4 raw-Metal loop on A19 -- findings + the remaining (parked)
 *     levers", section "What moved the needle", constant-memory byte-LUT item).
 *   - each output scalar's K-dot kept in one fixed accumulation order
 *     ("raw-metal-loop-playbook", prefill-regimes table, K-order-fixed row;
 *     and the A19 page, same section, tile/G retune item).
 *   - residual add + RMSNorm folded into the following matvec
 *     (A19 page, "What moved the needle", dispatch-count fusion item).
 *   - literal op sequences, no FMA contraction (A19 page, "Traps", fp16
 *     op-sequence item; playbook, closing mathMode note).
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - bit order: code k of a row sits in word floor(k*b/32), at bit offset
 *     b*(k mod (32/b)) (LSB first);
 *   - encoding: offset binary, field u = v + 2^(b-1) for a signed code v;
 *   - scales: fp16, one per group of `group` consecutive k of a row (group 32,
 *     or group == K for one scale per row);
 *   - block order: a group's dot is summed serially over k inside blocks of
 *     32 codes (the whole group when group <= 32); blocks are then added
 *     serially; the group's sum is multiplied by its scale (one rounding) and
 *     added to the row accumulator (a second rounding), groups in order;
 *   - RMSNorm: h = fp16(x + r); ss = sum of h*h, serial inside blocks of 32
 *     then serial over blocks; inv = 1 / sqrt(ss/K + eps);
 *     y = fp16((h * inv) * gamma), gamma used as-is.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_BLOCK 32

/* ---------------------------------------------------------------- fp16 --- */
/* IEEE-754 binary16 <-> binary32, written from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormals are
 * fraction * 2^-24; conversion to binary16 rounds to nearest, ties to even. */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

float orc_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu;
    uint32_t m = h & 0x3FFu;
    if (e == 0x1Fu)                      /* inf / nan: keep the payload */
        return bits_f32(sign | 0x7F800000u | (m << 13));
    if (e != 0)                          /* normal */
        return bits_f32(sign | ((e - 15u + 127u) << 23) | (m << 13));
    if (m == 0)
        return bits_f32(sign);
    /* subnormal: value m * 2^-24; m < 2^10 is exact in binary32 */
    {
        float v = (float)m * (1.0f / 16777216.0f);   /* exact power-of-two scale */
        return sign ? -v : v;
    }
}

uint16_t orc_f32_to_f16(float f)
{
    uint32_t x = f32_bits(f);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7FFFFFFFu;
    int e;
    if (ax >= 0x7F800000u) {             /* inf or nan */
        if (ax == 0x7F800000u) return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | 0x7E00u | ((ax >> 13) & 0x3FFu));
    }
    e = (int)(ax >> 23) - 127;           /* unbiased exponent */
    if (e > 15)
        return (uint16_t)(sign | 0x7C00u);   /* |f| >= 2^16: overflow */
    if (e >= -14) {                      /* lands in the normal binary16 range */
        uint32_t mant = ax & 0x7FFFFFu;
        uint32_t hv = ((uint32_t)(e + 15) << 10) | (mant >> 13);
        uint32_t rem = mant & 0x1FFFu;
        if (rem > 0x1000u || (rem == 0x1000u && (hv & 1u)))
            hv += 1;                     /* a carry may reach the exponent: correct, up to inf */
        return (uint16_t)(sign | hv);
    }
    if (e < -25)
        return sign;                     /* below half the smallest subnormal */
    {
        /* subnormal result m = round(|f| * 2^24); |f| = mant24 * 2^(e-23) */
        uint32_t mant = (ax & 0x7FFFFFu) | 0x800000u;
        int shift = -e - 1;              /* 14 .. 24 */
        uint32_t hv = mant >> shift;
        uint32_t rem = mant & ((1u << shift) - 1u);
        uint32_t halfway = 1u << (shift - 1);
        if (rem > halfway || (rem == halfway && (hv & 1u)))
            hv += 1;
        return (uint16_t)(sign | hv);
    }
}

void orc_f16_to_f32_array(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f32(in[i]);
}

void orc_f32_to_f16_array(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(in[i]);
}

/* -------------------------------------------------------- pack / decode --- */

static int bits_ok(int bits) { return bits == 2 || bits == 4 || bits == 8; }

/* signed codes [N][K] (int8) -> words [N][K*bits/32] (uint32).
 * Returns 0, or -1 on a bad width / shape, -2 on a code out of range. */
int orc_pack(const int8_t *codes, int64_t N, int64_t K, int bits, uint32_t *words)
{
    if (!bits_ok(bits) || N < 0 || K < 0 || (K * bits) % 32 != 0) return -1;
    {
        const int per_word = 32 / bits;
        const int bias = 1 << (bits - 1);
        const uint32_t mask = (1u << bits) - 1u;
        const int64_t wpr = K * bits / 32;
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t w = 0; w < wpr; ++w) words[n * wpr + w] = 0u;
            for (int64_t k = 0; k < K; ++k) {
                int v = codes[n * K + k];
                int u = v + bias;
                if (v < -bias || v >= bias) return -2;
                words[n * wpr + k / per_word] |=
                    ((uint32_t)u & mask) << (bits * (int)(k % per_word));
            }
        }
    }
    return 0;
}

/* words [N][K*bits/32] -> signed codes [N][K]; v = u - 2^(bits-1). */
int orc_unpack(const uint32_t *words, int64_t N, int64_t K, int bits, int8_t *codes)
{
    if (!bits_ok(bits) || N < 0 || K < 0 || (K * bits) % 32 != 0) return -1;
    {
        const int per_word = 32 / bits;
        const int bias = 1 << (bits - 1);
        const uint32_t mask = (1u << bits) - 1u;
        const int64_t wpr = K * bits / 32;
        for (int64_t n = 0; n < N; ++n)
            for (int64_t k = 0; k < K; ++k) {
                uint32_t w = words[n * wpr + k / per_word];
                uint32_t u = (w >> (bits * (int)(k % per_word))) & mask;
                codes[n * K + k] = (int8_t)((int)u - bias);
            }
    }
    return 0;
}

/* ---------------------------------------------------- residual + RMSNorm --- */

/* h_k = fp16(float(x_k) + float(r_k)) */
void orc_residual_add(const uint16_t *x, const uint16_t *r, int64_t K, uint16_t *h)
{
    for (int64_t k = 0; k < K; ++k) {
        float s = orc_f16_to_f32(x[k]) + orc_f16_to_f32(r[k]);
        h[k] = orc_f32_to_f16(s);
    }
}

/* Sum of squares of K fp16 values.  order 0: serial inside blocks of 32
 * consecutive k, then serial over the block sums (the library's order);
 * order 1: one serial chain over all k (used only by the self-tests). */
float orc_sumsq(const uint16_t *h, int64_t K, int order)
{
    if (order == 1) {
        float ss = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = orc_f16_to_f32(h[k]);
            float sq = v * v;                /* exact: 11-bit by 11-bit */
            ss = ss + sq;
        }
        return ss;
    } else {
        float ss = 0.0f;
        for (int64_t b0 = 0; b0 < K; b0 += ORC_BLOCK) {
            float blk = 0.0f;
            int64_t b1 = b0 + ORC_BLOCK < K ? b0 + ORC_BLOCK : K;
            for (int64_t k = b0; k < b1; ++k) {
                float v = orc_f16_to_f32(h[k]);
                float sq = v * v;
                blk = blk + sq;
            }
            ss = ss + blk;
        }
        return ss;
    }
}

/* inv = 1 / sqrt(ss / K + eps), each step one rounded fp32 operation */
float orc_rms_inv(float ss, int64_t K, float eps)
{
    float mean = ss / (float)K;
    float t = mean + eps;
    float rt = sqrtf(t);
    float inv = 1.0f / rt;
    return inv;
}

/* y_k = fp16((float(h_k) * inv) * float(gamma_k)) -- unfused form. */
void orc_rmsnorm(const uint16_t *h, const uint16_t *gamma, int64_t K, float eps,
                 int order, uint16_t *y)
{
    float inv = orc_rms_inv(orc_sumsq(h, K, order), K, eps);
    for (int64_t k = 0; k < K; ++k) {
        float a = orc_f16_to_f32(h[k]) * inv;
        float b = a * orc_f16_to_f32(gamma[k]);
        y[k] = orc_f32_to_f16(b);
    }
}

/* Fused form, written as one pass of its own (not by calling the unfused
 * functions) so that "fused equals unfused" is a real check: for each of
 * M columns (rows of the M x K inputs), h = fp16(x + r), the blocked sum of
 * squares accumulated while h is formed, then y.  h_out may be NULL. */
void orc_fused_residual_rmsnorm(const uint16_t *x, const uint16_t *r,
                                const uint16_t *gamma, int64_t M, int64_t K,
                                float eps, uint16_t *h_out, uint16_t *y)
{
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *xm = x + m * K, *rm = r + m * K;
        float ss = 0.0f, blk = 0.0f, mean, t, rt, inv;
        for (int64_t k = 0; k < K; ++k) {
            float s = orc_f16_to_f32(xm[k]) + orc_f16_to_f32(rm[k]);
            uint16_t hk = orc_f32_to_f16(s);
            float hv = orc_f16_to_f32(hk);
            float sq = hv * hv;
            if (h_out) h_out[m * K + k] = hk;
            blk = blk + sq;
            if ((k + 1) % ORC_BLOCK == 0 || k + 1 == K) {
                ss = ss + blk;
                blk = 0.0f;
            }
        }
        mean = ss / (float)K;
        t = mean + eps;
        rt = sqrtf(t);
        inv = 1.0f / rt;
        for (int64_t k = 0; k < K; ++k) {
            float s = orc_f16_to_f32(xm[k]) + orc_f16_to_f32(rm[k]);
            float hv = orc_f16_to_f32(orc_f32_to_f16(s));
            float a = hv * inv;
            float b = a * orc_f16_to_f32(gamma[k]);
            y[m * K + k] = orc_f32_to_f16(b);
        }
    }
}

/* ------------------------------------------------------------- matvec --- */

/* out[m][n] = sum over groups g of (sum over k in g of y[m][k] * v[n][k]) * s[n][g]
 *
 * codes : [N][K] signed codes (int8), the values v the packed words decode to
 * scales: [N][K/group] fp16 bits
 * y     : [M][K] fp16 bits (the activation of each of M columns)
 * out   : [M][N] fp32
 * group : divides K; a group longer than 32 must be a multiple of 32 and is
 *         summed in blocks of 32.
 * Returns 0, or -1 on a bad shape. */
int orc_gemv(const int8_t *codes, const uint16_t *scales, int64_t N, int64_t K,
             int64_t group, const uint16_t *y, int64_t M, float *out)
{
    if (N < 0 || K <= 0 || M < 0 || group <= 0 || K % group != 0) return -1;
    if (group > ORC_BLOCK && group % ORC_BLOCK != 0) return -1;
    {
        const int64_t G = K / group;
        for (int64_t m = 0; m < M; ++m) {
            const uint16_t *ym = y + m * K;
            for (int64_t n = 0; n < N; ++n) {
                const int8_t *vn = codes + n * K;
                float acc = 0.0f;
                for (int64_t g = 0; g < G; ++g) {
                    const int64_t g0 = g * group, g1 = (g + 1) * group;
                    float q = 0.0f;              /* the group's dot */
                    for (int64_t b0 = g0; b0 < g1; b0 += ORC_BLOCK) {
                        const int64_t b1 = b0 + ORC_BLOCK < g1 ? b0 + ORC_BLOCK : g1;
                        float p = 0.0f;          /* one block, serial in k */
                        for (int64_t k = b0; k < b1; ++k) {
                            float prod = orc_f16_to_f32(ym[k]) * (float)vn[k];  /* exact */
                            p = p + prod;
                        }
                        if (b0 == g0) q = p; else q = q + p;
                    }
                    {
                        float t = q * orc_f16_to_f32(scales[n * G + g]);   /* rounded */
                        acc = acc + t;                                     /* rounded */
                    }
                }
                out[m * N + n] = acc;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------- argmax --- */
/* The greedy token after the lm_head matvec ("Gemma4 raw-Metal loop on A19",
 * "The parked levers" table, argmax stage1+2 merge row: one dispatch that
 * keeps the first-max tie-break): the index of the largest y[n], the lowest
 * index among equal maxima.  Values compare as numbers (-0 equals +0); a NaN
 * is never the maximum.  *max_out (nullable) receives y at that index.
 * Returns the index, or -1 when N < 1 or every value is NaN. */
int64_t orc_argmax(const float *y, int64_t N, float *max_out)
{
    int64_t best = -1;
    for (int64_t n = 0; n < N; ++n) {
        if (y[n] != y[n]) continue;                 /* NaN */
        if (best < 0 || y[n] > y[best]) best = n;   /* strictly greater: first max wins */
    }
    if (max_out && best >= 0) *max_out = y[best];
    return best;
}
