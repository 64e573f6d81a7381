/*
 * NVFP4 oracle: a plain, slow, single-threaded CPU restatement of what the
 * NVFP4 quantize + block-scaled matmul path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library path links, loads or calls
 * this file; it exists so the CUDA kernels can be checked against an
 * independent implementation.  It shares no source with the CUDA code.
 *
 * Pages followed (cited by title and section):
 *  [P1] "Entrenamiento de Modelos de Lenguaje con 4 Bits de Precisión"
 *       (focoia.com.mx), sections "Características del Formato NVFP4" and
 *       "Metodología de Entrenamiento", and the closing feature list.
 *  [P2] "FP4 All the Way: Formación totalmente cuantificada de LLM"
 *       (slashpage digest of Chmiel, Fishman, Banner, Soudry), section
 *       "Describir" (the abstract).
 *  [P3] "I ricercatori di Nvidia sbloccano il tutorial LLM ..."
 *       (massacarraranews.com), section "Come funziona NVFP4?".
 *
 * What the pages fix: E2M1 elements with values ±0, ±0.5, ±1, ±1.5, ±2, ±3,
 * ±4, ±6 [P1 "Características"], one E4M3 scale per 16 contiguous elements
 * [P1 "Características"; P2 "Describir"], a multi-level scaling [P3 "Come
 * funziona NVFP4?"], 2-D block scaling for weights, random Hadamard transforms
 * and stochastic rounding of gradients [P1 "Metodología"], round-to-nearest in
 * the forward pass and stochastic rounding in backward/update [P2 "Describir"].
 * Everything the pages leave open is a stated reading (see the design notes);
 * each is marked "reading" below.
 *
 * Floating point: every value that decides an integer (a scale byte, a code)
 * is computed in IEEE binary32 with round-to-nearest-even, one operation at a
 * time, in the order written here.  Build with -ffp-contract=off and without
 * fast-math.  The matmul accumulates in binary64.
 *
 * Parity status per function: every function here is pinned by the CPU
 * tests -- e2m1/e4m3 codecs, tensor amaxes (plain and Hadamard), quantizers
 * (1x16, 2-D, RHT), stochastic
 * rounding, scale layout, GEMM, noise meter, MXFP4 quantizer and GEMM by
 * tables from the pages, closed forms, invariants, brute force and
 * hand-worked examples; philox4x32_10 by the known-answer vectors published
 * with the method (Salmon et al., SC'11); sr_values by hand-derived values of
 * one block from those vectors and a decision-independence test of the
 * elements that share a word; rht_signs by its word, bit range and counter.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>
#include <float.h>

#define OR_OK 0
#define OR_ERR_NONFINITE 4
#define OR_ERR_SHAPE 2

/* ------------------------------------------------------------------------ */
/* Element format: E2M1 [P1 "Características del Formato NVFP4"]            */
/* ------------------------------------------------------------------------ */

/* The eight magnitudes the page lists, indexed by the 3 low bits of a code.
 * Reading: code bits are s e1 e0 m (sign = bit 3), exponent bias 1, so the
 * magnitude codes 0..7 enumerate the listed values in increasing order. */
static const float E2M1_MAG[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float or_e2m1_value(int code)
{
    float m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* Round-to-nearest onto the E2M1 grid [P2 "Describir": nearest rounding in
 * the forward pass].  Reading: ties go to the code whose mantissa bit is 0
 * (round-half-even), magnitudes above 6 saturate to 6, and the sign bit is
 * kept even when the magnitude rounds to 0.  Written as a search for the
 * nearest of the eight magnitudes. */
int or_e2m1_rn(float v)
{
    int sign = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    if (a > 6.0)
        return sign | 7;
    int best = 0;
    for (int c = 1; c < 8; ++c) {
        double dc = fabs(a - (double)E2M1_MAG[c]);
        double db = fabs(a - (double)E2M1_MAG[best]);
        if (dc < db || (dc == db && (c & 1) == 0))
            best = c;
    }
    return sign | best;
}

/* Stochastic rounding onto the E2M1 grid [P1 "Metodología": stochastic
 * rounding on gradients; P2 "Describir": stochastic rounding in backward and
 * update].  Reading: with lo/hi the neighbouring grid magnitudes around
 * a = |v| and f = (a - lo) / (hi - lo) in [0, 1), the result is hi when
 * floor(f * 2^16) + R >= 2^16 for the 16-bit random value R (the fraction,
 * kept to 16 bits, plus R carries into the kept digit), else lo; so hi comes
 * with probability floor(f * 2^16) / 2^16.  |v| >= 6 gives 6; the sign is
 * kept.  f * 2^16 is computed exactly in binary64 (a has at most 24
 * significant bits and (hi - lo) is a power of two). */
int or_e2m1_sr(float v, unsigned R)
{
    int sign = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    if (!(a < 6.0))
        return sign | 7;
    int lo = 0;
    for (int c = 1; c < 8; ++c)
        if ((double)E2M1_MAG[c] <= a)
            lo = c;
    int hi = lo + 1;
    double gap = (double)E2M1_MAG[hi] - (double)E2M1_MAG[lo];
    double f16 = floor((a - (double)E2M1_MAG[lo]) / gap * 65536.0);
    return sign | ((f16 + (double)(R & 0xFFFFu) >= 65536.0) ? hi : lo);
}

/* ------------------------------------------------------------------------ */
/* Scale format: E4M3 [P1 "Características": one E4M3 factor per 16]        */
/* ------------------------------------------------------------------------ */

/* Reading: OCP E4M3 "FN" — 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 * subnormals at exponent 0, no infinities, S.1111.111 is NaN, largest finite
 * value 448. */
float or_e4m3_value(int code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    float v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexpf((float)m, -9);              /* m/8 * 2^(1-7) */
    else
        v = ldexpf((float)(8 + m), e - 10);    /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* Nearest finite E4M3 value with ties to the even code, for x >= 0 (the
 * block scale is never negative).  Values beyond 448 (including +inf)
 * saturate to 448; values at or below half the smallest subnormal round to 0.
 * Written as a search over all 127 non-negative finite codes. */
int or_e4m3_rn_sat(float x)
{
    double a = (double)x;
    if (a != a)
        return 0x7F;
    if (a < 0)
        a = 0; /* callers only pass non-negative values */
    if (isinf(a))
        return 0x7E;
    int best = 0;
    for (int c = 1; c <= 0x7E; ++c) {
        double dc = fabs(a - (double)or_e4m3_value(c));
        double db = fabs(a - (double)or_e4m3_value(best));
        if (dc < db || (dc == db && (c & 1) == 0))
            best = c;
    }
    return best;
}

/* ------------------------------------------------------------------------ */
/* Counter-based generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw,      */
/* "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11).  Ten rounds of    */
/* the 4x32 Philox S-box with the Weyl key schedule, as that paper defines.  */
/* ------------------------------------------------------------------------ */

static void philox_round(uint32_t c[4], const uint32_t k[2])
{
    const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c[1] ^ k[0];
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c[3] ^ k[1];
    uint32_t n3 = lo0;
    c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
}

void or_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k[0] += 0x9E3779B9u;
            k[1] += 0xBB67AE85u;
        }
        philox_round(c, k);
    }
    memcpy(out, c, sizeof c);
}

static unsigned rev8(unsigned x)
{
    unsigned y = 0;
    for (int i = 0; i < 8; ++i)
        if (x & (1u << i))
            y |= 1u << (7 - i);
    return y;
}

/* Random values of output block blk (reading): Philox with key = seed,
 * counter = (blk lo, blk hi, 0, 0) gives words w0..w3; elements 4m..4m+3 of
 * the block draw their 16-bit values from word m, bytes b0..b3 (least
 * significant first):
 *   element 4m     R = b2 * 256 + b0
 *   element 4m + 1 R = rev(b0) * 256 + rev(b2)
 *   element 4m + 2 R = b3 * 256 + b1
 *   element 4m + 3 R = rev(b1) * 256 + rev(b3)
 * with rev() reversing the 8 bits of a byte: each element sees 16 uniform
 * bits, and two elements share each half of the word (one of them in
 * bit-reversed order) -- the pairing the GB300 stochastic-rounding
 * conversion instruction uses for four elements and one 32-bit random word,
 * so that the kernels can round with that instruction. */
static void sr_values(uint64_t seed, uint64_t blk, unsigned R[16])
{
    uint32_t ctr[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), 0u, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    or_philox4x32_10(ctr, key, w);
    for (int m = 0; m < 4; ++m) {
        unsigned b0 = w[m] & 0xFFu, b1 = (w[m] >> 8) & 0xFFu, b2 = (w[m] >> 16) & 0xFFu, b3 = w[m] >> 24;
        R[4 * m + 0] = b2 * 256u + b0;
        R[4 * m + 1] = rev8(b0) * 256u + rev8(b2);
        R[4 * m + 2] = b3 * 256u + b1;
        R[4 * m + 3] = rev8(b1) * 256u + rev8(b3);
    }
}

/* ------------------------------------------------------------------------ */
/* Random Hadamard transform [P1 "Metodología": random Hadamard transforms]  */
/* ------------------------------------------------------------------------ */

/* Sign diagonal (reading): bit i of word 0 of Philox(key = seed,
 * counter = (0, 0, 1, 0)); a set bit flips lane i. */
uint32_t or_rht_signs(uint64_t rht_seed)
{
    uint32_t ctr[4] = {0u, 0u, 1u, 0u};
    uint32_t key[2] = {(uint32_t)rht_seed, (uint32_t)(rht_seed >> 32)};
    uint32_t w[4];
    or_philox4x32_10(ctr, key, w);
    return w[0] & 0xFFFFu;
}

/* y = (1/4) H16 D v with H16 the Sylvester Hadamard matrix of order 16.
 * Reading of the arithmetic: flip signs (exact), then the fast Walsh-Hadamard
 * butterflies with strides 1, 2, 4, 8 in that order, each pair (a, b) ->
 * (a + b, a - b) rounded to binary32, then multiply by 0.25. */
void or_rht16(const float v[16], uint32_t sign_bits, float y[16])
{
    float u[16];
    for (int i = 0; i < 16; ++i)
        u[i] = ((sign_bits >> i) & 1u) ? -v[i] : v[i];
    for (int h = 1; h < 16; h *= 2) {
        for (int i = 0; i < 16; ++i) {
            if (i & h)
                continue;
            float a = u[i], b = u[i + h];
            u[i] = a + b;
            u[i + h] = a - b;
        }
    }
    for (int i = 0; i < 16; ++i)
        y[i] = u[i] * 0.25f;
}

/* ------------------------------------------------------------------------ */
/* Scale-factor layout (reading): 128-row x 4-block atoms of 512 bytes, the  */
/* layout block-scaled tensor-core matmuls read scale factors in.            */
/* ------------------------------------------------------------------------ */

int64_t or_sf_groups(int64_t kblocks) { return (kblocks + 3) / 4; }

size_t or_sf_bytes(int64_t rows, int64_t cols)
{
    int64_t rt = (rows + 127) / 128;
    return (size_t)(rt * or_sf_groups(cols / 16) * 512);
}

size_t or_sf_offset(int64_t r, int64_t kb, int64_t kblocks)
{
    int64_t cp = or_sf_groups(kblocks);
    return (size_t)(((r / 128) * cp + kb / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (kb % 4));
}

/* ------------------------------------------------------------------------ */
/* Quantizers                                                               */
/* ------------------------------------------------------------------------ */

static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Second (tensor) level of the multi-level scaling [P3 "Come funziona
 * NVFP4?"]; binary32 per-tensor scale (reading): s_enc = 2688 / amax with
 * 2688 = 6 * 448 (largest E2M1 times largest E4M3), saturated to FLT_MAX; the
 * stored decode scale is g = amax / 2688.  amax == 0 gives g = 0. */
static void tensor_scales(float amax, float* s_enc, float* g)
{
    if (amax == 0.0f) {
        *s_enc = 0.0f;
        *g = 0.0f;
        return;
    }
    float s = 2688.0f / amax;
    if (isinf(s))
        s = FLT_MAX;
    *s_enc = s;
    *g = amax / 2688.0f;
}

/* First (block) level: the E4M3 scale of a block with maximum magnitude
 * bamax [P1 "Características"; P2 "Describir"].  Reading:
 * sb = e4m3(rn(rn(bamax / 6) * s_enc)). */
static int block_scale(float bamax, float s_enc)
{
    float t = bamax / 6.0f;
    float sbf = t * s_enc;
    return or_e4m3_rn_sat(sbf);
}

/* Quantize the 16 values of one block with scale byte sb (reading):
 * f = rn(s_enc / dec(sb)); v = rn(x * f) (zero stays signed zero; dec(sb) == 0
 * sends every element to signed zero); then RN or SR onto E2M1. */
static void quantize_block(const float x[16], float s_enc, int sb, int mode,
                           uint64_t seed, uint64_t blk, int codes[16])
{
    float d = or_e4m3_value(sb);
    float f = (d == 0.0f) ? 0.0f : s_enc / d;
    unsigned R[16] = {0};
    if (mode == 1)
        sr_values(seed, blk, R);
    for (int j = 0; j < 16; ++j) {
        float v;
        if (d == 0.0f || x[j] == 0.0f)
            v = signbit(x[j]) ? -0.0f : 0.0f;
        else
            v = x[j] * f;
        codes[j] = (mode == 1) ? or_e2m1_sr(v, R[j]) : or_e2m1_rn(v);
    }
}

static void put_code(uint8_t* q, int64_t row_bytes, int64_t r, int64_t c, int code)
{
    uint8_t* p = q + r * row_bytes + c / 2;
    if (c & 1)
        *p = (uint8_t)((*p & 0x0F) | (code << 4));
    else
        *p = (uint8_t)((*p & 0xF0) | code);
}

/* Tensor amax: max |x| over an R x C bf16 matrix (leading dimension ld), the
 * quantity the tensor scale is made from [P3 "Come funziona NVFP4?":
 * multi-level scaling].  A non-finite element is an error. */
int or_amax(const uint16_t* x, int64_t R, int64_t C, int64_t ld, float* amax_out)
{
    float amax = 0.0f;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            float a = fabsf(bf16_to_f32(x[r * ld + c]));
            if (!(a <= FLT_MAX))
                return OR_ERR_NONFINITE;
            if (a > amax)
                amax = a;
        }
    *amax_out = amax;
    return OR_OK;
}

/* Tensor amax of the Hadamard form: max |y| over y = (1/4) H16 D v for every
 * channel c and 16-token chunk v of x [T, C] [P1 "Metodología": random
 * Hadamard transforms; the tensor scale of the transformed operand uses the
 * transformed values].  T % 16 == 0; a non-finite y is an error. */
int or_rht_amax(const uint16_t* x, int64_t T, int64_t C, int64_t ld, uint64_t rht_seed, float* amax_out)
{
    if (T % 16 != 0 || T < 0 || C < 0)
        return OR_ERR_SHAPE;
    const uint32_t signs = or_rht_signs(rht_seed);
    float amax = 0.0f;
    for (int64_t c = 0; c < C; ++c)
        for (int64_t kb = 0; kb < T / 16; ++kb) {
            float v[16], y[16];
            for (int i = 0; i < 16; ++i)
                v[i] = bf16_to_f32(x[(kb * 16 + i) * ld + c]);
            or_rht16(v, signs, y);
            for (int i = 0; i < 16; ++i) {
                float a = fabsf(y[i]);
                if (!(a <= FLT_MAX))
                    return OR_ERR_NONFINITE;
                if (a > amax)
                    amax = a;
            }
        }
    *amax_out = amax;
    return OR_OK;
}

/* 1x16 quantization along rows (the contiguous axis) [P1 "Características":
 * each block of 16 contiguous elements shares an E4M3 scale].
 * x: bf16 bits, R x C with leading dimension ld.  Outputs: q (R x C/2 bytes,
 * element 2i in the low nibble), sf (swizzled, padding zero), *g.
 * mode 0 = round-to-nearest, 1 = stochastic (random byte per element). */
int or_quantize(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int mode, uint64_t seed,
                uint8_t* q, uint8_t* sf, float* g)
{
    if (C % 16 != 0 || R < 0 || C < 0)
        return OR_ERR_SHAPE;
    const int64_t KB = C / 16;
    float amax = 0.0f;
    int st = or_amax(x, R, C, ld, &amax);
    if (st != OR_OK)
        return st;
    float s_enc, gd;
    tensor_scales(amax, &s_enc, &gd);
    *g = gd;
    memset(sf, 0, or_sf_bytes(R, C));
    memset(q, 0, (size_t)(R * (C / 2)));
    for (int64_t r = 0; r < R; ++r)
        for (int64_t kb = 0; kb < KB; ++kb) {
            float xb[16];
            float bamax = 0.0f;
            for (int j = 0; j < 16; ++j) {
                xb[j] = bf16_to_f32(x[r * ld + kb * 16 + j]);
                if (fabsf(xb[j]) > bamax)
                    bamax = fabsf(xb[j]);
            }
            int sb = (amax == 0.0f) ? 0 : block_scale(bamax, s_enc);
            int codes[16];
            quantize_block(xb, s_enc, sb, mode, seed, (uint64_t)(r * KB + kb), codes);
            for (int j = 0; j < 16; ++j)
                put_code(q, C / 2, r, kb * 16 + j, codes[j]);
            sf[or_sf_offset(r, kb, KB)] = (uint8_t)sb;
        }
    return OR_OK;
}

/* 2-D block scaling for weights [P1 "Metodología": two-dimensional block
 * scaling for weights]; 16 x 16 tiles (reading).  One scale per tile, from the
 * tile's maximum magnitude, stored in every row's entry; elements are rounded
 * to nearest.  Optional transposed outputs: qT (C x R/2) is the exact
 * transpose of the codes and sfT gives tile (i, j)'s scale to tile (j, i). */
int or_quantize_2d(const uint16_t* w, int64_t R, int64_t C, int64_t ld,
                   uint8_t* q, uint8_t* sf, uint8_t* qT, uint8_t* sfT, float* g)
{
    if (C % 16 != 0 || R % 16 != 0 || R < 0 || C < 0)
        return OR_ERR_SHAPE;
    const int64_t KB = C / 16, KBT = R / 16;
    float amax = 0.0f;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            float a = fabsf(bf16_to_f32(w[r * ld + c]));
            if (!(a <= FLT_MAX))
                return OR_ERR_NONFINITE;
            if (a > amax)
                amax = a;
        }
    float s_enc, gd;
    tensor_scales(amax, &s_enc, &gd);
    *g = gd;
    memset(sf, 0, or_sf_bytes(R, C));
    memset(q, 0, (size_t)(R * (C / 2)));
    if (qT) memset(qT, 0, (size_t)(C * (R / 2)));
    if (sfT) memset(sfT, 0, or_sf_bytes(C, R));
    for (int64_t tr = 0; tr < R / 16; ++tr)
        for (int64_t tc = 0; tc < KB; ++tc) {
            float bamax = 0.0f;
            for (int i = 0; i < 16; ++i)
                for (int j = 0; j < 16; ++j) {
                    float a = fabsf(bf16_to_f32(w[(tr * 16 + i) * ld + tc * 16 + j]));
                    if (a > bamax)
                        bamax = a;
                }
            int sb = (amax == 0.0f) ? 0 : block_scale(bamax, s_enc);
            for (int i = 0; i < 16; ++i) {
                int64_t r = tr * 16 + i;
                float xb[16];
                for (int j = 0; j < 16; ++j)
                    xb[j] = bf16_to_f32(w[r * ld + tc * 16 + j]);
                int codes[16];
                quantize_block(xb, s_enc, sb, 0, 0, 0, codes);
                for (int j = 0; j < 16; ++j) {
                    put_code(q, C / 2, r, tc * 16 + j, codes[j]);
                    if (qT)
                        put_code(qT, R / 2, tc * 16 + j, r, codes[j]);
                }
                sf[or_sf_offset(r, tc, KB)] = (uint8_t)sb;
            }
            if (sfT)
                for (int j = 0; j < 16; ++j)
                    sfT[or_sf_offset(tc * 16 + j, tr, KBT)] = (uint8_t)sb;
        }
    return OR_OK;
}

/* Wgrad operand: random Hadamard transform along the token axis, then 1x16
 * quantization along that axis, written transposed [P1 "Metodología": random
 * Hadamard transforms, stochastic rounding on gradients].  Reading: for each
 * channel c and each 16-token chunk, y = (1/4) H16 D v with the seeded sign
 * diagonal D (the same for every chunk); the tensor scale uses the maximum
 * magnitude of the transformed values; the transformed binary32 values are
 * quantized as they are.  Output qT is C x T/2 (channel-major, tokens
 * contiguous), sfT is swizzled with C rows and T/16 blocks; the SR counter is
 * the block index in that output layout. */
int or_rht_quantize(const uint16_t* x, int64_t T, int64_t C, int64_t ld, uint64_t rht_seed,
                    int mode, uint64_t sr_seed, uint8_t* qT, uint8_t* sfT, float* g)
{
    if (T % 16 != 0 || T < 0 || C < 0)
        return OR_ERR_SHAPE;
    const int64_t KB = T / 16;
    const uint32_t signs = or_rht_signs(rht_seed);
    float amax = 0.0f;
    int st = or_rht_amax(x, T, C, ld, rht_seed, &amax);
    if (st != OR_OK)
        return st;
    float s_enc, gd;
    tensor_scales(amax, &s_enc, &gd);
    *g = gd;
    memset(sfT, 0, or_sf_bytes(C, T));
    memset(qT, 0, (size_t)(C * (T / 2)));
    for (int64_t c = 0; c < C; ++c)
        for (int64_t kb = 0; kb < KB; ++kb) {
            float v[16], y[16];
            for (int i = 0; i < 16; ++i)
                v[i] = bf16_to_f32(x[(kb * 16 + i) * ld + c]);
            or_rht16(v, signs, y);
            float bamax = 0.0f;
            for (int i = 0; i < 16; ++i)
                if (fabsf(y[i]) > bamax)
                    bamax = fabsf(y[i]);
            int sb = (amax == 0.0f) ? 0 : block_scale(bamax, s_enc);
            int codes[16];
            quantize_block(y, s_enc, sb, mode, sr_seed, (uint64_t)(c * KB + kb), codes);
            for (int i = 0; i < 16; ++i)
                put_code(qT, T / 2, c, kb * 16 + i, codes[i]);
            sfT[or_sf_offset(c, kb, KB)] = (uint8_t)sb;
        }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Dequantization and the block-scaled matmul [P1: NVFP4 runs on Blackwell  */
/* tensor cores]: value = e2m1(code) * e4m3(block scale) * g.               */
/* ------------------------------------------------------------------------ */

static double deq(const uint8_t* q, const uint8_t* sf, int64_t r, int64_t c, int64_t C)
{
    uint8_t byte = q[r * (C / 2) + c / 2];
    int code = (c & 1) ? (byte >> 4) : (byte & 15);
    double s = (double)or_e4m3_value(sf[or_sf_offset(r, c / 16, C / 16)]);
    return (double)or_e2m1_value(code) * s;
}

void or_dequantize(const uint8_t* q, const uint8_t* sf, float g, int64_t R, int64_t C, double* out)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            out[r * C + c] = deq(q, sf, r, c, C) * (double)g;
}

/* D[m][n] = gA gB sum_k deqA[m][k] deqB[n][k] with A (M x K) and B (N x K)
 * both stored K-contiguous; accumulated in binary64.  dabs receives
 * gA gB sum_k |deqA deqB| (for error bounds).  Either output may be NULL. */
void or_gemm_f64(const uint8_t* a, const uint8_t* sfa, float ga, const uint8_t* b,
                 const uint8_t* sfb, float gb, int64_t M, int64_t N, int64_t K,
                 double* d, double* dabs)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0, sa = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = deq(a, sfa, m, k, K) * deq(b, sfb, n, k, K);
                s += p;
                sa += fabs(p);
            }
            if (d) d[m * N + n] = (double)ga * (double)gb * s;
            if (dabs) dabs[m * N + n] = (double)ga * (double)gb * sa;
        }
}

/* The same matmul evaluated only at the listed (m, n) pairs. */
void or_gemm_f64_sampled(const uint8_t* a, const uint8_t* sfa, float ga, const uint8_t* b,
                         const uint8_t* sfb, float gb, int64_t M, int64_t N, int64_t K,
                         const int64_t* ms, const int64_t* ns, int64_t count,
                         double* d, double* dabs)
{
    (void)M; (void)N;
    for (int64_t i = 0; i < count; ++i) {
        double s = 0.0, sa = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = deq(a, sfa, ms[i], k, K) * deq(b, sfb, ns[i], k, K);
            s += p;
            sa += fabs(p);
        }
        d[i] = (double)ga * (double)gb * s;
        dabs[i] = (double)ga * (double)gb * sa;
    }
}

/* ------------------------------------------------------------------------ */
/* Quantization-noise meter [P2 "Describir": quantized training loses        */
/* efficiency once the gradient norm falls below about sqrt(3) times the     */
/* quantization noise].  Reading: the noise is the Euclidean norm of          */
/* Q(x) - x over the tensor, Q(x) the decoded NVFP4 value; the gradient norm  */
/* is the Euclidean norm of x.  sums[0] = sum (Q(x) - x)^2, sums[1] = sum x^2,*/
/* both in binary64 (Q(x) = code * scale * g is exact in binary64).          */
/* ------------------------------------------------------------------------ */

void or_quant_noise(const uint16_t* x, int64_t R, int64_t C, int64_t ld, const uint8_t* q,
                    const uint8_t* sf, float g, double sums[2])
{
    double se = 0.0, sx = 0.0;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
            double xv = (double)bf16_to_f32(x[r * ld + c]);
            double d = deq(q, sf, r, c, C) * (double)g - xv;
            se += d * d;
            sx += xv * xv;
        }
    sums[0] = se;
    sums[1] = sx;
}

/* ------------------------------------------------------------------------ */
/* MXFP4, the comparison format [P3 "Come funziona NVFP4?": MXFP4 needed     */
/* markedly more data for the same accuracy].  The pages do not define it;   */
/* this restates the OCP Microscaling (MX) v1.0 conversion: 32-element       */
/* blocks, E2M1 elements, one UE8M0 scale X = 2^e per block with             */
/* e = floor(log2(max|V|)) - emax(E2M1) = floor(log2(max|V|)) - 2, clamped   */
/* to the UE8M0 range; elements = E2M1 nearest-even of V / X, saturating.    */
/* Readings: a block max of 0 (or below the smallest normal binary32, whose  */
/* log2 floor lies under the range) takes e = -127; a block holding Inf/NaN  */
/* takes the UE8M0 NaN byte 0xFF with zero codes and the call reports        */
/* non-finite input.  Scale storage: one 32-bit word per row per 64          */
/* elements in the 128 x 4 atom layout, block scales in bytes 0 and 1.       */
/* ------------------------------------------------------------------------ */

double or_e8m0_value(int code)
{
    if (code == 255)
        return NAN;
    return ldexp(1.0, code - 127);
}

size_t or_mx_sf_offset(int64_t r, int64_t kb, int64_t kblocks)
{
    int64_t steps = (kblocks + 1) / 2; /* 64-element steps per row */
    return (size_t)(((r / 128) * steps + kb / 2) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 2);
}

int or_mx_quantize(const uint16_t* x, int64_t R, int64_t C, int64_t ld, uint8_t* q, uint8_t* sf)
{
    if (R <= 0 || C <= 0 || C % 32 != 0)
        return OR_ERR_SHAPE;
    int status = OR_OK;
    int64_t kblocks = C / 32;
    memset(sf, 0, or_sf_bytes(R, C));
    for (int64_t r = 0; r < R; ++r)
        for (int64_t kb = 0; kb < kblocks; ++kb) {
            double amax = 0.0;
            int finite = 1;
            for (int j = 0; j < 32; ++j) {
                float v = bf16_to_f32(x[r * ld + kb * 32 + j]);
                if (!isfinite(v))
                    finite = 0;
                else if (fabs((double)v) > amax)
                    amax = fabs((double)v);
            }
            size_t so = or_mx_sf_offset(r, kb, kblocks);
            if (!finite) {
                status = OR_ERR_NONFINITE;
                sf[so] = 0xFF;
                for (int j = 0; j < 32; ++j)
                    put_code(q, C / 2, r, kb * 32 + j, 0);
                continue;
            }
            int e = -127;
            if (amax >= (double)FLT_MIN) {
                int ex;
                frexp(amax, &ex); /* amax = m 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1 */
                e = (ex - 1) - 2;
                if (e < -127)
                    e = -127;
                if (e > 127)
                    e = 127;
            }
            sf[so] = (uint8_t)(e + 127);
            for (int j = 0; j < 32; ++j) {
                double v = (double)bf16_to_f32(x[r * ld + kb * 32 + j]);
                put_code(q, C / 2, r, kb * 32 + j, or_e2m1_rn((float)ldexp(v, -e)));
            }
        }
    return status;
}

static double mx_deq(const uint8_t* q, const uint8_t* sf, int64_t r, int64_t c, int64_t C)
{
    uint8_t byte = q[r * (C / 2) + c / 2];
    int code = (c & 1) ? (byte >> 4) : (byte & 15);
    return (double)or_e2m1_value(code) * or_e8m0_value(sf[or_mx_sf_offset(r, c / 32, C / 32)]);
}

void or_mx_dequantize(const uint8_t* q, const uint8_t* sf, int64_t R, int64_t C, double* out)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            out[r * C + c] = mx_deq(q, sf, r, c, C);
}

/* D[m][n] = sum_k deqA[m][k] deqB[n][k] (no tensor scale), binary64; dabs as
 * for or_gemm_f64.  Evaluated at the listed (m, n) pairs. */
void or_mx_gemm_f64_sampled(const uint8_t* a, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb,
                            int64_t K, const int64_t* ms, const int64_t* ns, int64_t count,
                            double* d, double* dabs)
{
    for (int64_t i = 0; i < count; ++i) {
        double s = 0.0, sa = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = mx_deq(a, sfa, ms[i], k, K) * mx_deq(b, sfb, ns[i], k, K);
            s += p;
            sa += fabs(p);
        }
        d[i] = s;
        dabs[i] = sa;
    }
}

/* Batch helpers so tests can sweep the element codecs without a Python loop. */
void or_e2m1_rn_many(const float* v, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint8_t)or_e2m1_rn(v[i]);
}

void or_e2m1_sr_many(const float* v, const uint16_t* R, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint8_t)or_e2m1_sr(v[i], R[i]);
}

/* The 16 random values of one block (for tests). */
void or_sr_values(uint64_t seed, uint64_t blk, uint32_t out[16])
{
    unsigned R[16];
    sr_values(seed, blk, R);
    for (int j = 0; j < 16; ++j)
        out[j] = R[j];
}

void or_e4m3_rn_sat_many(const float* v, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint8_t)or_e4m3_rn_sat(v[i]);
}
