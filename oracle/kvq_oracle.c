/*
 * kvq_oracle.c -- plain, slow CPU oracle for attention over a block-quantized
 * KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; it shares no code, header, table or constant generator
 * with the CUDA path.  Only the tests, the smoke check and the benchmark's CPU
 * baseline use it.
 *
 * What it computes, and where each piece comes from:
 *
 *  - Block codecs f16 / q8_0 / q4_0 ("Codecs" table of the buun-llama-cpp
 *    listing: f16 16.0, q8_0 8.5 and q4_0 4.5 bits per value, i.e. 32-value
 *    blocks of a 2-byte fp16 scale plus 32 int8 or 16 packed nibble bytes).
 *    The encoders are the written fp32 formulas this library defines:
 *      q8_0: amax = max|x|; d = amax / 127 (fp32 RN division);
 *            q = round-half-away-from-zero(x / d) (fp32 RN division), 0 if d == 0;
 *            stored d16 = fp16_RN(d).
 *      q4_0: m = the signed x of largest |x| (lowest index wins ties);
 *            d = m / -8 (fp32 RN); t = x / d (0 if d == 0); u = t + 8.5 (fp32 RN);
 *            q = min(15, trunc(u)); byte j = q[j] | q[j+16] << 4; stored fp16_RN(d).
 *    Decoding is exact: x^ = d16 * q (q8_0), d16 * (q - 8) (q4_0).
 *  - turbo4, a Walsh-Hadamard-rotated 4-bit scalar codec at 4.125 bits per
 *    value (the turbo4 row of the same "Codecs" table; its "How it works"
 *    list: an FWHT rotation with random sign flips makes the entries of a KV
 *    vector close to i.i.d. Gaussian).  The pages give only the rotation and
 *    the size (4 bits per value + 16 bits per 128-value row); this library's
 *    reading, written out here:
 *      signs s_j = -1 where bit 63 of output j (j = 0..127) of SplitMix64
 *            seeded with 0x4B5651 is set, else +1;
 *      t = s * x (fp32), then the unnormalised fast Walsh-Hadamard transform
 *            in Sylvester order, stage h = 1, 2, ..., 64 turning each pair
 *            (j, j + h) with j & h == 0 into (a + b, a - b), fp32 additions;
 *      y = t / 8 (exact); then the q4_0 rule over all 128 values of y (one
 *            scale per row); nibbles packed per 32-value group as in q4_0.
 *    Decoding: y^ = d16 * (q - 8), x^ = s * H y^ / 16 (H H = 128 I, so the
 *    rotation is orthogonal up to the exact factors 1/8 and 1/16; x^ is
 *    exact in fp32 and fp64).  Canonical row: d16 then 64 packed bytes.
 *  - The per-(layer, side) codec choice of the classic F16 -> Q8_0 -> Q4_0
 *    ladder ("VBR -- Variable Bit-Rate KV Cache" section of the same listing)
 *    is just the codec argument of every call below.
 *  - Softmax attention, the plain definition, in fp64 over the dequantized
 *    cache: s_t = scale * q . k^_t over the attended keys, p = softmax(s),
 *    o = sum_t p_t v^_t, lse = max s + log sum exp(s - max s).  Decode attends
 *    every cached key; a prefill chunk attends causally (query at absolute
 *    position P sees keys 0..P), after the chunk's own keys were appended
 *    (the ubatch discussion of the serverAppConfigs commit log).
 *  - Degrading one (layer, side) tensor down the classic ladder (the same
 *    VBR section: the cache degrades one tensor at a time, f16 -> q8_0 ->
 *    q4_0, and the classic order is strictly banded, every movable tensor
 *    reaching q8_0 before any reaches q4_0; a degrade stops at the last step
 *    whose aggregate bits per value stays at or above the floor).  A tensor is
 *    re-encoded from its decoded values: x^ (exact in fp32) goes through the
 *    encoder of the new codec as fp32 input; an f16 target rounds x^ to fp16.
 *    Bits per value of a codec = row bytes * 8 / 128; the aggregate over
 *    tensors of equal size is their mean.
 *  - Paged caches (block-level KV management of the vLLM PagedAttention
 *    entry in the references of the buun-llama-cpp listing; pools shared by
 *    slots and 256-aligned, serverAppConfigs commit log): a page is 256
 *    tokens (16 units) of every kv head of one sequence; a side's pool is
 *    [n_pages][n_kv_head][16 units][unit bytes]; unit j of stream (s, h)
 *    lives at pool unit (table[s][j / 16] * n_kv + h) * 16 + j % 16.  The
 *    oracle computes on the contiguous layout and moves whole units between
 *    the two layouts (kvqo_page_scatter / kvqo_page_gather).
 *  - Probe-scored eviction (the "Sparse KV eviction" item of the "How It
 *    Works" section of the GitHot listing of VITRIOL: an attention probe,
 *    q.K softmax with exponential decay, scores the cells; the lowest-scored
 *    middle cells are evicted first; sinks and recent cells are protected).  The probe mass of token t
 *    of a sequence is the softmax weight the decode query of every query head
 *    puts on t, summed over the query heads; score = decay * score + mass.
 *    Eviction picks the n lowest (score, t) pairs among the middle tokens
 *    [n_sink, len - n_recent) and removes them: the kept tokens move down
 *    in order, bytes unchanged.
 *  - The cache byte layout, written from its specification (the library's
 *    public header documents the same layout): the cache of one layer and
 *    side is [seq][kv_head][capacity/16 units][unit bytes]; a unit holds 16
 *    consecutive tokens; every canonical row byte (the row's blocks laid end
 *    to end) has exactly one place in the unit, given by kvqo_unit_offset.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KVQO_D 128
#define KVQO_UNIT_TOKENS 16

enum { KVQO_F16 = 0, KVQO_Q8_0 = 1, KVQO_Q4_0 = 2, KVQO_TURBO4 = 3 };
#define KVQO_TURBO_SEED 0x4B5651ull
enum { KVQO_SIDE_K = 0, KVQO_SIDE_V = 1 };

/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32, written out bit by bit.                       */
/* ------------------------------------------------------------------------ */

float kvqo_half_to_float(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    int exp = (h >> 10) & 0x1f;
    uint32_t man = h & 0x3ffu;
    float mag;
    if (exp == 0) {
        /* zero or subnormal: man * 2^-24, exact in fp32 */
        mag = ldexpf((float)man, -24);
    } else if (exp == 31) {
        mag = man ? NAN : INFINITY;
    } else {
        mag = ldexpf((float)(man | 0x400u), exp - 25);
    }
    return sign ? -mag : mag;
}

double kvqo_half_to_double(uint16_t h) { return (double)kvqo_half_to_float(h); }

/* Round an fp32 value to the nearest binary16, ties to even; values beyond the
 * largest finite half become infinity, tiny values become subnormals or zero. */
uint16_t kvqo_float_to_half_rn(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, 4);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    uint32_t fexp = (bits >> 23) & 0xffu;
    uint32_t fman = bits & 0x7fffffu;
    if (fexp == 0xff) /* inf / nan */
        return (uint16_t)(sign | 0x7c00u | (fman ? 0x200u : 0u));
    if (fexp == 0 && fman == 0)
        return sign;
    /* value = 1.fman * 2^(fexp-127) (fp32 subnormals are far below half range) */
    int e = (int)fexp - 127;
    if (e > 15)
        return (uint16_t)(sign | 0x7c00u);
    uint32_t sig = fman | 0x800000u; /* 24-bit significand, value = sig * 2^(e-23) */
    int shift;                       /* right shift turning sig into a half mantissa */
    int hexp;
    if (e >= -14) {                  /* normal half: 11-bit significand */
        shift = 13;
        hexp = e + 15;
    } else {                         /* subnormal half: units of 2^-24 */
        shift = 13 + (-14 - e);
        hexp = 0;
        if (shift > 25)              /* below half of the smallest subnormal */
            return sign;
    }
    uint32_t kept = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (kept & 1u)))
        kept += 1;
    uint32_t out;
    if (hexp == 0) {
        out = kept; /* may carry into the smallest normal, which is then exact */
    } else {
        /* kept holds 1.mmmmmmmmmm (11 bits), maybe carried to 2^11 */
        if (kept >= 0x800u) {
            kept >>= 1;
            hexp += 1;
        }
        if (hexp >= 31)
            return (uint16_t)(sign | 0x7c00u);
        out = ((uint32_t)hexp << 10) | (kept & 0x3ffu);
    }
    return (uint16_t)(sign | out);
}

/* ------------------------------------------------------------------------ */
/* Block codecs (canonical byte form: fp16 scale little-endian, then quants). */
/* ------------------------------------------------------------------------ */

static int kvqo_all_finite(const float *x, int n)
{
    for (int j = 0; j < n; ++j)
        if (!isfinite(x[j]))
            return 0;
    return 1;
}

/* q8_0 of 32 fp32 values: 34 bytes = d16 (2) + 32 x int8.
 * Returns 0, or -1 for non-finite input. */
int kvqo_q8_0_encode_block_f32(const float *x, uint8_t *out)
{
    if (!kvqo_all_finite(x, 32))
        return -1;
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) {
        float a = fabsf(x[j]);
        if (a > amax)
            amax = a;
    }
    float d = amax / 127.0f;
    uint16_t d16 = kvqo_float_to_half_rn(d);
    out[0] = (uint8_t)(d16 & 0xffu);
    out[1] = (uint8_t)(d16 >> 8);
    for (int j = 0; j < 32; ++j) {
        int q = 0;
        if (d != 0.0f) {
            float t = x[j] / d;
            q = (int)roundf(t); /* C roundf: halfway cases away from zero */
        }
        out[2 + j] = (uint8_t)(int8_t)q;
    }
    return 0;
}

/* The same from 32 fp16 values (converted to fp32 exactly). */
int kvqo_q8_0_encode_block(const uint16_t *x16, uint8_t *out)
{
    float x[32];
    for (int j = 0; j < 32; ++j)
        x[j] = kvqo_half_to_float(x16[j]);
    return kvqo_q8_0_encode_block_f32(x, out);
}

/* q4_0 of 32 fp32 values: 18 bytes = d16 (2) + 16 bytes,
 * byte j = q[j] | q[j+16] << 4. */
int kvqo_q4_0_encode_block_f32(const float *x, uint8_t *out)
{
    if (!kvqo_all_finite(x, 32))
        return -1;
    int jmax = 0;
    float amax = fabsf(x[0]);
    for (int j = 1; j < 32; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) { /* strict: the lowest index keeps a tie */
            amax = a;
            jmax = j;
        }
    }
    float m = x[jmax];
    float d = m / -8.0f;
    uint16_t d16 = kvqo_float_to_half_rn(d);
    out[0] = (uint8_t)(d16 & 0xffu);
    out[1] = (uint8_t)(d16 >> 8);
    int q[32];
    for (int j = 0; j < 32; ++j) {
        float t = (d != 0.0f) ? x[j] / d : 0.0f;
        float u = t + 8.5f;
        int v = (int)u; /* truncation toward zero; u >= 0.5 here */
        q[j] = v > 15 ? 15 : v;
    }
    for (int j = 0; j < 16; ++j)
        out[2 + j] = (uint8_t)((q[j] & 0xf) | ((q[j + 16] & 0xf) << 4));
    return 0;
}

int kvqo_q4_0_encode_block(const uint16_t *x16, uint8_t *out)
{
    float x[32];
    for (int j = 0; j < 32; ++j)
        x[j] = kvqo_half_to_float(x16[j]);
    return kvqo_q4_0_encode_block_f32(x, out);
}

void kvqo_q8_0_decode_block(const uint8_t *in, double *out)
{
    uint16_t d16 = (uint16_t)(in[0] | (in[1] << 8));
    double d = kvqo_half_to_double(d16);
    for (int j = 0; j < 32; ++j)
        out[j] = d * (double)(int8_t)in[2 + j];
}

void kvqo_q4_0_decode_block(const uint8_t *in, double *out)
{
    uint16_t d16 = (uint16_t)(in[0] | (in[1] << 8));
    double d = kvqo_half_to_double(d16);
    for (int j = 0; j < 16; ++j) {
        out[j] = d * (double)((int)(in[2 + j] & 0xf) - 8);
        out[j + 16] = d * (double)((int)(in[2 + j] >> 4) - 8);
    }
}

/* ---- turbo4 ---------------------------------------------------------- */

/* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): the state advances by 0x9E3779B97F4A7C15 and is
 * mixed by two xor-shift-multiply steps and a final xor-shift. */
uint64_t kvqo_splitmix64_next(uint64_t *state)
{
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* The 128 turbo4 sign flips, +1 or -1. */
void kvqo_turbo_signs(int *sgn)
{
    uint64_t st = KVQO_TURBO_SEED;
    for (int j = 0; j < KVQO_D; ++j)
        sgn[j] = (kvqo_splitmix64_next(&st) >> 63) ? -1 : 1;
}

/* In-place unnormalised fast Walsh-Hadamard transform of 128 values. */
void kvqo_fwht128_f32(float *t)
{
    for (int h = 1; h < KVQO_D; h <<= 1)
        for (int i = 0; i < KVQO_D; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                float a = t[j], b = t[j + h];
                t[j] = a + b;
                t[j + h] = a - b;
            }
}

void kvqo_fwht128_f64(double *t)
{
    for (int h = 1; h < KVQO_D; h <<= 1)
        for (int i = 0; i < KVQO_D; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                double a = t[j], b = t[j + h];
                t[j] = a + b;
                t[j + h] = a - b;
            }
}

/* turbo4 of one row of 128 fp32 values: 66 bytes = d16 (2) + 64 bytes,
 * byte 16 g + j (group g of 32, j < 16) = q[32 g + j] | q[32 g + j + 16] << 4.
 * Returns 0, or -1 for non-finite input. */
int kvqo_turbo4_encode_row_f32(const float *x, uint8_t *out)
{
    if (!kvqo_all_finite(x, KVQO_D))
        return -1;
    int sgn[KVQO_D];
    kvqo_turbo_signs(sgn);
    float y[KVQO_D];
    for (int j = 0; j < KVQO_D; ++j)
        y[j] = sgn[j] < 0 ? -x[j] : x[j];
    kvqo_fwht128_f32(y);
    for (int j = 0; j < KVQO_D; ++j)
        y[j] = y[j] * 0.125f;
    int jmax = 0;
    float amax = fabsf(y[0]);
    for (int j = 1; j < KVQO_D; ++j) {
        float a = fabsf(y[j]);
        if (a > amax) { /* strict: the lowest index keeps a tie */
            amax = a;
            jmax = j;
        }
    }
    float m = y[jmax];
    float d = m / -8.0f;
    uint16_t d16 = kvqo_float_to_half_rn(d);
    out[0] = (uint8_t)(d16 & 0xffu);
    out[1] = (uint8_t)(d16 >> 8);
    int q[KVQO_D];
    for (int j = 0; j < KVQO_D; ++j) {
        float t = (d != 0.0f) ? y[j] / d : 0.0f;
        float u = t + 8.5f;
        int v = (int)u; /* truncation toward zero; u >= 0.5 here */
        q[j] = v > 15 ? 15 : v;
    }
    for (int g = 0; g < 4; ++g)
        for (int j = 0; j < 16; ++j)
            out[2 + 16 * g + j] =
                (uint8_t)((q[32 * g + j] & 0xf) | ((q[32 * g + j + 16] & 0xf) << 4));
    return 0;
}

int kvqo_turbo4_encode_row(const uint16_t *x16, uint8_t *out)
{
    float x[KVQO_D];
    for (int j = 0; j < KVQO_D; ++j)
        x[j] = kvqo_half_to_float(x16[j]);
    return kvqo_turbo4_encode_row_f32(x, out);
}

/* The rotated values y^ = d16 * (q - 8) of one turbo4 row (exact). */
void kvqo_turbo4_rotated(const uint8_t *in, double *yh)
{
    double d = kvqo_half_to_double((uint16_t)(in[0] | (in[1] << 8)));
    for (int g = 0; g < 4; ++g)
        for (int j = 0; j < 16; ++j) {
            yh[32 * g + j] = d * (double)((int)(in[2 + 16 * g + j] & 0xf) - 8);
            yh[32 * g + j + 16] = d * (double)((int)(in[2 + 16 * g + j] >> 4) - 8);
        }
}

/* x^ = s * H y^ / 16 of one turbo4 row (exact in fp64). */
void kvqo_turbo4_decode_row(const uint8_t *in, double *out)
{
    int sgn[KVQO_D];
    kvqo_turbo_signs(sgn);
    kvqo_turbo4_rotated(in, out);
    kvqo_fwht128_f64(out);
    for (int j = 0; j < KVQO_D; ++j)
        out[j] = sgn[j] * out[j] / 16.0;
}

/* Canonical row bytes for head_dim 128: the row's four blocks end to end
 * (turbo4: the row's scale, then its 64 packed bytes). */
int kvqo_row_bytes(int codec)
{
    switch (codec) {
    case KVQO_F16: return 2 * KVQO_D;
    case KVQO_Q8_0: return 4 * 34;
    case KVQO_Q4_0: return 4 * 18;
    case KVQO_TURBO4: return 2 + KVQO_D / 2;
    default: return -1;
    }
}

int kvqo_unit_bytes(int codec)
{
    int rb = kvqo_row_bytes(codec);
    return rb < 0 ? -1 : rb * KVQO_UNIT_TOKENS;
}

/* Encode n rows of 128 fp16 values into canonical row bytes. */
int kvqo_encode_rows(int codec, int64_t n, const uint16_t *x, uint8_t *out)
{
    int rb = kvqo_row_bytes(codec);
    if (rb < 0)
        return -1;
    for (int64_t i = 0; i < n; ++i) {
        const uint16_t *xr = x + i * KVQO_D;
        uint8_t *o = out + i * rb;
        if (codec == KVQO_F16) {
            for (int d = 0; d < KVQO_D; ++d) {
                o[2 * d] = (uint8_t)(xr[d] & 0xffu);
                o[2 * d + 1] = (uint8_t)(xr[d] >> 8);
            }
        } else if (codec == KVQO_TURBO4) {
            int rc = kvqo_turbo4_encode_row(xr, o);
            if (rc)
                return rc;
        } else {
            for (int b = 0; b < 4; ++b) {
                int rc = codec == KVQO_Q8_0 ? kvqo_q8_0_encode_block(xr + 32 * b, o + 34 * b)
                                            : kvqo_q4_0_encode_block(xr + 32 * b, o + 18 * b);
                if (rc)
                    return rc;
            }
        }
    }
    return 0;
}

/* Decode n canonical rows into fp64 values. */
int kvqo_decode_rows(int codec, int64_t n, const uint8_t *in, double *out)
{
    int rb = kvqo_row_bytes(codec);
    if (rb < 0)
        return -1;
    for (int64_t i = 0; i < n; ++i) {
        const uint8_t *r = in + i * rb;
        double *o = out + i * KVQO_D;
        if (codec == KVQO_F16) {
            for (int d = 0; d < KVQO_D; ++d)
                o[d] = kvqo_half_to_double((uint16_t)(r[2 * d] | (r[2 * d + 1] << 8)));
        } else if (codec == KVQO_Q8_0) {
            for (int b = 0; b < 4; ++b)
                kvqo_q8_0_decode_block(r + 34 * b, o + 32 * b);
        } else if (codec == KVQO_TURBO4) {
            kvqo_turbo4_decode_row(r, o);
        } else {
            for (int b = 0; b < 4; ++b)
                kvqo_q4_0_decode_block(r + 18 * b, o + 32 * b);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Cache layout: where canonical row byte cb of token row r (0..15) of a unit */
/* lives inside the unit.  K-side and V-side units differ.                   */
/* ------------------------------------------------------------------------ */

int kvqo_unit_offset(int codec, int side, int r, int cb)
{
    if (r < 0 || r >= KVQO_UNIT_TOKENS || cb < 0 || cb >= kvqo_row_bytes(codec))
        return -1;
    int g = r & 7, rh = r >> 3;              /* K side: row = g + 8 * rh */
    int tig = (r & 7) >> 1, par = r & 1;     /* V side: row = 2 * tig + par + 8 * rh */
    if (codec == KVQO_F16) {
        int d = cb >> 1, k = cb & 1;
        if (side == KVQO_SIDE_K) {
            int b = d >> 5, h = (d >> 4) & 1, w = (d >> 2) & 3, i = d & 3;
            return (2 * b + rh) * 512 + (4 * g + w) * 16 + h * 8 + i * 2 + k;
        } else {
            int mt = d >> 4, gq = (d & 15) >> 1, sub = d & 1;
            return mt * 512 + (4 * gq + tig) * 16 + (rh * 4 + sub * 2 + par) * 2 + k;
        }
    }
    if (codec == KVQO_Q8_0) {
        int b = cb / 34, o = cb % 34;
        if (o < 2) { /* scale byte o of block b */
            if (side == KVQO_SIDE_K)
                return 2048 + g * 16 + rh * 8 + b * 2 + o;
            return 2048 + tig * 32 + b * 8 + rh * 4 + par * 2 + o;
        }
        int e = o - 2, d = 32 * b + e;
        if (side == KVQO_SIDE_K) {
            int h = e >> 4, w = (e >> 2) & 3, i = e & 3;
            return b * 512 + (4 * g + w) * 16 + (2 * rh + h) * 4 + i;
        } else {
            int mt = d >> 4, gq = (d & 15) >> 1, sub = d & 1;
            return (mt >> 1) * 512 + (4 * gq + tig) * 16 + ((mt & 1) * 2 + rh) * 4 + par * 2 + sub;
        }
    }
    if (codec == KVQO_Q4_0) {
        int b = cb / 18, o = cb % 18;
        if (o < 2) {
            if (side == KVQO_SIDE_K)
                return 1024 + g * 16 + rh * 8 + b * 2 + o;
            return 1024 + tig * 32 + b * 8 + rh * 4 + par * 2 + o;
        }
        int jc = o - 2; /* canonical packed byte 0..15 of block b */
        if (side == KVQO_SIDE_K) {
            int w = jc >> 2, i = jc & 3;
            return (b >> 1) * 512 + (4 * g + w) * 16 + ((b & 1) * 2 + rh) * 4 + i;
        } else {
            int mt = 2 * b + (jc >> 3), gq = jc & 7;
            return (mt >> 2) * 512 + (4 * gq + tig) * 16 + (mt & 3) * 4 + par * 2 + rh;
        }
    }
    if (codec == KVQO_TURBO4) {
        /* packed bytes at the q4_0 places of group b; one scale per row */
        if (cb < 2) {
            if (side == KVQO_SIDE_K)
                return 1024 + g * 4 + rh * 2 + cb;
            return 1024 + tig * 8 + rh * 4 + par * 2 + cb;
        }
        int b = (cb - 2) >> 4, jc = (cb - 2) & 15;
        if (side == KVQO_SIDE_K) {
            int w = jc >> 2, i = jc & 3;
            return (b >> 1) * 512 + (4 * g + w) * 16 + ((b & 1) * 2 + rh) * 4 + i;
        } else {
            int mt = 2 * b + (jc >> 3), gq = jc & 7;
            return (mt >> 2) * 512 + (4 * gq + tig) * 16 + (mt & 3) * 4 + par * 2 + rh;
        }
    }
    return -1;
}

static uint8_t *kvqo_stream(uint8_t *cache, int codec, int n_kv, int capacity, int seq, int kvh)
{
    int64_t ub = kvqo_unit_bytes(codec);
    int64_t units = capacity / KVQO_UNIT_TOKENS;
    return cache + ((int64_t)seq * n_kv + kvh) * units * ub;
}

/* Scatter one canonical row into token position pos of a (seq, kv_head) stream. */
static void kvqo_put_row(uint8_t *stream, int codec, int side, int64_t pos, const uint8_t *row)
{
    int rb = kvqo_row_bytes(codec);
    uint8_t *unit = stream + (pos / KVQO_UNIT_TOKENS) * kvqo_unit_bytes(codec);
    int r = (int)(pos % KVQO_UNIT_TOKENS);
    for (int cb = 0; cb < rb; ++cb)
        unit[kvqo_unit_offset(codec, side, r, cb)] = row[cb];
}

static void kvqo_get_row(const uint8_t *stream, int codec, int side, int64_t pos, uint8_t *row)
{
    int rb = kvqo_row_bytes(codec);
    const uint8_t *unit = stream + (pos / KVQO_UNIT_TOKENS) * kvqo_unit_bytes(codec);
    int r = (int)(pos % KVQO_UNIT_TOKENS);
    for (int cb = 0; cb < rb; ++cb)
        row[cb] = unit[kvqo_unit_offset(codec, side, r, cb)];
}

/* Quantize-on-append for one side of one layer.
 * x_new: fp16 [n_seqs][max_new][n_kv][128]; row i < n_new[s] of sequence s
 * goes to token position seq_lens[s] + i.  Lengths are not updated here.
 * Returns 0, -1 on bad arguments or capacity overflow, -2 on non-finite input.
 * Rows are independent (each has its own token position), so OpenMP spreads
 * the rows of a sequence over threads; each row is encoded exactly as alone. */
int kvqo_append_side(int codec, int side, uint8_t *cache, int n_seqs, int n_kv, int capacity,
                     const int32_t *seq_lens, const int32_t *n_new, int max_new,
                     const uint16_t *x_new)
{
    int rb = kvqo_row_bytes(codec);
    if (rb < 0 || capacity % KVQO_UNIT_TOKENS)
        return -1;
    for (int s = 0; s < n_seqs; ++s)
        if (n_new[s] < 0 || n_new[s] > max_new || seq_lens[s] < 0 ||
            (int64_t)seq_lens[s] + n_new[s] > capacity)
            return -1;
    int bad = 0;
    for (int s = 0; s < n_seqs; ++s) {
        int64_t n_rows = (int64_t)n_new[s] * n_kv;
#pragma omp parallel for schedule(static)
        for (int64_t ih = 0; ih < n_rows; ++ih) {
            int64_t i = ih / n_kv;
            int h = (int)(ih % n_kv);
            uint8_t row[256];
            const uint16_t *x = x_new + (((int64_t)s * max_new + i) * n_kv + h) * KVQO_D;
            if (kvqo_encode_rows(codec, 1, x, row)) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            kvqo_put_row(kvqo_stream(cache, codec, n_kv, capacity, s, h), codec, side,
                         (int64_t)seq_lens[s] + i, row);
        }
        if (bad)
            return -2;
    }
    return 0;
}

/* Read tokens [0, n_tokens) of one (seq, kv_head) stream back as fp64 [n][128].
 * Tokens are decoded independently (OpenMP over tokens when not nested). */
int kvqo_dequant_stream(int codec, int side, const uint8_t *cache, int n_kv, int capacity,
                        int seq, int kvh, int64_t n_tokens, double *out)
{
    int rb = kvqo_row_bytes(codec);
    if (rb < 0 || n_tokens > capacity)
        return -1;
    const uint8_t *st = kvqo_stream((uint8_t *)cache, codec, n_kv, capacity, seq, kvh);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n_tokens; ++t) {
        uint8_t row[256];
        kvqo_get_row(st, codec, side, t, row);
        kvqo_decode_rows(codec, 1, row, out + t * KVQO_D);
    }
    return 0;
}

/* max |x^| over tokens [0, n_tokens) of one stream (0 for an empty stream):
 * the reference magnitude of the attention tolerance. */
double kvqo_stream_absmax(int codec, int side, const uint8_t *cache, int n_kv, int capacity,
                          int seq, int kvh, int64_t n_tokens)
{
    int rb = kvqo_row_bytes(codec);
    if (rb < 0 || n_tokens > capacity)
        return -1.0;
    const uint8_t *st = kvqo_stream((uint8_t *)cache, codec, n_kv, capacity, seq, kvh);
    double m = 0.0;
#pragma omp parallel for schedule(static) reduction(max : m)
    for (int64_t t = 0; t < n_tokens; ++t) {
        uint8_t row[256];
        double x[KVQO_D];
        kvqo_get_row(st, codec, side, t, row);
        kvqo_decode_rows(codec, 1, row, x);
        for (int d = 0; d < KVQO_D; ++d)
            if (fabs(x[d]) > m)
                m = fabs(x[d]);
    }
    return m;
}

/* ------------------------------------------------------------------------ */
/* Paged layout: units moved between a contiguous cache and a page pool.     */
/* ------------------------------------------------------------------------ */

#define KVQO_PAGE_UNITS 16

/* Pool unit index of unit j of stream (s, h), or -1 for an unmapped page. */
int64_t kvqo_paged_unit(int s, int h, int64_t j, int n_kv, const int32_t *table,
                        int pages_per_seq, int n_pages)
{
    int64_t pg = j / KVQO_PAGE_UNITS;
    if (pg >= pages_per_seq)
        return -1;
    int32_t page = table[(int64_t)s * pages_per_seq + pg];
    if (page < 0 || page >= n_pages)
        return -1;
    return ((int64_t)page * n_kv + h) * KVQO_PAGE_UNITS + j % KVQO_PAGE_UNITS;
}

/* Copy every unit of the contiguous cache [n_seqs][n_kv][capacity/16] whose
 * page is mapped into the pool (to_pool != 0), or back (to_pool == 0).
 * capacity must equal pages_per_seq * 256.  Returns 0 or -1. */
int kvqo_page_move(int codec, uint8_t *cache, int n_seqs, int n_kv, int capacity,
                   const int32_t *table, int pages_per_seq, uint8_t *pool, int n_pages,
                   int to_pool)
{
    int64_t ub = kvqo_unit_bytes(codec);
    if (ub < 0 || capacity != pages_per_seq * KVQO_PAGE_UNITS * KVQO_UNIT_TOKENS)
        return -1;
    int64_t units = capacity / KVQO_UNIT_TOKENS;
    for (int s = 0; s < n_seqs; ++s)
        for (int h = 0; h < n_kv; ++h)
            for (int64_t j = 0; j < units; ++j) {
                int64_t pu = kvqo_paged_unit(s, h, j, n_kv, table, pages_per_seq, n_pages);
                if (pu < 0)
                    continue;
                uint8_t *c = cache + (((int64_t)s * n_kv + h) * units + j) * ub;
                uint8_t *q = pool + pu * ub;
                if (to_pool)
                    memcpy(q, c, (size_t)ub);
                else
                    memcpy(c, q, (size_t)ub);
            }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Degrade ladder: re-encode one tensor; bits per value; the banded step.    */
/* ------------------------------------------------------------------------ */

/* Re-encode tokens [0, seq_lens[s]) of every (seq, kv_head) stream of one
 * side from src_codec to dst_codec (dst is a separate cache of dst_codec).
 * Each row is decoded to fp32 (exact: d16 * q or d16 * (n - 8), the fp16
 * value, or turbo4's x^) and encoded again: q8_0 / q4_0 / turbo4 by the fp32
 * formulas above, f16 by rounding to fp16.  Returns 0, or -1 on bad arguments. */
int kvqo_requantize_side(int src_codec, int dst_codec, int side, const uint8_t *src,
                         uint8_t *dst, int n_seqs, int n_kv, int capacity,
                         const int32_t *seq_lens)
{
    if (kvqo_row_bytes(src_codec) < 0 || kvqo_row_bytes(dst_codec) < 0 ||
        capacity % KVQO_UNIT_TOKENS)
        return -1;
    for (int s = 0; s < n_seqs; ++s)
        if (seq_lens[s] < 0 || seq_lens[s] > capacity)
            return -1;
    int bad = 0;
    for (int s = 0; s < n_seqs; ++s) {
        for (int h = 0; h < n_kv; ++h) {
            const uint8_t *ss = kvqo_stream((uint8_t *)src, src_codec, n_kv, capacity, s, h);
            uint8_t *ds = kvqo_stream(dst, dst_codec, n_kv, capacity, s, h);
            /* rows are independent: OpenMP over tokens, same bytes on any
             * thread count */
#pragma omp parallel for schedule(static)
            for (int64_t t = 0; t < seq_lens[s]; ++t) {
                uint8_t row[256], out[256];
                double xd[KVQO_D];
                float x[KVQO_D];
                kvqo_get_row(ss, src_codec, side, t, row);
                kvqo_decode_rows(src_codec, 1, row, xd);
                for (int d = 0; d < KVQO_D; ++d)
                    x[d] = (float)xd[d]; /* exact: the products fit fp32 */
                if (dst_codec == KVQO_F16) {
                    for (int d = 0; d < KVQO_D; ++d) {
                        uint16_t hb = kvqo_float_to_half_rn(x[d]);
                        out[2 * d] = (uint8_t)(hb & 0xffu);
                        out[2 * d + 1] = (uint8_t)(hb >> 8);
                    }
                } else if (dst_codec == KVQO_TURBO4) {
                    if (kvqo_turbo4_encode_row_f32(x, out)) {
#pragma omp atomic write
                        bad = 1;
                        continue;
                    }
                } else {
                    int rc = 0;
                    for (int b = 0; b < 4; ++b)
                        rc |= dst_codec == KVQO_Q8_0
                                  ? kvqo_q8_0_encode_block_f32(x + 32 * b, out + 34 * b)
                                  : kvqo_q4_0_encode_block_f32(x + 32 * b, out + 18 * b);
                    if (rc) {
#pragma omp atomic write
                        bad = 1;
                        continue;
                    }
                }
                kvqo_put_row(ds, dst_codec, side, t, out);
            }
        }
    }
    return bad ? -1 : 0;
}

/* Bits per value of a codec: row bytes * 8 / head_dim (16, 8.5, 4.5). */
double kvqo_bits_per_value(int codec)
{
    int rb = kvqo_row_bytes(codec);
    return rb < 0 ? -1.0 : rb * 8.0 / KVQO_D;
}

/* Aggregate bits per value of n tensors holding equally many values. */
double kvqo_aggregate_bpv(const int *codecs, int n)
{
    double sum = 0.0;
    for (int i = 0; i < n; ++i)
        sum += kvqo_bits_per_value(codecs[i]);
    return n > 0 ? sum / n : 0.0;
}

/* The next step of the banded classic ladder: the first tensor in `order`
 * (n_order movable tensor indices, price order) still above rung q8_0 goes to
 * q8_0; once every movable tensor is at q8_0 or below, the first one still
 * above q4_0 goes to q4_0.  The step is taken only if the aggregate over all
 * n tensors afterwards is >= floor_bpv.  Writes the tensor and its new codec
 * and returns 1, or returns 0 when no step remains. */
int kvqo_ladder_next(const int *codecs, int n, const int *order, int n_order, double floor_bpv,
                     int *tensor, int *codec)
{
    static const int rungs[2] = {KVQO_Q8_0, KVQO_Q4_0};
    for (int k = 0; k < 2; ++k) {
        for (int i = 0; i < n_order; ++i) {
            int t = order[i];
            if (codecs[t] < rungs[k]) { /* codec ids grow as bits shrink */
                double sum = 0.0;
                for (int j = 0; j < n; ++j)
                    sum += kvqo_bits_per_value(j == t ? rungs[k] : codecs[j]);
                if (sum / n < floor_bpv)
                    return 0;
                *tensor = t;
                *codec = rungs[k];
                return 1;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Probe-scored eviction.                                                    */
/* ------------------------------------------------------------------------ */

/* mass[s][t] (t < seq_lens[s], capacity columns) = sum over the n_q query
 * heads of softmax_t(scale * q_h . k^_t) over the sequence's keys, in fp64. */
int kvqo_probe_mass(int codec_k, const uint8_t *cache_k, int n_seqs, int n_kv, int n_q,
                    int capacity, const int32_t *seq_lens, const uint16_t *q, double scale,
                    double *mass)
{
    if (n_kv <= 0 || n_q % n_kv)
        return -1;
    int G = n_q / n_kv;
    for (int s = 0; s < n_seqs; ++s) {
        int64_t T = seq_lens[s];
        if (T < 0 || T > capacity)
            return -1;
        double *m = mass + (int64_t)s * capacity;
        for (int64_t t = 0; t < capacity; ++t)
            m[t] = 0.0;
        if (T == 0)
            continue;
        double *K = (double *)malloc(sizeof(double) * (size_t)T * KVQO_D);
        double *sc = (double *)malloc(sizeof(double) * (size_t)T);
        if (!K || !sc) {
            free(K); free(sc);
            return -1;
        }
        for (int h = 0; h < n_kv; ++h) {
            kvqo_dequant_stream(codec_k, KVQO_SIDE_K, cache_k, n_kv, capacity, s, h, T, K);
            for (int j = 0; j < G; ++j) {
                const uint16_t *qh = q + ((int64_t)s * n_q + (int64_t)h * G + j) * KVQO_D;
                /* the scores and the per-token additions are independent per
                 * token (OpenMP over tokens); the normaliser is summed on one
                 * thread in token order, so the bits do not depend on the
                 * thread count */
                double mx = -INFINITY;
#pragma omp parallel for schedule(static) reduction(max : mx)
                for (int64_t t = 0; t < T; ++t) {
                    double d = 0.0;
                    for (int c = 0; c < KVQO_D; ++c)
                        d += kvqo_half_to_double(qh[c]) * K[t * KVQO_D + c];
                    sc[t] = scale * d;
                    if (sc[t] > mx)
                        mx = sc[t];
                }
                double sum = 0.0;
                for (int64_t t = 0; t < T; ++t)
                    sum += exp(sc[t] - mx);
#pragma omp parallel for schedule(static)
                for (int64_t t = 0; t < T; ++t)
                    m[t] += exp(sc[t] - mx) / sum;
            }
        }
        free(K);
        free(sc);
    }
    return 0;
}

/* The n_evict positions t in [n_sink, len - n_recent) with the smallest
 * (score[t], t), written in increasing t.  Returns how many were written
 * (fewer when the middle range is shorter). */
int kvqo_evict_select(const float *score, int len, int n_sink, int n_recent, int n_evict,
                      int32_t *out)
{
    int lo = n_sink, hi = len - n_recent;
    if (hi <= lo || n_evict <= 0)
        return 0;
    int n = hi - lo, k = n_evict < n ? n_evict : n;
    uint8_t *taken = (uint8_t *)calloc((size_t)n, 1);
    if (!taken)
        return -1;
    for (int r = 0; r < k; ++r) { /* k passes of a plain minimum search */
        int best = -1;
        for (int i = 0; i < n; ++i) {
            if (taken[i])
                continue;
            if (best < 0 || score[lo + i] < score[lo + best])
                best = i; /* strict: the lower t keeps a tie */
        }
        taken[best] = 1;
    }
    int w = 0;
    for (int i = 0; i < n; ++i)
        if (taken[i])
            out[w++] = lo + i;
    free(taken);
    return w;
}

/* Remove the listed positions (increasing, below seq_lens[s]) of every
 * sequence from one side's cache: kept tokens move down in order, bytes
 * unchanged; dst is a separate cache of the same codec (zero elsewhere).
 * evict: [n_seqs][max_evict] positions, n_ev[s] of them used. */
int kvqo_compact_side(int codec, int side, const uint8_t *src, uint8_t *dst, int n_seqs,
                      int n_kv, int capacity, const int32_t *seq_lens, const int32_t *evict,
                      const int32_t *n_ev, int max_evict)
{
    if (kvqo_row_bytes(codec) < 0)
        return -1;
    /* streams are independent: OpenMP over (seq, kv head), same bytes on any
     * thread count */
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int s = 0; s < n_seqs; ++s) {
        for (int h = 0; h < n_kv; ++h) {
            uint8_t row[256];
            const int32_t *ev = evict + (int64_t)s * max_evict;
            const uint8_t *ss = kvqo_stream((uint8_t *)src, codec, n_kv, capacity, s, h);
            uint8_t *ds = kvqo_stream(dst, codec, n_kv, capacity, s, h);
            int e = 0;
            int64_t w = 0;
            for (int64_t t = 0; t < seq_lens[s]; ++t) {
                if (e < n_ev[s] && ev[e] == t) {
                    ++e;
                    continue;
                }
                kvqo_get_row(ss, codec, side, t, row);
                kvqo_put_row(ds, codec, side, w++, row);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Softmax attention in fp64 (the plain definition).                         */
/* ------------------------------------------------------------------------ */

/* One query row against keys 0..n_keys-1. out: 128 doubles; *lse written. */
static void kvqo_attend_one(const uint16_t *q16, const double *K, const double *V, int64_t n_keys,
                            double scale, double *s_buf, double *out, double *lse)
{
    double q[KVQO_D];
    for (int d = 0; d < KVQO_D; ++d)
        q[d] = kvqo_half_to_double(q16[d]);
    for (int d = 0; d < KVQO_D; ++d)
        out[d] = 0.0;
    if (n_keys <= 0) {
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < n_keys; ++t) {
        const double *k = K + t * KVQO_D;
        double s = 0.0;
        for (int d = 0; d < KVQO_D; ++d)
            s += q[d] * k[d];
        s *= scale;
        s_buf[t] = s;
        if (s > m)
            m = s;
    }
    double z = 0.0;
    for (int64_t t = 0; t < n_keys; ++t) {
        double p = exp(s_buf[t] - m);
        z += p;
        const double *v = V + t * KVQO_D;
        for (int d = 0; d < KVQO_D; ++d)
            out[d] += p * v[d];
    }
    for (int d = 0; d < KVQO_D; ++d)
        out[d] /= z;
    *lse = m + log(z);
}

/* n_rows query rows (fp16 [n_rows][128]) against one key/value set
 * (fp64 [T][128]); row r attends keys 0..limit[r]-1.  OpenMP over rows when
 * compiled with it; each row is computed independently in fixed order. */
int kvqo_attend_rows(int n_rows, const uint16_t *q, int64_t T, const double *K, const double *V,
                     const int64_t *limit, double scale, double *out, double *lse)
{
    int bad = 0;
#pragma omp parallel
    {
        double *s_buf = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n_rows; ++r) {
            if (!s_buf) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            int64_t L = limit[r] < T ? limit[r] : T;
            kvqo_attend_one(q + (int64_t)r * KVQO_D, K, V, L, scale, s_buf,
                            out + (int64_t)r * KVQO_D, lse + r);
        }
        free(s_buf);
    }
    return bad ? -1 : 0;
}

/* Decode attention of one layer for a subset of (seq, kv_head) groups.
 * q: fp16 [n_seqs][n_q][128]; out fp64 [n_seqs][n_q][128]; lse fp64 [n_seqs][n_q].
 * Only groups with sel[seq * n_kv + kvh] != 0 are computed (sel may be NULL
 * for all).  Query head h reads kv head h / (n_q / n_kv).
 * The selected groups are taken in batches of at most ~2^28 dequantized
 * values: each batch's K and V streams are decoded (OpenMP over group and
 * side), then every (group, query head) row is attended on its own (OpenMP
 * over rows), each row in the fixed order of kvqo_attend_one. */
#define KVQO_DECODE_BATCH_VALUES ((int64_t)1 << 28)
int kvqo_decode_layer(int codec_k, int codec_v, const uint8_t *cache_k, const uint8_t *cache_v,
                      int n_seqs, int n_kv, int n_q, int capacity, const int32_t *seq_lens,
                      const uint16_t *q, double scale, const uint8_t *sel, double *out,
                      double *lse)
{
    if (n_kv <= 0 || n_q % n_kv)
        return -1;
    int G = n_q / n_kv;
    int n_groups = n_seqs * n_kv;
    int *grp = (int *)malloc(sizeof(int) * (size_t)(n_groups > 0 ? n_groups : 1));
    double **kv = (double **)calloc((size_t)(2 * (n_groups > 0 ? n_groups : 1)), sizeof(double *));
    if (!grp || !kv) {
        free(grp); free(kv);
        return -1;
    }
    int n_sel = 0;
    for (int gi = 0; gi < n_groups; ++gi) {
        if (sel && !sel[gi])
            continue;
        int s = gi / n_kv;
        if (seq_lens[s] < 0 || seq_lens[s] > capacity) {
            free(grp); free(kv);
            return -1;
        }
        grp[n_sel++] = gi;
    }
    int rc = 0;
    for (int b0 = 0; b0 < n_sel && !rc;) {
        /* this batch: groups b0 .. b1 - 1 */
        int b1 = b0;
        int64_t vals = 0;
        while (b1 < n_sel) {
            int64_t T = seq_lens[grp[b1] / n_kv];
            if (b1 > b0 && vals + 2 * T * KVQO_D > KVQO_DECODE_BATCH_VALUES)
                break;
            vals += 2 * T * KVQO_D;
            ++b1;
        }
        int nb = b1 - b0, bad = 0;
        for (int j = 0; j < 2 * nb; ++j) {
            int64_t T = seq_lens[grp[b0 + j / 2] / n_kv];
            kv[j] = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * KVQO_D);
            if (!kv[j])
                bad = 1;
        }
        if (!bad) {
#pragma omp parallel for schedule(dynamic, 1)
            for (int j = 0; j < 2 * nb; ++j) {
                int gi = grp[b0 + j / 2], s = gi / n_kv, h = gi % n_kv;
                if (j % 2 == 0)
                    kvqo_dequant_stream(codec_k, KVQO_SIDE_K, cache_k, n_kv, capacity, s, h,
                                        seq_lens[s], kv[j]);
                else
                    kvqo_dequant_stream(codec_v, KVQO_SIDE_V, cache_v, n_kv, capacity, s, h,
                                        seq_lens[s], kv[j]);
            }
#pragma omp parallel
            {
                int64_t Tmax = 1;
                for (int j = 0; j < nb; ++j)
                    if (seq_lens[grp[b0 + j] / n_kv] > Tmax)
                        Tmax = seq_lens[grp[b0 + j] / n_kv];
                double *s_buf = (double *)malloc(sizeof(double) * (size_t)Tmax);
#pragma omp for schedule(dynamic, 1)
                for (int jr = 0; jr < nb * G; ++jr) {
                    if (!s_buf) {
#pragma omp atomic write
                        bad = 1;
                        continue;
                    }
                    int j = jr / G, r = jr % G;
                    int gi = grp[b0 + j], s = gi / n_kv, h = gi % n_kv;
                    int64_t row = (int64_t)s * n_q + (int64_t)h * G + r;
                    kvqo_attend_one(q + row * KVQO_D, kv[2 * j], kv[2 * j + 1], seq_lens[s], scale,
                                    s_buf, out + row * KVQO_D, lse + row);
                }
                free(s_buf);
            }
        }
        for (int j = 0; j < 2 * nb; ++j) {
            free(kv[j]);
            kv[j] = NULL;
        }
        if (bad)
            rc = -1;
        b0 = b1;
    }
    free(grp);
    free(kv);
    return rc;
}

/* Causal attention of one prefill chunk of sequence `seq`: query i (absolute
 * position q_start + i) of head h attends keys 0..q_start+i.  The chunk's keys
 * must already be in the cache.  q: fp16 [n_tok][n_q][128]; out fp64
 * [n_tok][n_q][128]; lse [n_tok][n_q].  Only query rows with row_sel[i] != 0
 * are computed when row_sel is given. */
int kvqo_prefill_chunk(int codec_k, int codec_v, const uint8_t *cache_k, const uint8_t *cache_v,
                       int n_kv, int n_q, int capacity, int seq, int64_t q_start, int n_tok,
                       const uint16_t *q, double scale, const uint8_t *row_sel, double *out,
                       double *lse)
{
    if (n_kv <= 0 || n_q % n_kv)
        return -1;
    int G = n_q / n_kv;
    int64_t T = q_start + n_tok;
    if (T > capacity || q_start < 0)
        return -1;
    double *K = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * KVQO_D);
    double *V = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * KVQO_D);
    uint16_t *qg = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n_tok * G * KVQO_D);
    int64_t *lim = (int64_t *)malloc(sizeof(int64_t) * (size_t)n_tok * G);
    double *og = (double *)malloc(sizeof(double) * (size_t)n_tok * G * KVQO_D);
    double *lg = (double *)malloc(sizeof(double) * (size_t)n_tok * G);
    int rc = 0;
    if (!K || !V || !qg || !lim || !og || !lg) {
        rc = -1;
        goto done;
    }
    for (int h = 0; h < n_kv && !rc; ++h) {
        kvqo_dequant_stream(codec_k, KVQO_SIDE_K, cache_k, n_kv, capacity, seq, h, T, K);
        kvqo_dequant_stream(codec_v, KVQO_SIDE_V, cache_v, n_kv, capacity, seq, h, T, V);
        int nr = 0;
        for (int i = 0; i < n_tok; ++i) {
            if (row_sel && !row_sel[i])
                continue;
            for (int j = 0; j < G; ++j) {
                memcpy(qg + (int64_t)nr * KVQO_D, q + ((int64_t)i * n_q + h * G + j) * KVQO_D,
                       sizeof(uint16_t) * KVQO_D);
                lim[nr] = q_start + i + 1;
                ++nr;
            }
        }
        rc = kvqo_attend_rows(nr, qg, T, K, V, lim, scale, og, lg);
        nr = 0;
        for (int i = 0; i < n_tok && !rc; ++i) {
            if (row_sel && !row_sel[i])
                continue;
            for (int j = 0; j < G; ++j) {
                int64_t dst = (int64_t)i * n_q + h * G + j;
                memcpy(out + dst * KVQO_D, og + (int64_t)nr * KVQO_D, sizeof(double) * KVQO_D);
                lse[dst] = lg[nr];
                ++nr;
            }
        }
    }
done:
    free(K); free(V); free(qg); free(lim); free(og); free(lg);
    return rc;
}

int kvqo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the following OpenMP regions (n >= 1); returns the previous
 * count.  Used to time the oracle single-threaded and on all cores. */
int kvqo_set_num_threads(int n)
{
#ifdef _OPENMP
    int old = omp_get_max_threads();
    if (n >= 1)
        omp_set_num_threads(n);
    return old;
#else
    (void)n;
    return 1;
#endif
}
