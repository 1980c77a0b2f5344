/*
 * mxfp4_oracle.c -- plain CPU oracle for the block-scaled FP4 (MXFP4) serving
 * view: quantize, encode (changed code bytes and changed block scales) and
 * the byte apply it shares with the MXFP8 oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no header, helper, table or constant with the
 * CUDA path.
 *
 * Sources:
 *  [TALK]  "Taking Reinforcement Learning Cross Datacenter" -- Nan Jiang,
 *          Modal (talk transcript), 13:06-14:40: rollouts are served in MXFP4
 *          or NVFP4 as well as FP8; in a group-scaled format each weight is
 *          quantized against a shared group scale, and a scale change moves
 *          the whole group.
 *  [KR]    Korean write-up of the talk, section on lower-precision serving:
 *          MXFP4-style formats quantize against a shared group scale, so the
 *          scale itself shapes the patch.
 *  [PULSE] "Riepilogo Tecnico" of arXiv 2602.03839 (PULSE), "Potenziale
 *          Futuro": MXFP4 views should be sparser still; "1. PULSESync": the
 *          patch carries positions and new absolute values.
 *  [MX]    OCP "Microscaling Formats (MX) Specification" v1.0: MXFP4 = blocks
 *          of 32 elements sharing one E8M0 scale X = 2^e; e = floor(log2 of
 *          the block's largest magnitude) - emax of the element format (2 for
 *          E2M1); each element is the FP4 E2M1 encoding of V / X. E2M1: sign,
 *          2 exponent bits (bias 1), 1 mantissa bit, no infinities or NaN,
 *          magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 *
 * Readings where the pages and the specification leave a choice (each is
 * listed with its reason in the design notes):
 *  - element rounding is round-to-nearest, ties to the even code (mantissa
 *    bit 0), magnitudes at or above 6 after scaling become 6, the sign is
 *    kept (a negative value that rounds to zero gives code 0x8);
 *  - scales follow the MXFP8 reading: an all-zero block gets byte 0, a scale
 *    below 2^-127 is raised to it, a block holding a NaN or an infinity gets
 *    the NaN scale 0xFF; its element codes are all 0;
 *  - codes are stored two per byte, element 2j in the low nibble of byte j
 *    and element 2j + 1 in the high nibble (a tensor of odd length has a
 *    zero high nibble in its last byte);
 *  - the serving view changes byte by byte, so the code segment of a patch
 *    lists changed BYTES (byte index, new byte); the scale segment lists
 *    changed scales (block index, new byte); both ascending.
 *
 * Every function is the plain definition, one block and one element at a
 * time, in ascending order, in double precision (a value times a power of
 * two is exact there).
 *
 * Parity pins: the CPU tests pin the element rounding against a brute-force
 * nearest-value search over the 16 codes and an independent decoder, the
 * scale rule against closed forms and a brute-force exponent search, and
 * encode/apply against the reconstruction invariants. No function here is
 * parity-unpinned.
 */
#include <math.h>
#include <stdint.h>

#define MX4_BLOCK 32
#define E2M1_EMAX 2          /* exponent of the largest normal, 6 = 1.5 * 2^2 */
#define E2M1_BIAS 1
#define MX4_E8M0_BIAS 127

/* Round a non-negative double to the nearest integer, ties to even. */
static double mx4_round_half_even(double q)
{
    double fl = floor(q);
    double rem = q - fl;
    if (rem > 0.5)
        return fl + 1.0;
    if (rem < 0.5)
        return fl;
    return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

/*
 * Finite double y -> E2M1 code (bit 3 = sign), round to nearest even,
 * clamped to +-6. Grid: exponent field 0 holds 0 and 0.5 (m * 2^-1);
 * exponent field E = 1..3 holds (1 + m/2) * 2^(E-1).
 */
uint8_t oracle_e2m1_rne(double y)
{
    uint8_t sign = signbit(y) ? 0x8u : 0x0u;
    double a = fabs(y);
    if (a >= 6.0)
        return (uint8_t)(sign | 0x7u);
    if (a < 1.0) {
        /* multiples of 0.5; a result of 2 is 1.0, whose code is also 2
         * (exponent field 1, m = 0) */
        double r = mx4_round_half_even(a * 2.0);
        return (uint8_t)(sign | (uint8_t)r);
    }
    int ex;
    (void)frexp(a, &ex);                          /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                               /* floor(log2 a): 0, 1 or 2 */
    double r = mx4_round_half_even(ldexp(a, 1 - e));  /* 2 .. 4 */
    if (r == 4.0) {                               /* rounded up into the next binade */
        r = 2.0;
        e += 1;                                   /* stays <= 2: a < 6 */
    }
    return (uint8_t)(sign | (uint8_t)((e + E2M1_BIAS) << 1) | (uint8_t)(r - 2.0));
}

/*
 * E8M0 scale of one block of len (1..32) FP32 values, [MX]:
 * e = floor(log2(max |v|)) - 2, limited to [-127, 127]; returns e + 127.
 * Non-finite block: 0xFF. All-zero block: 0.
 */
uint8_t oracle_mxfp4_block_scale(const float *v, uint64_t len)
{
    double amax = 0.0;
    for (uint64_t i = 0; i < len; ++i) {
        if (!isfinite(v[i]))
            return 0xFFu;
        double a = fabs((double)v[i]);
        if (a > amax)
            amax = a;
    }
    if (amax == 0.0)
        return 0u;
    int ex;
    (void)frexp(amax, &ex);
    int e = (ex - 1) - E2M1_EMAX;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return (uint8_t)(e + MX4_E8M0_BIAS);
}

/* Element codes (one per byte, low nibble) of one block given its scale. */
static void mx4_block_codes(const float *v, uint64_t len, uint8_t scale, uint8_t *codes)
{
    for (uint64_t i = 0; i < len; ++i) {
        if (scale == 0xFFu) {
            codes[i] = 0u;
            continue;
        }
        double y = ldexp((double)v[i], MX4_E8M0_BIAS - (int)scale);   /* V / X, exact */
        codes[i] = oracle_e2m1_rne(y);
    }
}

/* Packed code byte j of a block from its element codes (len elements). */
static uint8_t mx4_pack(const uint8_t *codes, uint64_t len, uint64_t j)
{
    uint8_t lo = codes[2 * j];
    uint8_t hi = 2 * j + 1 < len ? codes[2 * j + 1] : 0u;
    return (uint8_t)(lo | (hi << 4));
}

/* The MXFP4 view of a tensor: codes[ceil(n / 2)] packed, scales[ceil(n / 32)]. */
void oracle_mxfp4_quantize(const float *master, uint64_t n, uint8_t *codes, uint8_t *scales)
{
    uint8_t c[MX4_BLOCK];
    for (uint64_t b = 0; b * MX4_BLOCK < n; ++b) {
        uint64_t start = b * MX4_BLOCK;
        uint64_t len = n - start < MX4_BLOCK ? n - start : MX4_BLOCK;
        scales[b] = oracle_mxfp4_block_scale(master + start, len);
        mx4_block_codes(master + start, len, scales[b], c);
        for (uint64_t j = 0; 2 * j < len; ++j)
            codes[start / 2 + j] = mx4_pack(c, len, j);
    }
}

/*
 * Trainer-side encode of the MXFP4 view ([TALK] 10:49-11:08 and 13:06-13:59,
 * [PULSE] "1. PULSESync"). Block by block in ascending order: the block's
 * new scale and packed code bytes; each byte that differs from prev_codes is
 * appended (byte index, byte) to the code segment and stored; a changed
 * scale is appended (block index, byte) to the scale segment and stored.
 * counts[0] = code entries, counts[1] = scale entries. idx/val need room for
 * ceil(n / 2) entries, sidx/sval for ceil(n / 32).
 */
void oracle_mxfp4_encode(const float *master, uint8_t *prev_codes, uint8_t *prev_scales,
                         uint64_t n, uint32_t *idx, uint8_t *val, uint32_t *sidx,
                         uint8_t *sval, uint64_t *counts)
{
    uint64_t k = 0, ks = 0;
    uint8_t c[MX4_BLOCK];
    for (uint64_t b = 0; b * MX4_BLOCK < n; ++b) {
        uint64_t start = b * MX4_BLOCK;
        uint64_t len = n - start < MX4_BLOCK ? n - start : MX4_BLOCK;
        uint8_t scale = oracle_mxfp4_block_scale(master + start, len);
        mx4_block_codes(master + start, len, scale, c);
        for (uint64_t j = 0; 2 * j < len; ++j) {
            uint64_t pos = start / 2 + j;
            uint8_t byte = mx4_pack(c, len, j);
            if (byte != prev_codes[pos]) {
                idx[k] = (uint32_t)pos;
                val[k] = byte;
                ++k;
                prev_codes[pos] = byte;
            }
        }
        if (scale != prev_scales[b]) {
            sidx[ks] = (uint32_t)b;
            sval[ks] = scale;
            ++ks;
            prev_scales[b] = scale;
        }
    }
    counts[0] = k;
    counts[1] = ks;
}
