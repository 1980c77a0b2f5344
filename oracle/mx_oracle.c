/*
 * mx_oracle.c -- plain CPU oracle for the block-scaled FP8 (MXFP8) serving
 * view: quantize, encode (changed codes and changed block scales) and apply.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no header, helper, table or constant with the
 * CUDA path.
 *
 * Sources:
 *  [TALK]  "Taking Reinforcement Learning Cross Datacenter" -- Nan Jiang,
 *          Modal (talk transcript), 13:06-14:40: rollouts are often served in
 *          lower precision than BF16 (FP8, MXFP4, NVFP4); for a plain float
 *          format the visibility floor is about theta / 2^(mantissa bits + 1);
 *          with a shared group scale a scale change moves a whole group; an
 *          FP8-served run changed about 0.15% of weights per step early and
 *          about 0.05% later.
 *  [PULSE] "Riepilogo Tecnico" of arXiv 2602.03839 (PULSE), "Potenziale
 *          Futuro": FP8 and MXFP4 views should be sparser still (coarser
 *          rounding cells); "1. PULSESync": the patch carries the indices and
 *          new absolute values of what changed in the served view.
 *  [MX]    OCP "Microscaling Formats (MX) Specification" v1.0: MXFP8 = blocks
 *          of 32 elements sharing one E8M0 scale X = 2^e; e = floor(log2 of the
 *          block's largest magnitude) - emax of the element format (8 for
 *          E4M3); each element is the FP8 E4M3 encoding of V / X, values past
 *          the largest normal clamped to it. E4M3 here is the OCP 8-bit float
 *          with bias 7, no infinities, NaN = S.1111.111, largest normal 448.
 *
 * Readings where the pages and the specification leave a choice (each is
 * listed with its reason in the design notes):
 *  - the FP8 serving view is MXFP8 (E4M3 elements, 32 consecutive elements of
 *    a tensor per scale, the last block of a tensor may be shorter);
 *  - element rounding is round-to-nearest, ties to even, subnormals kept, and
 *    magnitudes at or above 448 after scaling become 448 (sign kept);
 *  - a block whose largest magnitude is 0 gets the smallest scale, 2^-127
 *    (E8M0 byte 0); a scale below 2^-127 is raised to 2^-127;
 *  - a block holding a NaN or an infinity gets the NaN scale (byte 0xFF) and
 *    every element of it the code 0x7F;
 *  - the patch has two segments: changed element codes (tensor-local element
 *    index, new code) and changed block scales (tensor-local block index,
 *    new scale byte), each in ascending index order; encode refreshes both
 *    previous arrays.
 *
 * Every function is the plain definition, one block and one element at a
 * time, in ascending order, computed in double precision where the value is
 * exact (an FP32 value times a power of two).
 *
 * Parity pins: the CPU tests pin the element rounding against torch's CPU
 * float8_e4m3fn cast below the saturation point and against an independent
 * decoder of all 256 codes, the saturation and scale rules against closed
 * forms, and encode/apply against brute force and the reconstruction
 * invariants. No function here is parity-unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define MX_BLOCK 32
#define E4M3_EMAX 8          /* exponent of the largest normal, 448 = 1.75 * 2^8 */
#define E4M3_BIAS 7
#define E8M0_BIAS 127

/* Round a non-negative double to the nearest integer, ties to even. */
static double round_half_even(double q)
{
    double fl = floor(q);
    double rem = q - fl;            /* exact: q has few significant bits */
    if (rem > 0.5)
        return fl + 1.0;
    if (rem < 0.5)
        return fl;
    return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

/*
 * Finite double y (exactly an FP32 value times a power of two) -> E4M3 code,
 * round to nearest even, clamped to +-448.
 * Grid: subnormals m * 2^-9 (m = 0..7, exponent field 0); normals
 * (1 + m/8) * 2^(E-7) for exponent field E = 1..15 (E = 15, m = 7 is NaN).
 */
uint8_t oracle_e4m3_rne(double y)
{
    uint8_t sign = signbit(y) ? 0x80u : 0x00u;
    double a = fabs(y);
    if (a >= 448.0)                             /* rounds to 448 or past it */
        return (uint8_t)(sign | 0x7Eu);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; a result of 8 is 2^-6, the
         * smallest normal, whose code is also 8 (exponent field 1, m = 0) */
        double r = round_half_even(ldexp(a, 9));
        return (uint8_t)(sign | (uint8_t)r);
    }
    int ex;
    (void)frexp(a, &ex);                        /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                             /* floor(log2 a), -6 .. 8 */
    double r = round_half_even(ldexp(a, 3 - e)); /* 8 .. 16 */
    if (r == 16.0) {                            /* rounded up into the next binade */
        r = 8.0;
        e += 1;
    }
    return (uint8_t)(sign | (uint8_t)((e + E4M3_BIAS) << 3) | (uint8_t)(r - 8.0));
}

/*
 * E8M0 scale of one block of len (1..32) FP32 values, [MX]:
 * e = floor(log2(max |v|)) - 8, limited to [-127, 127]; returns e + 127.
 * Non-finite block: 0xFF. All-zero block: 0 (the smallest scale).
 */
uint8_t oracle_mx_block_scale(const float *v, uint64_t len)
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
    int e = (ex - 1) - E4M3_EMAX;
    if (e < -127)
        e = -127;
    if (e > 127)
        e = 127;
    return (uint8_t)(e + E8M0_BIAS);
}

/* Codes of one block given its scale byte. */
static void mx_block_codes(const float *v, uint64_t len, uint8_t scale, uint8_t *codes)
{
    for (uint64_t i = 0; i < len; ++i) {
        if (scale == 0xFFu) {
            codes[i] = 0x7Fu;
            continue;
        }
        double y = ldexp((double)v[i], E8M0_BIAS - (int)scale);   /* V / X, exact */
        codes[i] = oracle_e4m3_rne(y);
    }
}

/* The MXFP8 view of a whole tensor: codes[n], scales[ceil(n / 32)]. */
void oracle_mxfp8_quantize(const float *master, uint64_t n, uint8_t *codes, uint8_t *scales)
{
    for (uint64_t b = 0; b * MX_BLOCK < n; ++b) {
        uint64_t start = b * MX_BLOCK;
        uint64_t len = n - start < MX_BLOCK ? n - start : MX_BLOCK;
        scales[b] = oracle_mx_block_scale(master + start, len);
        mx_block_codes(master + start, len, scales[b], codes + start);
    }
}

/*
 * Trainer-side encode of the MXFP8 view ([TALK] 10:49-11:08 and 13:06-13:59,
 * [PULSE] "1. PULSESync"). Block by block in ascending order, compute the
 * block's new scale and codes, then
 *  - for each element i of the block in order: if the new code differs from
 *    prev_codes[i], append (i, code) to the code segment and store it into
 *    prev_codes[i];
 *  - if the new scale differs from prev_scales[b], append (b, scale) to the
 *    scale segment and store it.
 * Each segment is therefore in ascending index order.
 * counts[0] = code entries, counts[1] = scale entries. idx/val need room for
 * n entries, sidx/sval for nblocks.
 */
void oracle_mxfp8_encode(const float *master, uint8_t *prev_codes, uint8_t *prev_scales,
                         uint64_t n, uint32_t *idx, uint8_t *val, uint32_t *sidx,
                         uint8_t *sval, uint64_t *counts)
{
    uint64_t k = 0, ks = 0;
    uint8_t codes[MX_BLOCK];
    for (uint64_t b = 0; b * MX_BLOCK < n; ++b) {
        uint64_t start = b * MX_BLOCK;
        uint64_t len = n - start < MX_BLOCK ? n - start : MX_BLOCK;
        uint8_t scale = oracle_mx_block_scale(master + start, len);
        mx_block_codes(master + start, len, scale, codes);
        for (uint64_t i = 0; i < len; ++i) {
            if (codes[i] != prev_codes[start + i]) {
                idx[k] = (uint32_t)(start + i);
                val[k] = codes[i];
                ++k;
                prev_codes[start + i] = codes[i];
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

/* Sampler-side apply of one byte segment: w[idx[j]] = val[j], j in order. */
void oracle_apply_u8(uint8_t *w, const uint32_t *idx, const uint8_t *val, uint64_t k)
{
    for (uint64_t j = 0; j < k; ++j)
        w[idx[j]] = val[j];
}
