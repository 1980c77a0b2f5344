/*
 * pulse_oracle.c -- plain, slow, obviously-correct CPU oracle for the
 * compute-visible weight-delta path (encode / apply / XOR mask / XOR apply).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no header, helper, table or constant with the
 * CUDA path.
 *
 * Every function is the plain definition of the step, one element at a time,
 * in ascending index order, with no blocking, fusion or reordering.
 *
 * Sources (web pages, cited by title and section):
 *  [TALK]  "Taking Reinforcement Learning Cross Datacenter" -- Nan Jiang,
 *          Modal (talk transcript), timecodes 07:24-08:20 (BF16 view, ULP and
 *          rounding boundary), 10:49-11:30 (project to the serving dtype,
 *          compare version t-1 with t, patch = positions + replacement bits,
 *          selective overrides or XOR, bitwise reconstruction).
 *  [PULSE] "Riepilogo Tecnico" of arXiv 2602.03839 (PULSE), sections
 *          "Osservazione Centrale: Sparsita Visibile al Calcolo" (threshold
 *          about |w|/256) and "Metodologia: PULSE -- 1. PULSESync" (compare
 *          consecutive BF16 checkpoints, send indices + new values, apply the
 *          absolute values, bit-identical to a full checkpoint).
 *  [XOR]   "GPU agirlik isinlanmasi RL sampler'larini 4 saniyenin altinda ..."
 *          (humansand.ai summary), section "XOR maskeleri ile delta
 *          senkronizasyonu" (mask = bitwise XOR of pre- and post-step weights,
 *          same size as the weights; the sampler XORs it in).
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes):
 *  - the cast is IEEE-754 roundTiesToEven; subnormals are kept, overflow of
 *    the largest finite values goes to infinity, the sign of zero is kept;
 *  - every NaN input maps to the quiet NaN 0x7FC0 (sign and payload dropped);
 *  - "changed" is a comparison of the 16-bit patterns (so +0 -> -0 counts);
 *  - the patch lists changed positions in ascending order, indices are
 *    uint32 and tensor-local, values are the new absolute BF16 bits;
 *  - encode and xor_mask both leave prev equal to the new BF16 view.
 *
 * Parity pins: all functions are pinned by the CPU tests (exhaustive cast
 * against torch's CPU cast and against exact rational rounding, the pages'
 * worked values at theta = 1, brute force over tiny special-value inputs,
 * the reconstruction and XOR involution invariants). No function here is
 * parity-unpinned.
 */
#include <stdint.h>
#include <string.h>

static uint32_t f32_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/*
 * FP32 bit pattern -> BF16 bit pattern, round to nearest, ties to even.
 * [TALK] 07:24-08:20: the forward pass reads a BF16 view of the FP32 master;
 * [PULSE] "Osservazione Centrale": updates below the BF16 rounding cell are
 * absorbed by the cast.
 *
 * BF16 keeps the top 16 bits of the FP32 pattern. The 16 dropped bits are
 * the remainder r; the kept value is the truncation toward zero. Compared
 * with half of one BF16 ULP (r = 0x8000):
 *   r <  half: keep the truncation;
 *   r >  half: step one BF16 ULP away from zero;
 *   r == half: tie, step away from zero only if the kept pattern is odd.
 * Stepping away from zero is +1 on the magnitude bits, which carries into
 * the exponent at a binade edge and reaches 0x7F80 (infinity) above the
 * largest finite BF16, as roundTiesToEven with an unbounded exponent
 * prescribes.
 */
uint16_t oracle_bf16_rne(uint32_t u)
{
    uint32_t magnitude = u & 0x7FFFFFFFu;
    if (magnitude > 0x7F800000u)            /* NaN: canonical quiet NaN */
        return (uint16_t)0x7FC0u;
    if (magnitude == 0x7F800000u)           /* +-infinity stays infinity */
        return (uint16_t)(u >> 16);

    uint32_t kept = u >> 16;                /* sign + exponent + 7 mantissa bits */
    uint32_t remainder = u & 0xFFFFu;
    int step_up;
    if (remainder > 0x8000u)
        step_up = 1;
    else if (remainder < 0x8000u)
        step_up = 0;
    else
        step_up = (int)(kept & 1u);         /* tie: go to the even neighbour */
    return (uint16_t)(kept + (uint32_t)step_up);
}

void oracle_bf16_rne_array(const uint32_t *bits, uint16_t *out, uint64_t n)
{
    for (uint64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_rne(bits[i]);
}

/*
 * Trainer-side encode. [TALK] 10:49-11:08: project the weights to the
 * serving dtype, compare version t-1 with version t, the patch is the changed
 * positions plus replacement bits. [PULSE] "1. PULSESync": only the indices
 * and new values of parameters whose BF16 value changed are sent.
 *
 * For i = 0 .. n-1 in order: b = rne(master[i]); if b differs from prev[i]
 * bit for bit, append (i, b) to the patch and store b into prev[i].
 * Returns k, the number of patch entries. idx_out / val_out need room for
 * n entries.
 */
uint64_t oracle_encode(const float *master, uint16_t *prev, uint64_t n,
                       uint32_t *idx_out, uint16_t *val_out)
{
    uint64_t k = 0;
    for (uint64_t i = 0; i < n; ++i) {
        uint16_t b = oracle_bf16_rne(f32_bits(master[i]));
        if (b != prev[i]) {
            idx_out[k] = (uint32_t)i;
            val_out[k] = b;
            ++k;
            prev[i] = b;
        }
    }
    return k;
}

/* Count of changed elements without emitting the patch (same comparison). */
uint64_t oracle_count_changed(const float *master, const uint16_t *prev, uint64_t n)
{
    uint64_t k = 0;
    for (uint64_t i = 0; i < n; ++i)
        if (oracle_bf16_rne(f32_bits(master[i])) != prev[i])
            ++k;
    return k;
}

/*
 * Sampler-side apply. [TALK] 11:08-11:30 ("selective overrides"; the engine
 * that applies the patch reconstructs the served version bitwise);
 * [PULSE] "1. PULSESync" (patches hold absolute values, applied directly to
 * the local BF16 weights). For j = 0 .. k-1 in order: w[idx[j]] = val[j].
 */
void oracle_apply(uint16_t *w, const uint32_t *idx, const uint16_t *val, uint64_t k)
{
    for (uint64_t j = 0; j < k; ++j)
        w[idx[j]] = val[j];
}

/*
 * XOR mask. [XOR] "XOR maskeleri ile delta senkronizasyonu": the mask is the
 * bitwise XOR of the pre-step and post-step weights, the same size as the
 * weights; 1-bits mark changed bits. Here pre-step = prev, post-step = the
 * new BF16 view; prev is then refreshed to the new view.
 */
void oracle_xor_mask(const float *master, uint16_t *prev, uint64_t n, uint16_t *mask)
{
    for (uint64_t i = 0; i < n; ++i) {
        uint16_t b = oracle_bf16_rne(f32_bits(master[i]));
        mask[i] = (uint16_t)(b ^ prev[i]);
        prev[i] = b;
    }
}

/* XOR apply. [XOR] same section: a sampler holding the old weights XORs the
 * mask in and holds exactly the new weights. w[i] ^= mask[i]. */
void oracle_xor_apply(uint16_t *w, const uint16_t *mask, uint64_t n)
{
    for (uint64_t i = 0; i < n; ++i)
        w[i] = (uint16_t)(w[i] ^ mask[i]);
}
