/*
 * loco_oracle.c -- plain CPU oracle for the PULSELoCo sender step: the
 * compute-visibility gate on FP32 pseudo-gradients with an FP32 error-feedback
 * buffer, and the receiver's sparse accumulation.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no header, helper, table or constant with the
 * CUDA path.
 *
 * Source: "Riepilogo Tecnico" of arXiv 2602.03839 (PULSE), section
 * "Metodologia: PULSE -- 2. PULSELoCo": workers run H local Adam steps from a
 * shared global checkpoint; each forms a pseudo-gradient (the parameter
 * change over the H steps); the compute-visibility gate is applied to these
 * FP32 pseudo-gradients and only entries that would change the BF16
 * representation are synchronised; entries that do not pass are kept in an
 * FP32 error-feedback buffer and revisited in the next round. Section
 * "Prestazioni di PULSELoCo": 3.6-5.2% of the FP32 values are sent per round.
 *
 * Readings (listed with their reasons in the design notes):
 *  - pseudo-gradient d = local - global (the parameter change), FP32;
 *  - candidate u = d + err (error feedback added before the gate), FP32,
 *    each operation rounded to nearest even, no fused multiply-add; a NaN u
 *    is the quiet NaN 0x7FC00000 (the payload of a NaN result differs
 *    between processors, so it is fixed, as the BF16 view fixes it);
 *  - gate: u passes iff RNE_bf16(global + u) differs bitwise from
 *    RNE_bf16(global) (the update would change the BF16 view of the shared
 *    checkpoint), with the BF16 cast of the BF16 encode (every NaN -> 0x7FC0);
 *  - a passing entry is sent as (index, u) and its error becomes +0; a
 *    failing entry keeps u as its error;
 *  - sent entries are in ascending index order;
 *  - the receiver adds the sent values: acc[idx] += val, in FP32.
 *
 * Parity pins: the CPU tests pin the gate against numpy FP32 arithmetic and
 * torch's BF16 cast, conservation (sent + new error = d + old error, exactly),
 * the visibility floor, accumulation of sub-threshold updates over rounds,
 * and brute force over special values. No function here is parity-unpinned.
 */
#include <stdint.h>
#include <string.h>

static uint32_t bits_of(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

static float canonical_nan(void)
{
    const uint32_t q = 0x7FC00000u;
    float f;
    memcpy(&f, &q, sizeof f);
    return f;
}

/* FP32 bits -> BF16 bits, round to nearest even, every NaN -> 0x7FC0
 * (the same rule as the BF16 encode oracle, restated here). */
static uint16_t bf16_view(float f)
{
    uint32_t u = bits_of(f);
    uint32_t mag = u & 0x7FFFFFFFu;
    if (mag > 0x7F800000u)
        return 0x7FC0u;
    uint32_t kept = u >> 16, rem = u & 0xFFFFu;
    int up = rem > 0x8000u || (rem == 0x8000u && (kept & 1u));
    return (uint16_t)(kept + (uint32_t)up);
}

/*
 * The gate over i = 0 .. n-1 in order. Writes the passing entries to
 * idx_out/val_out (room for n) and returns their number; updates err.
 */
uint64_t oracle_loco_gate(const float *global, const float *local, float *err, uint64_t n,
                          uint32_t *idx_out, float *val_out)
{
    uint64_t k = 0;
    for (uint64_t i = 0; i < n; ++i) {
        /* built with -ffp-contract=off: each operation rounds once */
        float d = local[i] - global[i];
        float u = d + err[i];
        if (u != u)
            u = canonical_nan();
        float s = global[i] + u;
        if (bf16_view(s) != bf16_view(global[i])) {
            idx_out[k] = (uint32_t)i;
            val_out[k] = u;
            ++k;
            err[i] = 0.0f;
        } else {
            err[i] = u;
        }
    }
    return k;
}

/* Receiver: acc[idx[j]] += val[j] for j = 0 .. k-1 in order, FP32. */
void oracle_loco_accumulate(float *acc, const uint32_t *idx, const float *val, uint64_t k)
{
    for (uint64_t j = 0; j < k; ++j) {
        acc[idx[j]] = acc[idx[j]] + val[j];
    }
}
