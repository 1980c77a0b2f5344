/*
 * compose_oracle.c -- plain CPU oracle for patch-chain composition (the
 * sidecar's catch-up over several missing versions).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no header, helper, table or constant with the
 * CUDA path.
 *
 * Sources:
 *  [TALK]  "Taking Reinforcement Learning Cross Datacenter" -- Nan Jiang,
 *          Modal (talk transcript), 16:40-17:04: a sidecar makes a rollout
 *          engine version-aware; if the engine is behind but can catch up,
 *          the sidecar applies the missing transitions.
 *  [KR]    Korean write-up of the same talk, section "Cross-Globe RL을 위한
 *          Version-Aware Rollout Architecture" (the same three cases).
 *  [PULSE] "Riepilogo Tecnico" of arXiv 2602.03839, "1. PULSESync": a patch
 *          holds absolute new values, so applying it overwrites and never
 *          accumulates.
 *
 * Reading (listed with its reason in the design notes): catching up over
 * versions t -> t+1 -> ... -> t+m applies m patches in order; because entries
 * are absolute values, the same result comes from ONE patch that holds the
 * union of the indices with, for each index, the value of the latest patch
 * that lists it (last writer wins). compose(A, B) builds that patch for A
 * followed by B; a chain folds left. The result lists each index once, in
 * ascending order.
 *
 * Parity pins: the CPU tests check compose against a dictionary built in
 * Python, against applying the patches one after another with numpy fancy
 * assignment, and against the encode of the whole span; see the design notes.
 * No function here is parity-unpinned.
 */
#include <stdint.h>

/*
 * compose(A, B), 16-bit values. A and B each list strictly ascending indices.
 * Two-pointer merge: the smaller index goes first; on an equal index the
 * entry of B (the later patch) is taken and A's is dropped. Returns the
 * number of entries written (room for ka + kb is needed).
 */
uint64_t oracle_compose(const uint32_t *idx_a, const uint16_t *val_a, uint64_t ka,
                        const uint32_t *idx_b, const uint16_t *val_b, uint64_t kb,
                        uint32_t *idx_out, uint16_t *val_out)
{
    uint64_t i = 0, j = 0, k = 0;
    while (i < ka || j < kb) {
        if (j == kb || (i < ka && idx_a[i] < idx_b[j])) {
            idx_out[k] = idx_a[i];
            val_out[k] = val_a[i];
            ++i;
        } else if (i == ka || idx_b[j] < idx_a[i]) {
            idx_out[k] = idx_b[j];
            val_out[k] = val_b[j];
            ++j;
        } else {                     /* same index: the later patch wins */
            idx_out[k] = idx_b[j];
            val_out[k] = val_b[j];
            ++i;
            ++j;
        }
        ++k;
    }
    return k;
}

/* The same for 8-bit values (the code or scale segment of an MXFP8 patch). */
uint64_t oracle_compose_u8(const uint32_t *idx_a, const uint8_t *val_a, uint64_t ka,
                           const uint32_t *idx_b, const uint8_t *val_b, uint64_t kb,
                           uint32_t *idx_out, uint8_t *val_out)
{
    uint64_t i = 0, j = 0, k = 0;
    while (i < ka || j < kb) {
        if (j == kb || (i < ka && idx_a[i] < idx_b[j])) {
            idx_out[k] = idx_a[i];
            val_out[k] = val_a[i];
            ++i;
        } else if (i == ka || idx_b[j] < idx_a[i]) {
            idx_out[k] = idx_b[j];
            val_out[k] = val_b[j];
            ++j;
        } else {
            idx_out[k] = idx_b[j];
            val_out[k] = val_b[j];
            ++i;
            ++j;
        }
        ++k;
    }
    return k;
}
