/*
 * pack_oracle.c -- plain CPU oracle for the codec-friendly packing of patch
 * indices (gap + bit-packing) and its inverse.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no header, helper, table or constant with the
 * CUDA path.
 *
 * Sources: "Riepilogo Tecnico" of arXiv 2602.03839 (PULSE), "1. PULSESync --
 * Compressione": the sparse patches are further compressed with general
 * codecs (zstd); humansand.ai summary, "Pipeline'i GPU'lara tasimak": byte-
 * oriented LZ77-style codecs (LZ4 on nvCOMP) without an entropy stage, and
 * trainer-side compression latency that ate the gains of the naive path.
 * The pages leave the index representation open; this format turns the
 * ascending indices into small, byte-aligned numbers before such a codec.
 *
 * Format (the reading, listed with its reason in the design notes), for k
 * strictly ascending uint32 indices:
 *  - blocks of 128 entries (the last may be shorter); block i starts at
 *    entry 128 i; firsts[i] = its first index;
 *  - its gaps: slot s (s = 0 .. count-2) holds idx[128i + s + 1] -
 *    idx[128i + s] - 1 (>= 0);
 *  - widths[i] = b, the bit length of the largest gap of the block (0 when
 *    every gap is 0 or the block has one entry);
 *  - the block's payload is 16 b bytes (128 slots of b bits): slot s occupies
 *    bits [s b, s b + b) of the payload read as one little-endian bit string
 *    (bit t is bit t % 8 of byte t / 8); unused bits are 0;
 *  - payloads are stored back to back in block order; chunk_off[c] is the
 *    byte offset of block 32 c's payload (chunks of 32 blocks = 4096 entries),
 *    so a chunk can be decoded without reading the others.
 *
 * Parity pins: the CPU tests check the packed bytes against a hand-made
 * example, widths and offsets against numpy, the bit layout against
 * numpy.unpackbits, and the round trip. No function here is parity-unpinned.
 */
#include <stdint.h>
#include <string.h>

#define PACK_BLOCK 128
#define PACK_CHUNK_BLOCKS 32

static uint32_t bit_length(uint32_t v)
{
    uint32_t b = 0;
    while (v) {
        ++b;
        v >>= 1;
    }
    return b;
}

/* Returns the payload size in bytes. payload needs room for 16 * 32 bytes
 * per block (the widest case). */
uint64_t oracle_pack_indices(const uint32_t *idx, uint64_t k, uint32_t *firsts, uint8_t *widths,
                             uint64_t *chunk_off, uint8_t *payload)
{
    uint64_t nblocks = (k + PACK_BLOCK - 1) / PACK_BLOCK;
    uint64_t off = 0;
    for (uint64_t i = 0; i < nblocks; ++i) {
        uint64_t start = i * PACK_BLOCK;
        uint64_t count = k - start < PACK_BLOCK ? k - start : PACK_BLOCK;
        uint32_t maxgap = 0;
        for (uint64_t s = 0; s + 1 < count; ++s) {
            uint32_t gap = idx[start + s + 1] - idx[start + s] - 1u;
            if (gap > maxgap)
                maxgap = gap;
        }
        uint32_t b = bit_length(maxgap);
        firsts[i] = idx[start];
        widths[i] = (uint8_t)b;
        if (i % PACK_CHUNK_BLOCKS == 0)
            chunk_off[i / PACK_CHUNK_BLOCKS] = off;
        uint8_t *p = payload + off;
        memset(p, 0, 16u * b);
        for (uint64_t s = 0; s + 1 < count; ++s) {
            uint32_t gap = idx[start + s + 1] - idx[start + s] - 1u;
            for (uint32_t t = 0; t < b; ++t) {        /* one bit at a time */
                if ((gap >> t) & 1u) {
                    uint64_t bit = s * b + t;
                    p[bit / 8] = (uint8_t)(p[bit / 8] | (1u << (bit % 8)));
                }
            }
        }
        off += 16u * b;
    }
    return off;
}

/* Inverse: rebuilds the k indices. */
void oracle_unpack_indices(const uint32_t *firsts, const uint8_t *widths,
                           const uint64_t *chunk_off, const uint8_t *payload, uint64_t k,
                           uint32_t *idx_out)
{
    uint64_t nblocks = (k + PACK_BLOCK - 1) / PACK_BLOCK;
    uint64_t off = 0;
    for (uint64_t i = 0; i < nblocks; ++i) {
        if (i % PACK_CHUNK_BLOCKS == 0)
            off = chunk_off[i / PACK_CHUNK_BLOCKS];
        uint64_t start = i * PACK_BLOCK;
        uint64_t count = k - start < PACK_BLOCK ? k - start : PACK_BLOCK;
        uint32_t b = widths[i];
        const uint8_t *p = payload + off;
        uint32_t cur = firsts[i];
        idx_out[start] = cur;
        for (uint64_t s = 0; s + 1 < count; ++s) {
            uint32_t gap = 0;
            for (uint32_t t = 0; t < b; ++t) {
                uint64_t bit = s * b + t;
                gap |= (uint32_t)((p[bit / 8] >> (bit % 8)) & 1u) << t;
            }
            cur = cur + gap + 1u;
            idx_out[start + s + 1] = cur;
        }
        off += 16u * b;
    }
}
