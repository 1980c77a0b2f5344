/*
 * nvfp4_oracle.c -- plain CPU oracle for the NVFP4 serving view: FP4 (E2M1)
 * elements under two levels of scale, an E4M3 scale per 16 elements and an
 * FP32 scale per tensor; quantize and encode (changed code bytes, changed
 * block scales, the new tensor scale).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do. It shares no header, helper, table or constant with the
 * CUDA path.
 *
 * Sources:
 *  [TALK]  "Taking Reinforcement Learning Cross Datacenter" -- Nan Jiang,
 *          Modal (talk transcript), 13:06-14:00: rollouts are served in NVFP4;
 *          NVFP4 has hierarchical scales, and the same sparsity is observed.
 *  [XOR]   humansand.ai summary "GPU agirlik isinlanmasi ...", section
 *          "Bildirilen sayilar": the proxy
 *          workload is an NVFP4 checkpoint of which 0.085 % changes per step.
 *  The pages name the format but do not define it. The reading below is the
 *  publicly described NVFP4 layout (NVIDIA's Blackwell microscaling format):
 *  blocks of 16 consecutive elements, an unsigned E4M3 block scale, an FP32
 *  scale per tensor chosen so that the largest block scale fits E4M3.
 *
 * Reading (each choice is listed with its reason in the design notes). All
 * arithmetic is FP32, each operation rounded to nearest even, in this order:
 *  - A = the largest magnitude over the tensor's finite elements (0 if none);
 *    tensor scale S = A / 2688 (2688 = 448 * 6: E4M3's and E2M1's largest
 *    normals);
 *  - a block holding a NaN or an infinity gets the block scale byte 0x7F
 *    (E4M3 NaN) and every code 0;
 *  - otherwise a_b = the block's largest magnitude, u = (a_b / 6) / S, and the
 *    block scale byte d = E4M3 of u (round to nearest even, values past 448
 *    clamped to 448); d = 0 when S is 0;
 *  - element scale x = dec(d) * S, r = 1 / x, and each element's code is the
 *    E2M1 of v * r (round to nearest even, ties to the even code, past 6
 *    clamped to 6, sign kept); when d is 0, or x is 0 or r is not finite, the
 *    block's codes are all 0;
 *  - codes two per byte as in the MXFP4 view (element 2j in the low nibble);
 *    the patch lists changed code bytes and changed block scales, ascending,
 *    and carries the new tensor scale.
 *
 * Parity pins: the CPU tests pin the FP32 arithmetic against numpy float32
 * operations written independently, the E4M3 decoder against the format
 * definition and against torch's float8_e4m3fn, the element rounding against
 * the MXFP4 view's brute-force pins, and encode/apply against the
 * reconstruction invariants. No function here is parity-unpinned.
 */
#include <math.h>
#include <stdint.h>

#define NV_BLOCK 16

uint8_t oracle_e4m3_rne(double y);   /* mx_oracle.c */
uint8_t oracle_e2m1_rne(double y);   /* mxfp4_oracle.c */

/* Value of an E4M3 code (bias 7, subnormals m * 2^-9, no infinities). */
static float nv_e4m3_value(uint8_t c)
{
    int e = (c >> 3) & 0xF, m = c & 0x7;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return (float)((c & 0x80) ? -v : v);
}

/* Tensor scale S = A / 2688 of a tensor of n FP32 values. */
float oracle_nvfp4_tensor_scale(const float *v, uint64_t n)
{
    float amax = 0.0f;
    for (uint64_t i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (isfinite(a) && a > amax)
            amax = a;
    }
    return amax / 2688.0f;
}

/* Block scale byte and element codes (one per byte, low nibble) of one block
 * of len (1..16) values under tensor scale S. */
static uint8_t nv_block(const float *v, uint64_t len, float S, uint8_t *codes)
{
    float amax = 0.0f;
    int finite = 1;
    for (uint64_t i = 0; i < len; ++i) {
        if (!isfinite(v[i]))
            finite = 0;
        float a = fabsf(v[i]);
        if (a > amax)
            amax = a;
    }
    for (uint64_t i = 0; i < len; ++i)
        codes[i] = 0;
    if (!finite)
        return 0x7Fu;
    if (S == 0.0f)
        return 0u;
    volatile float t = amax / 6.0f;      /* each step rounded to FP32 */
    volatile float u = t / S;
    uint8_t d = oracle_e4m3_rne((double)u);
    if (d == 0)
        return 0u;
    volatile float x = nv_e4m3_value(d) * S;
    if (x == 0.0f)
        return d;
    volatile float r = 1.0f / x;
    if (!isfinite(r))
        return d;
    for (uint64_t i = 0; i < len; ++i) {
        volatile float y = v[i] * r;
        codes[i] = oracle_e2m1_rne((double)y);
    }
    return d;
}

static uint8_t nv_pack(const uint8_t *codes, uint64_t len, uint64_t j)
{
    uint8_t lo = codes[2 * j];
    uint8_t hi = 2 * j + 1 < len ? codes[2 * j + 1] : 0u;
    return (uint8_t)(lo | (hi << 4));
}

/* The NVFP4 view of a tensor: codes[ceil(n / 2)], scales[ceil(n / 16)], and
 * the tensor scale (returned). */
float oracle_nvfp4_quantize(const float *master, uint64_t n, uint8_t *codes, uint8_t *scales)
{
    float S = oracle_nvfp4_tensor_scale(master, n);
    uint8_t c[NV_BLOCK];
    for (uint64_t b = 0; b * NV_BLOCK < n; ++b) {
        uint64_t start = b * NV_BLOCK;
        uint64_t len = n - start < NV_BLOCK ? n - start : NV_BLOCK;
        scales[b] = nv_block(master + start, len, S, c);
        for (uint64_t j = 0; 2 * j < len; ++j)
            codes[start / 2 + j] = nv_pack(c, len, j);
    }
    return S;
}

/*
 * Trainer-side encode of the NVFP4 view ([TALK] 10:49-11:08 and 13:06-14:00):
 * the new view block by block in ascending order; each code byte that
 * differs from prev_codes is appended (byte index, byte) and stored; a
 * changed block scale is appended (block index, byte) and stored. counts[0]
 * = code entries, counts[1] = scale entries; returns the new tensor scale.
 * idx/val need room for ceil(n / 2) entries, sidx/sval for ceil(n / 16).
 */
float oracle_nvfp4_encode(const float *master, uint8_t *prev_codes, uint8_t *prev_scales,
                          uint64_t n, uint32_t *idx, uint8_t *val, uint32_t *sidx, uint8_t *sval,
                          uint64_t *counts)
{
    float S = oracle_nvfp4_tensor_scale(master, n);
    uint64_t k = 0, ks = 0;
    uint8_t c[NV_BLOCK];
    for (uint64_t b = 0; b * NV_BLOCK < n; ++b) {
        uint64_t start = b * NV_BLOCK;
        uint64_t len = n - start < NV_BLOCK ? n - start : NV_BLOCK;
        uint8_t d = nv_block(master + start, len, S, c);
        for (uint64_t j = 0; 2 * j < len; ++j) {
            uint64_t pos = start / 2 + j;
            uint8_t byte = nv_pack(c, len, j);
            if (byte != prev_codes[pos]) {
                idx[k] = (uint32_t)pos;
                val[k] = byte;
                ++k;
                prev_codes[pos] = byte;
            }
        }
        if (d != prev_scales[b]) {
            sidx[ks] = (uint32_t)b;
            sval[ks] = d;
            ++ks;
            prev_scales[b] = d;
        }
    }
    counts[0] = k;
    counts[1] = ks;
    return S;
}
