/*
 * pulse.h -- C ABI of the GB300 (sm_103a) compute-visible weight-delta
 * library: trainer-side encode of a BF16 patch or XOR mask from FP32 master
 * weights, and sampler-side apply of that patch or mask.
 *
 * Sources (web pages, cited by title and section):
 *  [TALK]  "Taking Reinforcement Learning Cross Datacenter" -- Nan Jiang,
 *          Modal (talk transcript): 07:24-08:20 the forward pass reads a BF16
 *          view of the FP32 master weights, spacing ~theta/128, visibility
 *          boundary ~theta/256; 10:49-11:30 project to the serving dtype,
 *          compare version t-1 with t, the patch is changed positions plus
 *          replacement bits plus metadata, applied as selective overrides or
 *          as XOR, reconstructing the served version bitwise.
 *  [PULSE] "Riepilogo Tecnico" of arXiv 2602.03839 (PULSE), section
 *          "Metodologia: PULSE -- 1. PULSESync": compare consecutive BF16
 *          checkpoints, send the indices and new values of the changed
 *          parameters, the sampler applies them to its BF16 weights; absolute
 *          values make the result bit-identical to a full checkpoint.
 *  [XOR]   humansand.ai summary "GPU agirlik isinlanmasi RL sampler'larini
 *          4 saniyenin altinda ...", sections "XOR maskeleri ile delta
 *          senkronizasyonu" (mask = XOR of pre- and post-step weights, same
 *          size as the weights, XOR-ed in place by the sampler) and
 *          "Pipeline'i GPU'lara tasimak" (one kernel launch covers the whole
 *          model, with tiling and address-map metadata prepared on the CPU).
 *  [MX]    OCP "Microscaling Formats (MX) Specification" v1.0 (not one of
 *          the pages): the MXFP8 format of the lower-precision view.
 *  [KR]    Korean write-up of the talk, section "Cross-Globe RL을 위한
 *          Version-Aware Rollout Architecture" (sidecar catch-up).
 *  [PPLX]  "Weight transfer for RL post-training in under 2 seconds"
 *          (Perplexity), section "Statyczny harmonogram": the transfer
 *          schedule is computed once at initialisation and replayed each step.
 *
 * Conventions shared by every entry point:
 *  - BF16 data (prev, w, val, mask) is passed as uint16_t bit patterns.
 *  - Unless a parameter says "host", every pointer is DEVICE memory of the
 *    CUDA device that is current on the calling thread. The caller owns all
 *    buffers and keeps them alive until `stream` has passed the call.
 *  - All calls are asynchronous on `stream` (0 = legacy default stream) and
 *    return a status code synchronously. A non-zero status from argument
 *    checking means nothing was launched. Device-side errors (a wait that
 *    gave up, an out-of-range patch index) are recorded in a device error
 *    word and reported by pulse_get_error / pulse_plan_get_error.
 *  - Element counts n are < 2^32 (patch indices are uint32, tensor-local).
 *  - The cast is IEEE round-to-nearest-even; subnormals are kept; values past
 *    the largest finite BF16 round to infinity; every NaN becomes 0x7FC0.
 *  - "Changed" compares 16-bit patterns, so +0 -> -0 is a change.
 *  - Output buffers must not overlap input buffers; prev and w are updated in
 *    place.
 *  - No call prints, aborts, traps or throws.
 */
#ifndef PULSE_H
#define PULSE_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define PULSE_OK           0  /* success */
#define PULSE_ERR_INVALID  1  /* null pointer where one is required, bad count, overlap */
#define PULSE_ERR_RANGE    2  /* an element count is >= 2^32 (past PULSE_NOALLOC_MAX_ELEMS for pulse_encode_noalloc) */
#define PULSE_ERR_CUDA     3  /* a CUDA runtime call or kernel launch failed */
#define PULSE_ERR_TIMEOUT  4  /* device: a bounded wait gave up; outputs of that call are invalid */
#define PULSE_ERR_INDEX    5  /* device: a checked apply met an index >= n and skipped it */
#define PULSE_ERR_NOMEM    6  /* workspace allocation failed */

/* Human-readable name of a status code (static storage, never NULL). */
const char *pulse_error_string(int status);

/* Elements per encode tile (compile-time constant of this build). */
uint32_t pulse_encode_tile_elems(void);

/*
 * pulse_encode -- trainer-side encode of one tensor. [TALK] 10:49-11:08,
 * [PULSE] "1. PULSESync".
 *
 * For every i in [0, n): b = RNE_bf16(master_f32[i]); if b differs bitwise
 * from prev_bf16[i], the pair (i, b) is part of the patch and prev_bf16[i]
 * is set to b. The patch is written densely, in ascending index order:
 * idx_out[0..k) = changed positions, val_out[0..k) = their new absolute BF16
 * bits; *count_out = k (device uint64). prev_bf16 ends equal to the new view.
 *
 *   master_f32  device, n floats, read only
 *   prev_bf16   device, n uint16, read and updated in place
 *   idx_out     device, room for n uint32 (the worst case, all changed)
 *   val_out     device, room for n uint16
 *   count_out   device, one uint64
 *
 * n == 0 writes *count_out = 0 and launches only that write. Uses a library
 * workspace per (device, stream), allocated on first use and grown on demand
 * (growth synchronises `stream`); concurrent calls on one stream are ordered
 * by the stream, calls on different streams use different workspaces.
 * Errors: PULSE_ERR_INVALID (null pointer when n > 0), PULSE_ERR_RANGE
 * (n >= 2^32), PULSE_ERR_NOMEM, PULSE_ERR_CUDA; device: PULSE_ERR_TIMEOUT.
 */
int pulse_encode(const float *master_f32, uint16_t *prev_bf16, uint64_t n,
                 uint32_t *idx_out, uint16_t *val_out, uint64_t *count_out,
                 cudaStream_t stream);

/*
 * pulse_apply -- sampler-side patch apply. [TALK] 11:08-11:30 ("selective
 * overrides"), [PULSE] "1. PULSESync".
 *
 * For j in [0, count): w_bf16[idx[j]] = val[j]. With the patch of an encode
 * (ascending, distinct indices) the result does not depend on order. The
 * caller guarantees idx[j] < size of w_bf16; use pulse_apply_checked when it
 * cannot.
 *
 *   w_bf16  device, updated in place
 *   idx     device, count uint32;  val  device, count uint16
 *   count   HOST value (the receiver knows the patch length)
 * count == 0 launches nothing. Errors: PULSE_ERR_INVALID, PULSE_ERR_CUDA.
 */
int pulse_apply(uint16_t *w_bf16, const uint32_t *idx, const uint16_t *val,
                uint64_t count, cudaStream_t stream);

/*
 * pulse_apply_checked -- as pulse_apply, for a w_bf16 of n elements; an entry
 * with idx[j] >= n is skipped and PULSE_ERR_INDEX is recorded in the device
 * error word of (device, stream), read by pulse_get_error.
 */
int pulse_apply_checked(uint16_t *w_bf16, uint64_t n, const uint32_t *idx,
                        const uint16_t *val, uint64_t count, cudaStream_t stream);

/*
 * pulse_xor_mask -- trainer-side XOR mask of one tensor. [XOR] "XOR maskeleri
 * ile delta senkronizasyonu".
 *
 * For every i in [0, n): b = RNE_bf16(master_f32[i]); mask_out[i] =
 * b ^ prev_bf16[i]; prev_bf16[i] = b. Non-zero mask words are exactly the
 * positions pulse_encode would list.
 *   master_f32 device n floats; prev_bf16 device n uint16 (in/out);
 *   mask_out device n uint16.
 * n == 0 launches nothing. Errors: PULSE_ERR_INVALID, PULSE_ERR_RANGE,
 * PULSE_ERR_CUDA.
 */
int pulse_xor_mask(const float *master_f32, uint16_t *prev_bf16, uint64_t n,
                   uint16_t *mask_out, cudaStream_t stream);

/*
 * pulse_xor_apply -- sampler-side XOR apply. [XOR] same section: w ^= mask
 * on raw bits; applying the same mask twice restores the original.
 *   w_bf16 device n uint16 (in/out); mask device n uint16.
 * n == 0 launches nothing. Errors: PULSE_ERR_INVALID, PULSE_ERR_RANGE,
 * PULSE_ERR_CUDA.
 */
int pulse_xor_apply(uint16_t *w_bf16, const uint16_t *mask, uint64_t n,
                    cudaStream_t stream);

/*
 * Device error word of the (current device, stream) workspace used by the
 * single-tensor calls. Synchronises `stream`, then returns and clears the
 * recorded error: PULSE_OK, PULSE_ERR_TIMEOUT or PULSE_ERR_INDEX (timeout
 * wins if both were recorded), or PULSE_ERR_CUDA if the synchronisation
 * itself failed.
 */
int pulse_get_error(cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Multi-tensor plans. [XOR] "Pipeline'i GPU'lara tasimak": the tile and
 * address map of a whole model is prepared on the host and one kernel launch
 * covers every tensor; [PPLX] "Statyczny harmonogram": the plan is built once
 * and replayed each step.
 *
 * One pulse_tensor per model tensor, in a fixed list order. Fields a given
 * operation does not use may be NULL:
 *   encode_multi     master, prev, idx, val
 *   apply_multi      w, idx, val
 *   xor_mask_multi   master, prev, mask
 *   xor_apply_multi  w, mask
 * idx/val of tensor t hold that tensor's own patch segment (indices local to
 * the tensor): room for n entries where encode_multi writes them or where
 * apply_multi_device reads device counts; for apply_multi with host counts,
 * room for the count applied is enough. n may be 0.
 * ---------------------------------------------------------------------- */
typedef struct pulse_tensor {
    const float *master;  /* device, n floats (trainer) */
    uint16_t *prev;       /* device, n uint16 (trainer, in/out) */
    uint16_t *w;          /* device, n uint16 (sampler, in/out) */
    uint64_t n;           /* elements, < 2^32 */
    uint32_t *idx;        /* device, room for n uint32 (patch segment) */
    uint16_t *val;        /* device, room for n uint16 (patch segment) */
    uint16_t *mask;       /* device, n uint16 (XOR mask) */
} pulse_tensor;

typedef struct pulse_plan pulse_plan;

/*
 * Build a plan for `ntensors` tensors (host array `tensors`, copied). Builds
 * the tile tables on the host, uploads them, and allocates the plan's
 * workspace on the current device; synchronous. *plan_out receives the
 * handle. Errors: PULSE_ERR_INVALID (null arguments, ntensors < 1),
 * PULSE_ERR_RANGE (some n >= 2^32), PULSE_ERR_NOMEM, PULSE_ERR_CUDA.
 */
int pulse_plan_create(const pulse_tensor *tensors, int ntensors, pulse_plan **plan_out);

/* Free a plan (synchronises the device first). NULL is accepted. */
int pulse_plan_destroy(pulse_plan *plan);

/* Number of tensors and total encode tiles of a plan (0 on a NULL plan). */
int pulse_plan_num_tensors(const pulse_plan *plan);
uint64_t pulse_plan_num_tiles(const pulse_plan *plan);

/*
 * Encode every tensor of the plan in one launch; counts_out (device,
 * ntensors uint64) receives each tensor's patch length k_t. Per tensor the
 * result equals pulse_encode on that tensor. Errors: PULSE_ERR_INVALID (a
 * required field is NULL in the plan), PULSE_ERR_CUDA; device:
 * PULSE_ERR_TIMEOUT.
 */
int pulse_encode_multi(pulse_plan *plan, uint64_t *counts_out, cudaStream_t stream);

/*
 * Apply every tensor's patch segment to the whole model. counts_host (HOST,
 * ntensors uint64) gives each segment's length; it is copied before the call
 * returns. One launch (per 16384 tensors) scatters every entry straight into
 * w: consecutive entries of a segment go to consecutive threads, so the
 * partial-sector stores of an ascending segment reach L2 as one request per
 * 32-byte sector, and only the touched sectors of w move (each read once for
 * its untouched bytes and written once). Segments from encode are ascending
 * with distinct indices; in a segment that repeats an index, which of the
 * repeated entries lands is unspecified. Entries with idx >= n are skipped
 * and recorded as PULSE_ERR_INDEX in the plan's error word, and a count
 * larger than its tensor is clamped to n and recorded the same way.
 */
int pulse_apply_multi(pulse_plan *plan, const uint64_t *counts_host, cudaStream_t stream);

/* As pulse_apply_multi with the counts in DEVICE memory (e.g. counts_out of
 * pulse_encode_multi), so no host round trip is needed. */
int pulse_apply_multi_device(pulse_plan *plan, const uint64_t *counts_dev, cudaStream_t stream);

/*
 * pulse_apply_chain_multi -- bring the plan's w forward by several versions
 * at once. [TALK] 16:40-17:04: a sidecar whose engine is behind applies the
 * transitions it missed, in order; [PULSE] "1. PULSESync": patch values are
 * absolute, so the later patch wins where two list the same index.
 *   patches   HOST array of nversions x ntensors references, version-major:
 *             patches[v * ntensors + t] is tensor t's patch of the v-th
 *             version applied (oldest first); copied before the call returns
 *   nversions >= 1
 * The result equals pulse_apply_multi with each version's segments, one
 * version after the other. Each segment must list ascending indices (what
 * encode writes). One pass over w per 16 versions: a chunk of w is loaded
 * once, receives every version's entries in version order, and its changed
 * 32-byte sectors are written back once. Needs w for every tensor with n > 0
 * (idx, val and master of the plan are not used). Growing the call's
 * internal tables synchronises `stream`; one stream at a time per plan.
 * This is the fastest way for a receiver that holds w to catch up: four
 * 8%-dense versions of an 8.03B-parameter model take about 8.2 ms, against
 * about 20 ms for four whole-model applies and 17 ms for composing them with
 * pulse_compose_chain_multi and applying the result. Compose only where the
 * single patch itself is wanted (to send one patch over the network).
 * Errors: PULSE_ERR_INVALID (NULL plan or patches, nversions < 1, a plan
 * tensor without w, count > 0 with NULL idx or val), PULSE_ERR_RANGE (a
 * count >= 2^32), PULSE_ERR_NOMEM, PULSE_ERR_CUDA; device (plan error word):
 * PULSE_ERR_INDEX (count > n, clamped; entries outside their chunk, skipped),
 * PULSE_ERR_TIMEOUT.
 */
typedef struct pulse_patch_ref {
    const uint32_t *idx;  /* device, count entries, ascending, local to the tensor */
    const uint16_t *val;  /* device, count entries (BF16 bit patterns) */
    uint64_t count;       /* host value */
} pulse_patch_ref;

int pulse_apply_chain_multi(pulse_plan *plan, const pulse_patch_ref *patches, int nversions,
                            cudaStream_t stream);

/*
 * pulse_compose_chain_multi -- compose the patches of nversions consecutive
 * versions (1 .. 16) of every tensor of the plan into ONE patch per tensor.
 * [TALK] 16:40-17:04 (a sidecar catching up), [PULSE] "1. PULSESync" (values
 * are absolute): the result lists every index any version lists, with the
 * value of the latest version that lists it, in ascending order; applying it
 * equals applying the versions in turn. Per tensor it equals folding
 * pulse_compose over the versions, oldest first.
 *   patches     HOST, nversions x ntensors references, version-major (as for
 *               pulse_apply_chain_multi); each segment ascending
 *   outs        HOST, ntensors: outs[t].idx / outs[t].val (device) receive
 *               tensor t's composed segment; outs[t].room (host) must be at
 *               least min(n, sum over versions of min(count, n))
 *   counts_out  DEVICE, ntensors uint64: entries written per tensor
 * One partition launch and one compose launch; the plan needs only the
 * tensors' sizes (no buffer of the plan is read or written). Output buffers
 * must not overlap the inputs. Errors: PULSE_ERR_INVALID (NULL argument,
 * nversions outside 1..16, an output segment without room), PULSE_ERR_RANGE,
 * PULSE_ERR_NOMEM, PULSE_ERR_CUDA; device (plan error word): PULSE_ERR_INDEX
 * (count > n, clamped; an entry outside its chunk, skipped),
 * PULSE_ERR_TIMEOUT. A receiver that holds w catches up faster with
 * pulse_apply_chain_multi; composing pays where one patch must be sent.
 */
typedef struct pulse_patch_out {
    uint32_t *idx;  /* device, room entries */
    uint16_t *val;  /* device, room entries */
    uint64_t room;  /* host value */
} pulse_patch_out;

int pulse_compose_chain_multi(pulse_plan *plan, const pulse_patch_ref *patches, int nversions,
                              const pulse_patch_out *outs, uint64_t *counts_out,
                              cudaStream_t stream);

/* XOR mask / XOR apply over every tensor of the plan, one launch each. */
int pulse_xor_mask_multi(pulse_plan *plan, cudaStream_t stream);
int pulse_xor_apply_multi(pulse_plan *plan, cudaStream_t stream);

/* Synchronise the device, then return and clear the plan's device error word
 * (PULSE_OK, PULSE_ERR_TIMEOUT or PULSE_ERR_INDEX). */
int pulse_plan_get_error(pulse_plan *plan);

/* ------------------------------------------------------------------------
 * PULSELoCo sender gate and receiver accumulation. [PULSE] "Metodologia:
 * PULSE -- 2. PULSELoCo": trainers run H local steps from a shared global
 * checkpoint, form FP32 pseudo-gradients, and synchronise only the entries
 * that would change the BF16 view; the rest stay in an FP32 error-feedback
 * buffer for the next round. Per element (each FP32 operation rounded once,
 * no fused multiply-add):
 *     d = local - global;  u = d + err;  (a NaN u is the quiet NaN 0x7FC00000)
 *     sent  iff  RNE_bf16(global + u) != RNE_bf16(global)  (bitwise; NaN -> 0x7FC0)
 *     sent: entry (i, u) and err = +0;  not sent: err = u.
 * Sent entries are written in ascending index order.
 * ---------------------------------------------------------------------- */

/*
 * pulse_loco_gate -- one tensor.
 *   global_w, local_w  device, n floats (read only)
 *   err                device, n floats, in/out (the error-feedback buffer)
 *   idx_out / val_out  device, room for n uint32 / n floats
 *   count_out          device uint64: entries sent
 * 16-byte aligned global_w/local_w/err take the fast path. Uses the same
 * per-(device, stream) workspace as pulse_encode. n == 0 writes count 0.
 * Errors: PULSE_ERR_INVALID, PULSE_ERR_RANGE, PULSE_ERR_NOMEM, PULSE_ERR_CUDA;
 * device: PULSE_ERR_TIMEOUT (pulse_get_error).
 */
int pulse_loco_gate(const float *global_w, const float *local_w, float *err, uint64_t n,
                    uint32_t *idx_out, float *val_out, uint64_t *count_out, cudaStream_t stream);

/*
 * pulse_loco_accumulate -- receiver: acc[idx[j]] += val[j] (FP32) for
 * j < count (HOST value). Within one call indices must be distinct (what the
 * gate produces); entries with idx >= n are skipped and PULSE_ERR_INDEX is
 * recorded for pulse_get_error(stream).
 */
int pulse_loco_accumulate(float *acc, uint64_t n, const uint32_t *idx, const float *val,
                          uint64_t count, cudaStream_t stream);

/* Multi-tensor form (one launch per operation for a whole model). Fields an
 * operation does not use may be NULL: gate_multi needs global_w, local_w,
 * err, idx, val; accumulate_multi needs acc, idx, val. */
typedef struct pulse_loco_tensor {
    const float *global_w;  /* device, n */
    const float *local_w;   /* device, n */
    float *err;             /* device, n, in/out */
    uint64_t n;             /* elements, < 2^32 */
    uint32_t *idx;          /* device, room for n (sent indices) */
    float *val;             /* device, room for n (sent values) */
    float *acc;             /* device, n (receiver accumulator) */
} pulse_loco_tensor;

typedef struct pulse_loco_plan pulse_loco_plan;

int pulse_loco_plan_create(const pulse_loco_tensor *tensors, int ntensors, pulse_loco_plan **plan_out);
int pulse_loco_plan_destroy(pulse_loco_plan *plan);
/* counts_out: device, ntensors uint64. */
int pulse_loco_gate_multi(pulse_loco_plan *plan, uint64_t *counts_out, cudaStream_t stream);
/* counts_dev: device, ntensors uint64 (e.g. the counts_out of a gate). */
int pulse_loco_accumulate_multi(pulse_loco_plan *plan, const uint64_t *counts_dev, cudaStream_t stream);
int pulse_loco_plan_get_error(pulse_loco_plan *plan);

/* ------------------------------------------------------------------------
 * Codec-friendly index packing. [PULSE] "1. PULSESync -- Compressione":
 * patches are further compressed with general codecs (zstd); [XOR]
 * "Pipeline'i GPU'lara tasimak": byte-oriented LZ4 on the GPU, and
 * trainer-side compression latency matters. The pages leave the index
 * representation open; this format (a reading of this library) turns the
 * strictly ascending uint32 indices of a patch segment into small packed
 * gaps before such a codec:
 *  - blocks of PULSE_PACK_BLOCK = 128 entries (the last may be shorter);
 *    firsts[i] = block i's first index;
 *  - gap of slot s = idx[128 i + s + 1] - idx[128 i + s] - 1;
 *    widths[i] = bit length of the block's largest gap (0 if none);
 *  - block i's payload = 16 * widths[i] bytes: slot s in bits
 *    [s w, s w + w) of a little-endian bit string (bit t = bit t % 8 of
 *    byte t / 8), unused bits 0; payloads back to back in block order;
 *  - chunks of 32 blocks (PULSE_PACK_CHUNK = 4096 entries):
 *    chunk_off[c] = byte offset of block 32 c's payload, so each chunk
 *    decodes independently.
 * ---------------------------------------------------------------------- */
#define PULSE_PACK_BLOCK 128
#define PULSE_PACK_CHUNK 4096

/*
 * pulse_pack_indices -- pack count indices (DEVICE, strictly ascending).
 *   firsts     device, ceil(count / 128) uint32
 *   widths     device, ceil(count / 128) uint8
 *   chunk_off  device, ceil(count / 4096) uint64
 *   payload    device, 16-byte aligned, room for 512 * ceil(count / 128)
 *              bytes (the widest case)
 *   payload_bytes  device uint64: payload bytes written
 * Uses the per-(device, stream) workspace of pulse_encode. count == 0 writes
 * payload_bytes = 0. Errors: PULSE_ERR_INVALID, PULSE_ERR_RANGE,
 * PULSE_ERR_NOMEM, PULSE_ERR_CUDA; device: PULSE_ERR_TIMEOUT.
 */
int pulse_pack_indices(const uint32_t *idx, uint64_t count, uint32_t *firsts, uint8_t *widths,
                       uint64_t *chunk_off, uint8_t *payload, uint64_t *payload_bytes,
                       cudaStream_t stream);

/*
 * pulse_unpack_indices -- the inverse: rebuild count indices (count is a
 * HOST value) into idx_out (device, count uint32). payload 4-byte aligned.
 */
int pulse_unpack_indices(const uint32_t *firsts, const uint8_t *widths, const uint64_t *chunk_off,
                         const uint8_t *payload, uint64_t count, uint32_t *idx_out,
                         cudaStream_t stream);

/*
 * pulse_pack_indices_multi -- pack the index segments of a whole model in
 * one launch (every chunk of every segment). segs: HOST array of nsegs
 * segments, copied before the call returns; each is packed exactly as
 * pulse_pack_indices packs it (idx is read). payload_bytes: DEVICE, nsegs
 * uint64: segment s's payload size (0 for an empty segment). Uses the
 * per-(device, stream) workspace of pulse_encode; growing it synchronises
 * `stream`. Errors: PULSE_ERR_INVALID (NULL segs or payload_bytes, nsegs < 1,
 * a NULL or misaligned buffer of a non-empty segment), PULSE_ERR_RANGE (a
 * count >= 2^32), PULSE_ERR_NOMEM, PULSE_ERR_CUDA; device: PULSE_ERR_TIMEOUT.
 *
 * pulse_unpack_indices_multi -- the inverse over the same segment table:
 * rebuilds each segment's count indices into its idx (written), one launch.
 * payload 4-byte aligned.
 */
typedef struct pulse_pack_segment {
    uint32_t *idx;        /* device, count indices: read by pack, written by unpack */
    uint64_t count;       /* host value */
    uint32_t *firsts;     /* device, ceil(count / 128) */
    uint8_t *widths;      /* device, ceil(count / 128) */
    uint64_t *chunk_off;  /* device, ceil(count / 4096) */
    uint8_t *payload;     /* device, room for 512 * ceil(count / 128) bytes */
} pulse_pack_segment;

int pulse_pack_indices_multi(const pulse_pack_segment *segs, int nsegs, uint64_t *payload_bytes,
                             cudaStream_t stream);
int pulse_unpack_indices_multi(const pulse_pack_segment *segs, int nsegs, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Patch-chain composition. [TALK] 16:40-17:04: a sidecar whose engine is
 * behind applies the missing transitions; [PULSE] "1. PULSESync": patch
 * values are absolute. So patch A followed by patch B equals ONE patch:
 * every index listed by A or B, with B's value where both list it (the later
 * patch wins), in ascending order. A chain of m patches composes by folding
 * left; applying the result once equals applying the m patches in order.
 * For a whole model, pulse_compose_chain_multi composes up to 16 versions in
 * one pass (and pulse_apply_chain_multi applies them without composing),
 * both far faster than folding pairs with these calls.
 * Preconditions: within each input, indices strictly ascending (what encode
 * produces); output buffers hold count_a + count_b entries and overlap no
 * input. Counts in are HOST values, count out is DEVICE memory.
 * ---------------------------------------------------------------------- */

/*
 * pulse_compose -- compose two BF16 patches (16-bit values).
 *   idx_a/val_a  device, count_a entries (the earlier patch)
 *   idx_b/val_b  device, count_b entries (the later patch)
 *   idx_out/val_out device, room for count_a + count_b entries
 *   count_out    device uint64: entries written
 * Uses a library workspace per (device, stream) (allocated on first use and
 * grown on demand; growth synchronises `stream`). Errors: PULSE_ERR_INVALID,
 * PULSE_ERR_RANGE (a count >= 2^32), PULSE_ERR_NOMEM, PULSE_ERR_CUDA; device:
 * PULSE_ERR_TIMEOUT (pulse_get_error).
 */
int pulse_compose(const uint32_t *idx_a, const uint16_t *val_a, uint64_t count_a,
                  const uint32_t *idx_b, const uint16_t *val_b, uint64_t count_b,
                  uint32_t *idx_out, uint16_t *val_out, uint64_t *count_out,
                  cudaStream_t stream);

/* pulse_compose_u8 -- the same for 8-bit values (an MXFP8 code or scale segment). */
int pulse_compose_u8(const uint32_t *idx_a, const uint8_t *val_a, uint64_t count_a,
                     const uint32_t *idx_b, const uint8_t *val_b, uint64_t count_b,
                     uint32_t *idx_out, uint8_t *val_out, uint64_t *count_out,
                     cudaStream_t stream);

/*
 * pulse_compose_multi -- compose the segments of a whole model in one pass
 * (one partition launch + one compose launch). segs: HOST array of nsegs
 * segment pairs (copied before the call returns); value_bytes: 2 (BF16
 * patches) or 1 (MXFP8 segments); counts_out: DEVICE, nsegs uint64.
 */
typedef struct pulse_compose_segment {
    const uint32_t *idx_a;   /* device, count_a entries */
    const void *val_a;
    uint64_t count_a;        /* host value */
    const uint32_t *idx_b;   /* device, count_b entries */
    const void *val_b;
    uint64_t count_b;        /* host value */
    uint32_t *idx_out;       /* device, room for count_a + count_b */
    void *val_out;
} pulse_compose_segment;

int pulse_compose_multi(const pulse_compose_segment *segs, int nsegs, int value_bytes,
                        uint64_t *counts_out, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * MXFP8 serving view. [TALK] 13:06-14:40: rollouts are often served below
 * BF16 (FP8, MXFP4, NVFP4); a plain float format hides updates below about
 * theta / 2^(mantissa bits + 1), and with a shared group scale a scale
 * change moves the whole group. [PULSE] "Potenziale Futuro": FP8 and MX
 * views should be sparser still. [MX] OCP "Microscaling Formats (MX)
 * Specification" v1.0 fixes the format (the pages do not):
 *
 *  - blocks of 32 consecutive elements of a tensor (the last block may be
 *    shorter) share one E8M0 scale byte s, value 2^(s - 127);
 *    s = floor(log2(max |v| over the block)) - 8 + 127, limited to
 *    [0, 254]; a block whose maximum is 0 gets s = 0; a block holding a NaN
 *    or an infinity gets s = 0xFF (NaN) and every code 0x7F;
 *  - each element's code is the E4M3 encoding (OCP 8-bit float: bias 7, no
 *    infinities, 0x7F/0xFF NaN, largest normal 448) of v / 2^(s - 127),
 *    rounded to nearest even, magnitudes past 448 clamped to 448, sign kept
 *    (-0 -> 0x80), subnormals kept.
 *
 * A view is two arrays: codes (n uint8) and scales (ceil(n / 32) uint8). An
 * MXFP8 patch has two segments, each in ascending index order: changed codes
 * (element index uint32, new code uint8) and changed scales (block index
 * uint32, new scale uint8). n < 2^32 as everywhere.
 * ---------------------------------------------------------------------- */
#define PULSE_MX_BLOCK 32

/*
 * pulse_mx_quantize -- the MXFP8 view of one tensor (to initialise a
 * trainer's previous view or a receiver).
 *   master_f32  device, n floats;  codes_out device, n uint8;
 *   scales_out  device, ceil(n / 32) uint8.
 * n == 0 launches nothing. Errors: PULSE_ERR_INVALID, PULSE_ERR_RANGE,
 * PULSE_ERR_CUDA.
 */
int pulse_mx_quantize(const float *master_f32, uint64_t n, uint8_t *codes_out,
                      uint8_t *scales_out, cudaStream_t stream);

/*
 * pulse_mx_encode -- trainer-side encode of the MXFP8 view of one tensor.
 * Computes the new view of master_f32, compares it bitwise with
 * (prev_codes, prev_scales), writes both patch segments and refreshes both
 * previous arrays in place:
 *   idx_out[0..k)  / val_out[0..k)    changed codes (room for n entries)
 *   sidx_out[0..ks) / sval_out[0..ks) changed scales (room for ceil(n/32))
 *   counts_out     device, two uint64: {k, ks}
 * master_f32, prev_codes and prev_scales 16-byte aligned take the fast
 * path; any alignment is correct. Uses a library workspace per (device,
 * stream), separate from pulse_encode's, allocated on first use; each call
 * also clears that workspace's tile status words (one memset). n == 0 writes
 * counts {0, 0}. Errors: PULSE_ERR_INVALID, PULSE_ERR_RANGE, PULSE_ERR_NOMEM,
 * PULSE_ERR_CUDA; device: PULSE_ERR_TIMEOUT (pulse_get_error).
 */
int pulse_mx_encode(const float *master_f32, uint8_t *prev_codes, uint8_t *prev_scales,
                    uint64_t n, uint32_t *idx_out, uint8_t *val_out, uint32_t *sidx_out,
                    uint8_t *sval_out, uint64_t *counts_out, cudaStream_t stream);

/*
 * pulse_mx_apply -- sampler-side apply of both segments of an MXFP8 patch to
 * a view of n elements: codes[idx[j]] = val[j] for j < count, then
 * scales[sidx[j]] = sval[j] for j < scount (counts are HOST values). Entries
 * past the view (idx >= n, sidx >= ceil(n/32)) are skipped and recorded as
 * PULSE_ERR_INDEX for pulse_get_error(stream).
 */
int pulse_mx_apply(uint8_t *codes, uint8_t *scales, uint64_t n, const uint32_t *idx,
                   const uint8_t *val, uint64_t count, const uint32_t *sidx,
                   const uint8_t *sval, uint64_t scount, cudaStream_t stream);

/*
 * MXFP8 multi-tensor plans: as pulse_plan, one launch for the whole model.
 * Fields an operation does not use may be NULL:
 *   mx_encode_multi  master, prev_codes, prev_scales, idx, val, sidx, sval
 *   mx_apply_multi   codes, scales, idx, val, sidx, sval
 * Counts are 2 x ntensors uint64 in list order: {k_0, ks_0, k_1, ks_1, ...}.
 * At most 8192 tensors per plan.
 */
typedef struct pulse_mx_tensor {
    const float *master;   /* device, n floats (trainer) */
    uint8_t *prev_codes;   /* device, n uint8 (trainer, in/out) */
    uint8_t *prev_scales;  /* device, ceil(n/32) uint8 (trainer, in/out) */
    uint8_t *codes;        /* device, n uint8 (sampler, in/out) */
    uint8_t *scales;       /* device, ceil(n/32) uint8 (sampler, in/out) */
    uint64_t n;            /* elements, < 2^32 */
    uint32_t *idx;         /* device, room for n uint32 (code segment) */
    uint8_t *val;          /* device, room for n uint8 */
    uint32_t *sidx;        /* device, room for ceil(n/32) uint32 (scale segment) */
    uint8_t *sval;         /* device, room for ceil(n/32) uint8 */
} pulse_mx_tensor;

typedef struct pulse_mx_plan pulse_mx_plan;

int pulse_mx_plan_create(const pulse_mx_tensor *tensors, int ntensors, pulse_mx_plan **plan_out);
int pulse_mx_plan_destroy(pulse_mx_plan *plan);
int pulse_mx_plan_num_tensors(const pulse_mx_plan *plan);
/* counts_out: device, 2 x ntensors uint64. */
int pulse_mx_encode_multi(pulse_mx_plan *plan, uint64_t *counts_out, cudaStream_t stream);
/* counts_host: HOST, 2 x ntensors uint64 (copied before return). */
int pulse_mx_apply_multi(pulse_mx_plan *plan, const uint64_t *counts_host, cudaStream_t stream);
/* counts_dev: DEVICE, 2 x ntensors uint64 (e.g. counts_out of pulse_mx_encode_multi). */
int pulse_mx_apply_multi_device(pulse_mx_plan *plan, const uint64_t *counts_dev, cudaStream_t stream);
int pulse_mx_plan_get_error(pulse_mx_plan *plan);

/* ------------------------------------------------------------------------
 * MXFP4 serving view. [TALK] 13:06-14:40 names MXFP4 and NVFP4 serving: each
 * weight is quantized against a shared group scale, and a scale change moves
 * the whole group; [KR] same section; [PULSE] "Potenziale Futuro": MXFP4
 * views should be sparser still. [MX] fixes the format:
 *
 *  - blocks of 32 consecutive elements share one E8M0 scale byte s exactly
 *    as in the MXFP8 view but with the E2M1 maximum exponent:
 *    s = floor(log2(max |v| over the block)) - 2 + 127, limited to
 *    [0, 254]; an all-zero block gets s = 0; a block holding a NaN or an
 *    infinity gets s = 0xFF and every code 0;
 *  - each element's code is the E2M1 encoding (sign, 2 exponent bits with
 *    bias 1, 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) of
 *    v / 2^(s - 127), rounded to nearest even, magnitudes past 6 clamped to
 *    6, sign kept (a negative value rounding to zero gives code 0x8);
 *  - codes are stored two per byte: element 2j in the low nibble of byte j,
 *    element 2j + 1 in the high nibble; a tensor of odd length has a zero
 *    high nibble in its last byte.
 *
 * A view is codes (ceil(n / 2) bytes) and scales (ceil(n / 32) bytes). Its
 * patch lists changed code BYTES (byte index, new byte) and changed scales
 * (block index, new byte), each ascending; applying it is the byte apply of
 * the MXFP8 view. The _fmt forms below take the format and otherwise behave
 * as the MXFP8 calls above, with "codes" and "code segment" counted in bytes
 * (ceil(n / 2) for E2M1). The MXFP8 calls equal the _fmt calls with
 * PULSE_MX_E4M3.
 * ---------------------------------------------------------------------- */
#define PULSE_MX_E4M3 0  /* MXFP8: one E4M3 code per byte */
#define PULSE_MX_E2M1 1  /* MXFP4: two E2M1 codes per byte */

/* Errors as the MXFP8 calls, plus PULSE_ERR_INVALID for an unknown format.
 * The quantize and encode forms take PULSE_MX_E4M3 or PULSE_MX_E2M1 (NVFP4
 * has its own entry points below); apply and plans take all three. */
int pulse_mx_quantize_fmt(int format, const float *master_f32, uint64_t n, uint8_t *codes_out,
                          uint8_t *scales_out, cudaStream_t stream);
int pulse_mx_encode_fmt(int format, const float *master_f32, uint8_t *prev_codes,
                        uint8_t *prev_scales, uint64_t n, uint32_t *idx_out, uint8_t *val_out,
                        uint32_t *sidx_out, uint8_t *sval_out, uint64_t *counts_out,
                        cudaStream_t stream);
int pulse_mx_apply_fmt(int format, uint8_t *codes, uint8_t *scales, uint64_t n,
                       const uint32_t *idx, const uint8_t *val, uint64_t count,
                       const uint32_t *sidx, const uint8_t *sval, uint64_t scount,
                       cudaStream_t stream);
/* A plan of one format: prev_codes, codes, idx and val of each tensor hold
 * code bytes (ceil(n / 2) for E2M1 and NVFP4); prev_scales, scales, sidx and
 * sval hold block scales (ceil(n / 16) for NVFP4). */
int pulse_mx_plan_create_fmt(const pulse_mx_tensor *tensors, int ntensors, int format,
                             pulse_mx_plan **plan_out);

/* ------------------------------------------------------------------------
 * NVFP4 serving view. [TALK] 13:06-14:00 names NVFP4 serving and its
 * hierarchical scales; [XOR] section "Bildirilen sayilar" uses an NVFP4
 * checkpoint as its workload (0.085 % of it changes per step). The pages do
 * not define the format; this library reads it as the publicly described
 * NVFP4 layout, with every scale step one FP32 operation rounded to nearest
 * even, in this order:
 *  - A = the tensor's largest finite magnitude; tensor scale S = A / 2688
 *    (2688 = 448 * 6);
 *  - blocks of 16 consecutive elements; a block holding a NaN or an infinity
 *    gets scale byte 0x7F and codes 0; otherwise the block scale byte is the
 *    E4M3 (round to nearest even, clamped to 448) of (max |v| / 6) / S, and
 *    0 when S is 0;
 *  - element codes: E2M1 (as in the MXFP4 view, two per byte, element 2j in
 *    the low nibble) of v * (1 / (dec(scale byte) * S)); all 0 when the
 *    scale byte is 0 or that product is 0 or its reciprocal is not finite.
 * A view is codes (ceil(n / 2) bytes), block scales (ceil(n / 16) bytes)
 * and S. A patch lists changed code bytes and changed block scales (as the
 * MX patches) and carries the new S (4 bytes of metadata per tensor). Apply
 * with pulse_mx_apply_fmt(PULSE_MX_NVFP4, ...) or an NVFP4 plan's
 * pulse_mx_apply_multi*, and take S from the patch.
 * ---------------------------------------------------------------------- */
#define PULSE_MX_NVFP4 2  /* NVFP4: E2M1 codes, E4M3 scale per 16, FP32 scale per tensor */

/* The NVFP4 view of one tensor; tscale_out: device, one float (S). Two
 * launches (the tensor maximum, then the view). Errors as pulse_mx_quantize. */
int pulse_nvfp4_quantize(const float *master_f32, uint64_t n, uint8_t *codes_out,
                         uint8_t *scales_out, float *tscale_out, cudaStream_t stream);

/* As pulse_mx_encode for the NVFP4 view; tscale_out (device, one float)
 * receives the new view's S. The tensor maximum is one extra pass over
 * master_f32 before the encode launch. */
int pulse_nvfp4_encode(const float *master_f32, uint8_t *prev_codes, uint8_t *prev_scales,
                       uint64_t n, uint32_t *idx_out, uint8_t *val_out, uint32_t *sidx_out,
                       uint8_t *sval_out, uint64_t *counts_out, float *tscale_out,
                       cudaStream_t stream);

/* Whole-model NVFP4 encode on a plan created with PULSE_MX_NVFP4 (which
 * pulse_mx_encode_multi refuses); tscales_out: device, ntensors floats. */
int pulse_nvfp4_encode_multi(pulse_mx_plan *plan, uint64_t *counts_out, float *tscales_out,
                             cudaStream_t stream);

/*
 * pulse_encode_noalloc -- pulse_encode for callers that must not allocate
 * device memory. The pages describe no counterpart; this entry point exists
 * for integration only.
 *
 * pulse_encode allocates its look-back scratch with cudaMalloc the first time
 * a (device, stream) pair is seen and grows it for larger tensors. Callers
 * that cannot allocate at that point -- engines that give all device memory
 * to their own pool at start-up, runtimes that forbid allocation once serving
 * has begun, code that must not let an allocation synchronise the device --
 * use this variant: it computes exactly what pulse_encode computes, with the
 * same arguments, but keeps its scratch in one fixed device array inside the
 * library (512 KB + 256 bytes, held by every GPU that loads the library until
 * the process exits) and calls no cudaMalloc, cudaFree or other allocating
 * routine.
 *
 *  - n may be at most PULSE_NOALLOC_MAX_ELEMS (2^28); larger n returns
 *    PULSE_ERR_RANGE and launches nothing.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current and keeps it for the
 *    rest of the process; make that first call before any stream capture.
 *    After cudaDeviceReset the kept address is stale: do not call this entry
 *    point on a device that has been reset.
 *  - All calls share the array and it keeps the previous call's contents;
 *    each call clears, on its stream before its kernel, the part it reads
 *    (8 bytes per 4096 elements plus 256 bytes). Calls whose work may
 *    overlap on the GPU (different streams without ordering) race on the
 *    array: order them.
 *  - Device-side errors are not kept for pulse_get_error: a wait that gave
 *    up is reported as *count_out == UINT64_MAX (outputs invalid).
 */
#define PULSE_NOALLOC_MAX_ELEMS 268435456ull
int pulse_encode_noalloc(const float *master_f32, uint16_t *prev_bf16, uint64_t n,
                         uint32_t *idx_out, uint16_t *val_out, uint64_t *count_out,
                         cudaStream_t stream);

/*
 * Test hook for the look-back watchdog (not for production use). Runs
 * pulse_encode with a wait limit of `wait_limit_ns` nanoseconds while tile 0
 * is never processed, so tile 1 waits for a predecessor that never
 * publishes. Expected outcome: the wait gives up, PULSE_ERR_TIMEOUT is
 * recorded for pulse_get_error(stream), every write stays inside the
 * caller's buffers, and the context stays usable. Needs n > one tile.
 */
int pulse_debug_encode_orphan_tile(const float *master_f32, uint16_t *prev_bf16, uint64_t n,
                                   uint32_t *idx_out, uint16_t *val_out, uint64_t *count_out,
                                   uint64_t wait_limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PULSE_H */
