// pulse_internal.h -- descriptors and launchers shared by the library's
// translation units (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pulse {

// ---------------------------------------------------------------- encode
// Tile geometry: kEncThreads compute threads x kEncRounds rounds x 4
// elements. Each CTA adds one producer warp and kEncLookbackWarps look-back
// warps.
constexpr int kEncThreads = 256;
constexpr int kEncRounds = 4;
constexpr int kEncTile = kEncThreads * kEncRounds * 4;  // 4096 elements
#ifndef PULSE_ENC_STAGES
#define PULSE_ENC_STAGES 2
#endif
#ifndef PULSE_ENC_LOOKBACK_WARPS
#define PULSE_ENC_LOOKBACK_WARPS 1
#endif
// Parked tiles per CTA awaiting copy-out, and parked tiles resolved per
// look-back round trip (PULSE_ENC_LB_BATCH), for the kernels built on the
// encode pipeline. On the 8.03B step 16 and 2 measured faster than 8 and 4
// (BF16 encode 0.3 % at 8 % density and 1.6 % at 1.2 %, MXFP8 2.9 %, MXFP4
// 5.6 %, LoCo gate 1.1 %, index packing 1.7 %), and 16 and 1 faster again
// (BF16 encode 0.5 %, MXFP8 1.8 %, MXFP4 1.2 %); 32 slots cost MXFP8 its
// third CTA per SM. The two composition kernels keep 8 and 4 of their own.
#ifndef PULSE_ENC_PARKED
#define PULSE_ENC_PARKED 16
#endif
#ifndef PULSE_ENC_RING
#define PULSE_ENC_RING 4096
#endif
#ifndef PULSE_ENC_MIN_BLOCKS
#define PULSE_ENC_MIN_BLOCKS 3
#endif
// Look-back words per lane and round trip: 4 (a 128-tile window) measured
// faster than 2 with one tile per look-back (MXFP8 9.19 against 9.24 ms on
// the 8.03B step, MXFP4 8.18 against 8.28, LoCo gate 20.0 against 20.2). The
// BF16 encode (dense tiles) and NVFP4 keep 2, the composition kernels too.
#ifndef PULSE_ENC_LOOKBACK
#define PULSE_ENC_LOOKBACK 4
#endif
#ifndef PULSE_ENC_LB_BATCH
#define PULSE_ENC_LB_BATCH 1
#endif

constexpr int kEncStages = PULSE_ENC_STAGES;                // bulk-copy ring depth
constexpr int kEncLookbackWarps = PULSE_ENC_LOOKBACK_WARPS;  // concurrent look-backs per CTA
constexpr int kEncParked = PULSE_ENC_PARKED;                // parked tiles per CTA awaiting copy-out
constexpr int kEncRing = PULSE_ENC_RING;                    // parked patch entries per CTA
constexpr int kEncMinBlocks = PULSE_ENC_MIN_BLOCKS;          // resident CTAs per SM
constexpr int kEncLookbackPerLane = PULSE_ENC_LOOKBACK;     // look-back words per lane per round trip
constexpr int kEncLookbackBatch = PULSE_ENC_LB_BATCH;        // parked tiles resolved per round trip
constexpr int kEncBlockThreads = kEncThreads + 32 * (1 + kEncLookbackWarps);
static_assert(kEncRing >= kEncTile, "the parked-entry ring holds at least one full tile");

// Device view of one tensor for the encode / XOR-mask / apply kernels.
struct TensorDesc {
  const float* master;
  uint16_t* prev;
  uint16_t* w;
  uint32_t* idx;
  uint16_t* val;
  uint16_t* mask;
  uint64_t n;
  uint64_t tile_begin;  // first global encode tile of this tensor
  uint32_t bulk_ok;     // master and prev 16-byte aligned: encode may bulk-copy tiles
  uint32_t vec_ok;      // kVecMask | kVecApply bits: XOR kernels may use vector accesses
};
constexpr uint32_t kVecMask = 2u;   // master 16-byte, prev and mask 8-byte aligned
constexpr uint32_t kVecApply = 4u;  // w and mask 8-byte aligned

// Library-owned scratch of one launch context (a stream, or a plan).
struct Workspace {
  uint64_t* status = nullptr;    // one look-back word per tile
  uint32_t* counters = nullptr;  // [0] tile ticket, [1] CTAs finished, [2] error word
  uint64_t capacity_tiles = 0;
  uint32_t epoch = 0;            // host-side launch counter (30 bits used)
  int device = -1;
};

struct EncodeLaunch {
  TensorDesc one;                // single-tensor mode
  const TensorDesc* tensors;     // multi-tensor mode: device array
  const uint64_t* tile_begin;    // multi-tensor mode: ntensors + 1 entries (device)
  int ntensors;                  // 1 in single-tensor mode
  uint64_t total_tiles;
  uint64_t* status;
  uint32_t* counters;
  uint64_t* counts_out;          // ntensors device uint64
  uint32_t epoch;
  uint32_t first_ticket;         // 0, or 1 for the watchdog test hook
  uint64_t wait_limit_ns;
};

int encode_grid_size(int device);
cudaError_t launch_encode(const EncodeLaunch& a, bool multi, int grid, cudaStream_t stream);

// ------------------------------------------------------- MX view encode
// Same CTA layout and tile as the BF16 encode; a tile holds kEncTile / 32
// blocks of 32 elements sharing one E8M0 scale.
constexpr int kMxBlock = 32;

struct MxTensorDesc {
  const float* master;
  uint8_t* prev_codes;   // code bytes (n for E4M3, ceil(n / 2) for E2M1), in/out
  uint8_t* prev_scales;  // ceil(n / 32) E8M0 scales, in/out
  uint32_t* idx;         // code segment: code-byte indices
  uint8_t* val;          //               new code bytes
  uint32_t* sidx;        // scale segment: block indices
  uint8_t* sval;         //                new scales
  uint64_t n;
  uint64_t tile_begin;   // first global encode tile of this tensor
  uint32_t bulk_ok;      // master, prev_codes, prev_scales 16-byte aligned
  uint32_t reserved;
};

struct MxLaunch {
  MxTensorDesc one;              // single-tensor mode
  const MxTensorDesc* tensors;   // multi-tensor mode: device array
  const uint64_t* tile_begin;    // multi-tensor mode: ntensors + 1 entries (device)
  int ntensors;
  uint64_t total_tiles;
  uint64_t* status;              // cleared (all zero) before the launch
  uint32_t* counters;
  uint64_t* counts_out;          // 2 x ntensors device uint64: codes, scales per tensor
  uint32_t epoch;                // unused (the packed status words carry no epoch)
  uint32_t first_ticket;
  uint64_t wait_limit_ns;
  const uint32_t* amax_bits;     // NVFP4: per tensor, largest finite magnitude (float bits)
  float* tscale_out;             // NVFP4: per tensor, the new view's tensor scale
};

// Element formats of the MX views (values of the public PULSE_MX_* constants).
constexpr int kFmtE4M3 = 0;  // MXFP8: one E4M3 code per byte
constexpr int kFmtE2M1 = 1;  // MXFP4: two E2M1 codes per byte, element 2j in the low nibble
constexpr int kFmtNvfp4 = 2; // NVFP4: E2M1 codes as MXFP4, E4M3 scale per 16, FP32 per tensor

int encode_mx_grid_size(int device, int format);
cudaError_t launch_encode_mx(const MxLaunch& a, int format, bool multi, int grid,
                             cudaStream_t stream);
// amax_bits / tscale_out: NVFP4 only (one tensor).
cudaError_t launch_mx_quantize(int format, const float* master, uint64_t n, uint8_t* codes,
                               uint8_t* scales, const uint32_t* amax_bits, float* tscale_out,
                               cudaStream_t stream);
// Per-tensor largest finite magnitude of the launch's tensors into amax_bits
// (zeroed by the caller), for the NVFP4 tensor scale.
cudaError_t launch_mx_amax(const MxLaunch& a, bool multi, uint32_t* amax_bits, cudaStream_t stream);

// ---------------------------------------------------------------- PULSELoCo
struct LocoTensorDesc {
  const float* global;  // shared checkpoint
  const float* local;   // this worker's parameters after its local steps
  float* err;           // FP32 error feedback, in/out
  uint32_t* idx;        // sent entries: indices
  float* val;           //               values
  float* acc;           // receiver accumulator (accumulate)
  uint64_t n;
  uint64_t tile_begin;  // first global gate tile of this tensor
  uint32_t bulk_ok;     // global, local, err 16-byte aligned
  uint32_t reserved;
};

struct LocoLaunch {
  LocoTensorDesc one;
  const LocoTensorDesc* tensors;
  const uint64_t* tile_begin;
  int ntensors;
  uint64_t total_tiles;
  uint64_t* status;
  uint32_t* counters;
  uint64_t* counts_out;
  uint32_t epoch;
  uint32_t first_ticket;
  uint64_t wait_limit_ns;
};

uint64_t loco_tiles(uint64_t n);
int loco_grid_size(int device);
cudaError_t launch_loco_gate(const LocoLaunch& a, bool multi, int grid, cudaStream_t stream);
cudaError_t launch_loco_accumulate(float* acc, uint64_t n, const uint32_t* idx, const float* val,
                                   uint64_t count, uint32_t* err, cudaStream_t stream);
cudaError_t launch_loco_accumulate_multi(const LocoTensorDesc* tensors, int ntensors,
                                         const uint64_t* counts, uint32_t* err, int grid,
                                         cudaStream_t stream);

// ---------------------------------------------------------------- index packing
// One segment of indices to pack (or to rebuild: idx is then written).
struct PackSegment {
  uint32_t* idx;
  uint64_t count;
  uint32_t* firsts;
  uint8_t* widths;
  uint64_t* chunk_off;
  uint8_t* payload;
  uint64_t* payload_bytes;  // pack: this segment's device word
  uint64_t chunk_begin;     // first global chunk of this segment
};
uint64_t pack_chunks(uint64_t count);
// segs / chunk_begin: device tables (nsegs, nsegs + 1 entries).
cudaError_t launch_pack_multi(const PackSegment* segs, const uint64_t* chunk_begin, int nsegs,
                              uint64_t total_chunks, uint64_t* status, uint32_t* counters,
                              uint32_t epoch, uint64_t wait_limit_ns, cudaStream_t stream);
cudaError_t launch_unpack_multi(const PackSegment* segs, const uint64_t* chunk_begin, int nsegs,
                                uint64_t total_chunks, cudaStream_t stream);
cudaError_t launch_pack(const uint32_t* idx, uint64_t count, uint32_t* firsts, uint8_t* widths,
                        uint64_t* chunk_off, uint8_t* payload, uint64_t* payload_bytes,
                        uint64_t* status, uint32_t* counters, uint32_t epoch,
                        uint64_t wait_limit_ns, cudaStream_t stream);
cudaError_t launch_unpack(const uint32_t* firsts, const uint8_t* widths, const uint64_t* chunk_off,
                          const uint8_t* payload, uint64_t count, uint32_t* idx_out,
                          cudaStream_t stream);

// ---------------------------------------------------------------- compose
// One pair of patch segments to compose (values 1 or 2 bytes wide) and its
// output; tile_begin is the segment's first global compose tile.
struct CmpSegment {
  const uint32_t* idx_a;
  const void* val_a;
  uint64_t count_a;
  const uint32_t* idx_b;
  const void* val_b;
  uint64_t count_b;
  uint32_t* idx_out;
  void* val_out;
  uint64_t tile_begin;
};

uint64_t compose_tiles(uint64_t entries);
// segs_dev == nullptr: single-segment mode using `one`.
cudaError_t launch_compose(const CmpSegment* segs_dev, const CmpSegment& one,
                           const uint64_t* tile_begin_dev, int nsegs, uint64_t total_tiles,
                           uint32_t* splits, uint32_t* tile_seg, uint64_t* status,
                           uint32_t* counters,
                           uint64_t* counts_out, uint32_t epoch, uint64_t wait_limit_ns,
                           int value_bytes, cudaStream_t stream);

// ---------------------------------------------------------------- apply
#ifndef PULSE_APPLY_PER_THREAD
#define PULSE_APPLY_PER_THREAD 4
#endif
#ifndef PULSE_XOR_ROUNDS
#define PULSE_XOR_ROUNDS 4
#endif
constexpr int kApplyThreads = 256;
constexpr int kApplyPerThread = PULSE_APPLY_PER_THREAD;     // entries per thread per tile
constexpr int kApplyTile = kApplyThreads * kApplyPerThread;  // 1024 entries

cudaError_t launch_apply(uint16_t* w, uint64_t n, bool checked, const uint32_t* idx,
                         const uint16_t* val, uint64_t count, uint32_t* error_word,
                         cudaStream_t stream);
cudaError_t launch_apply_multi(const TensorDesc* tensors, int ntensors,
                               const uint64_t* counts_dev, uint32_t* error_word,
                               int grid, cudaStream_t stream);

// Chained apply: chunks of kApplyChunk elements; chunk_begin[t] = first
// global chunk of tensor t (ntensors + 1), chunk_tensor[g] = tensor of chunk
// g. A chunk with at least kApplyDenseMin entries (over all versions) is
// read into shared memory whole.
#ifndef PULSE_APPLY_CHUNK
#define PULSE_APPLY_CHUNK 8192
#endif
#ifndef PULSE_APPLY_DENSE_MIN
#define PULSE_APPLY_DENSE_MIN 64
#endif
constexpr int kApplyChunk = PULSE_APPLY_CHUNK;
constexpr uint32_t kApplyDenseMin = PULSE_APPLY_DENSE_MIN;

// Chained apply: one tensor's patch of one version (ascending indices).
struct ChainSeg {
  const uint32_t* idx;
  const uint16_t* val;
  uint64_t count;
};
// Versions one chained-apply launch takes (longer chains take several
// launches, in order, on the same stream).
constexpr int kChainMaxVersions = 16;
// segs: nversions x ntensors, version-major; chain_first: scratch of
// nversions x total_chunks words. nversions in [1, kChainMaxVersions].
cudaError_t launch_apply_chain(const TensorDesc* tensors, const uint64_t* chunk_begin,
                               const uint32_t* chunk_tensor, uint32_t* chain_first,
                               const ChainSeg* segs, int ntensors, int nversions,
                               uint64_t total_chunks, uint32_t* error_word, uint64_t wait_limit_ns,
                               cudaStream_t stream);

// Chain partition (shared by the chained apply and the k-way compose):
// chain_first[v * total_chunks + g] = first entry of version v's segment at
// or after chunk g's start (kApplyChunk elements per chunk).
cudaError_t launch_chain_partition(const TensorDesc* tensors, const uint64_t* chunk_begin,
                                   const uint32_t* chunk_tensor, const ChainSeg* segs,
                                   int ntensors, int nversions, uint64_t total_chunks,
                                   uint32_t* chain_first, uint32_t* error_word,
                                   cudaStream_t stream);

// k-way composition of a chain of patches (compose_chunk.cu).
struct CcOut {
  uint32_t* idx;  // composed segment of one tensor
  uint16_t* val;
  uint64_t cap;   // room in entries
};
struct CcArgs {
  const TensorDesc* tensors;     // n of each tensor
  const uint64_t* chunk_begin;   // ntensors + 1
  const uint32_t* chunk_tensor;  // total_chunks
  const uint32_t* first;         // chain partition: nversions x total_chunks
  const ChainSeg* segs;          // nversions x ntensors, version-major (oldest first)
  const CcOut* outs;             // ntensors
  uint64_t* counts_out;          // ntensors (device), zeroed before the launch
  int ntensors;
  int nversions;                 // 1 .. kChainMaxVersions
  uint64_t total_chunks;
  uint64_t* status;              // one look-back word per chunk
  uint32_t* counters;            // [0] ticket, [1] CTAs finished, [2] error word
  uint32_t epoch;
  uint64_t wait_limit_ns;
};
cudaError_t launch_compose_chunks(const CcArgs& a, cudaStream_t stream);

// One byte-valued patch segment (an MXFP8 code or scale array).
struct ByteSegment {
  uint8_t* w;
  uint32_t* idx;
  uint8_t* val;
  uint64_t n;
};
cudaError_t launch_apply_u8(uint8_t* w, uint64_t n, bool checked, const uint32_t* idx,
                            const uint8_t* val, uint64_t count, uint32_t* error_word,
                            cudaStream_t stream);
cudaError_t launch_apply_u8_multi(const ByteSegment* segs, int nsegs, const uint64_t* counts_dev,
                                  uint32_t* error_word, int grid, cudaStream_t stream);

// ---------------------------------------------------------------- XOR
constexpr int kXorRounds = PULSE_XOR_ROUNDS;            // 4-element loads in flight per thread
constexpr int kXorTile = kEncTile;                        // XOR kernels reuse the encode tile table
constexpr int kXorThreads = kXorTile / (4 * kXorRounds);  // one tile per CTA pass
static_assert(kXorThreads * kXorRounds * 4 == kXorTile && kXorThreads >= 32, "tile geometry");

cudaError_t launch_xor_mask(const TensorDesc& one, const TensorDesc* tensors,
                            const uint64_t* tile_begin, int ntensors, uint64_t total_tiles,
                            bool multi, int grid, cudaStream_t stream);
cudaError_t launch_xor_apply(const TensorDesc& one, const TensorDesc* tensors,
                             const uint64_t* tile_begin, int ntensors, uint64_t total_tiles,
                             bool multi, int grid, cudaStream_t stream);

int sm_count(int device);

}  // namespace pulse
