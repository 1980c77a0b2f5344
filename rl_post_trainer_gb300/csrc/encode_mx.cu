// encode_mx.cu -- the MXFP8 serving view: quantize, and the fused
// quantize + compare + order-preserving compaction of what changed.
//
// Lower-precision serving ("Taking Reinforcement Learning Cross Datacenter",
// talk 13:06-14:40: rollouts served in FP8 / MXFP4 / NVFP4; a plain float
// format hides updates below about theta / 2^(mantissa bits + 1); with a
// shared group scale, a scale change moves a whole group) and the PULSE
// summary ("Potenziale Futuro": FP8 and MX views should be sparser still).
// The view is MXFP8 as the OCP Microscaling (MX) v1.0 specification defines
// it, the block-scaled FP8 that Blackwell tensor cores read directly: blocks
// of 32 consecutive elements share one E8M0 scale 2^e with
// e = floor(log2 max|v|) - 8 (limited to [-127, 127]); each element is the
// E4M3 encoding (round to nearest even, magnitudes past 448 clamped to 448)
// of v / 2^e. A block holding a NaN or an infinity gets the NaN scale 0xFF
// and the code 0x7F everywhere; an all-zero block gets the scale 2^-127.
//
// The patch has two segments per tensor, each in ascending index order:
// changed codes (element index, new code) and changed scales (block index,
// new scale). Encode refreshes both previous arrays in place.
//
// Kernel: the BF16 encode's persistent warp-specialized CTA (producer warp
// with bulk copies into a 2-stage ring, 8 compute warps, one look-back warp
// that resolves parked tiles with a decoupled look-back and copies them out).
// Per 4096-element tile the compute warps handle 4 consecutive elements per
// thread per round, so one 32-element block spans 8 consecutive lanes: the
// block maximum is 3 butterfly shuffles, the scale is read from the maximum's
// exponent bits, and the elements are scaled by an exact power of two and
// converted with the hardware's saturating E4M3 convert. The tile's status
// word carries both counts (codes in the low 32 bits, scales above), so one
// look-back yields both segment offsets.
#include <type_traits>

#include "encode_common.cuh"

namespace pulse {
namespace {

using namespace enc;

constexpr uint32_t kStageMasterBytes = kEncTile * 4;               // 16 KB
constexpr int kMaxTileBlocks = kEncTile / 16;                      // blocks of the smallest size

// Element formats: F = kFmtE4M3 (MXFP8, one code byte per element) or
// kFmtE2M1 (MXFP4, two codes per byte, element 2j in the low nibble of byte
// j). kEmax: exponent of the format's largest normal (448 = 1.75 * 2^8,
// 6 = 1.5 * 2^2).
// kBlock: elements per block scale. NVFP4 (kFmtNvfp4): E2M1 codes two per
// byte under an E4M3 scale per 16 elements and an FP32 scale per tensor.
template <int F>
struct Fmt;
template <>
struct Fmt<kFmtE4M3> {
  static constexpr uint32_t kEmax = 8;
  static constexpr uint32_t kElemsPerByte = 1;
  static constexpr uint32_t kBlock = 32;
};
template <>
struct Fmt<kFmtE2M1> {
  static constexpr uint32_t kEmax = 2;
  static constexpr uint32_t kElemsPerByte = 2;
  static constexpr uint32_t kBlock = 32;
};
template <>
struct Fmt<kFmtNvfp4> {
  static constexpr uint32_t kElemsPerByte = 2;
  static constexpr uint32_t kBlock = 16;
};
// Stage layout of a tile for format F: master, previous code bytes,
// previous scales.
// Stages in flight per CTA and parked-entry ring per format: a tile holds at
// most kEncTile / elements-per-byte code entries, so the FP4 formats need
// half the ring. A third stage costs MXFP8 its third CTA per SM (10.95
// against 9.20 ms on the 8.03B step) and leaves MXFP4 unchanged (8.21 against
// 8.19); NVFP4, whose tiles take longer to quantize, gains from it (13.94
// against 14.05 ms).
#ifndef PULSE_MX8_STAGES
#define PULSE_MX8_STAGES 2
#endif
#ifndef PULSE_MX4_STAGES
#define PULSE_MX4_STAGES 2
#endif
#ifndef PULSE_NV4_STAGES
#define PULSE_NV4_STAGES 3
#endif
constexpr int kMaxMxStages = 4;

template <int F>
struct Stage {
  static constexpr uint32_t kCodeBytes = kEncTile / Fmt<F>::kElemsPerByte;
  static constexpr uint32_t kScaleBytes = kEncTile / Fmt<F>::kBlock;  // one per block
  static constexpr uint32_t kBytes = kStageMasterBytes + kCodeBytes + kScaleBytes;
  static constexpr int kStages =
      F == kFmtE4M3 ? PULSE_MX8_STAGES : (F == kFmtNvfp4 ? PULSE_NV4_STAGES : PULSE_MX4_STAGES);
  static constexpr uint32_t kRing = kCodeBytes;  // parked code entries per CTA
  static constexpr uint32_t kRingMask = kRing - 1u;
  static constexpr size_t kDynSmem = size_t(kStages) * kBytes + size_t(kRing) * 4 + 128;
  static_assert(kBytes % 128 == 0, "stages stay 128-byte aligned");
  static_assert((kRing & (kRing - 1)) == 0, "the ring is a power of two");
  static_assert(kStages >= 2 && kStages <= kMaxMxStages, "stage count");
};

// ---------------------------------------------------------- MXFP8 arithmetic

// Saturating round-to-nearest-even FP32 -> E4M3 of two values; `hi` lands in
// the upper byte of the result.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Codes of 4 consecutive elements (element 0 in the low byte) under scale
// byte `scale`. The factor 2^(127 - scale) is a normal FP32 power of two
// (scale <= 246), so each product is exact unless it falls below 2^-126, and
// such a value rounds to a zero code either way.
__device__ __forceinline__ uint32_t mx_codes4(const float4& v, uint32_t scale) {
  if (scale == 0xFFu) return 0x7F7F7F7Fu;
  const float f = __uint_as_float(0x7F000000u - (scale << 23));  // (254 - scale) << 23
  return cvt_e4m3x2(__fmul_rn(v.y, f), __fmul_rn(v.x, f)) |
         (cvt_e4m3x2(__fmul_rn(v.w, f), __fmul_rn(v.z, f)) << 16);
}

// Saturating round-to-nearest-even FP32 -> E2M1 of 8 values under scale byte
// `scale`: byte j holds element 2j in its low nibble and 2j + 1 in its high
// nibble. Same scaling argument as mx_codes4 (scale <= 252 here).
__device__ __forceinline__ uint32_t fp4_codes8(const float4& a, const float4& b, uint32_t scale) {
  if (scale == 0xFFu) return 0u;
  const float f = __uint_as_float(0x7F000000u - (scale << 23));
  uint32_t r;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "f"(__fmul_rn(a.x, f)), "f"(__fmul_rn(a.y, f)), "f"(__fmul_rn(a.z, f)),
        "f"(__fmul_rn(a.w, f)), "f"(__fmul_rn(b.x, f)), "f"(__fmul_rn(b.y, f)),
        "f"(__fmul_rn(b.z, f)), "f"(__fmul_rn(b.w, f)));
  return r;
}

// -------------------------------------------------------------- shared state

struct StageMeta {
  uint32_t tile;
  uint32_t tensor;
  uint32_t mode;
  uint32_t len;  // elements in the tile
  float tscale;  // NVFP4: the tensor's FP32 scale
  uint64_t base;
  uint64_t first;
  uint64_t n;
  const float* master;
  uint8_t* prev_codes;
  uint8_t* prev_scales;
  uint32_t* idx;
  uint8_t* val;
  uint32_t* sidx;
  uint8_t* sval;
};

struct ParkedMeta {
  uint32_t tile;
  uint32_t tensor;
  uint32_t agg_c;  // changed code bytes in the tile
  uint32_t agg_s;  // changed scales in the tile
  uint32_t last;   // 1: last tile of its tensor; 2: no more tiles for this look-back warp
  uint32_t ring_start;
  uint64_t first;
  uint64_t n;
  uint64_t base;
  uint64_t code_base;  // code-byte index of the tile's first element
  uint64_t code_cap;   // code bytes of the tensor (the code segment's room)
  uint64_t scale_base; // block index of the tile's first element
  uint64_t scale_cap;  // blocks of the tensor (the scale segment's room)
  uint32_t* idx;
  uint8_t* val;
  uint32_t* sidx;
  uint8_t* sval;
};

struct __align__(16) MxShared {
  uint64_t full[kMaxMxStages];
  uint64_t empty[kMaxMxStages];
  uint64_t agg_ready[kPendSlots];
  uint64_t slot_free[kPendSlots];
  StageMeta meta[kMaxMxStages];
  ParkedMeta parked[kPendSlots];
  uint32_t warp_tot[2][kWarps];   // per warp: changed codes per round, one byte each
  uint32_t warp_stot[2][kWarps];  // per warp: changed scales per round, one byte each
  uint32_t ring_tail;
  uint16_t sring[kPendSlots][kMaxTileBlocks];  // parked scale entries: block | scale << 8
};
static_assert(kEncLookbackWarps == 1, "parked tiles are freed in order by one look-back warp");

// ------------------------------------------------------------ producer warp
template <int F, bool MULTI>
__device__ __forceinline__ void producer_loop(const MxLaunch& a, MxShared& sh, uint8_t* stages) {
  constexpr uint32_t kStageBytes = Stage<F>::kBytes, kStageCodeBytes = Stage<F>::kCodeBytes;
  constexpr int kEncStages = Stage<F>::kStages;
  const uint64_t pol_stream = l2_policy_evict_first();
  uint32_t fills_done = 0;
  uint32_t ticket = atomicAdd(a.counters + 0, 1u) + a.first_ticket;
  uint32_t cur_t = 0;
  uint64_t cur_begin = 1, cur_end = 0;
  MxTensorDesc d = a.one;
  // NVFP4: S = (largest finite magnitude of the tensor) / 2688, FP32
  auto tensor_scale = [&](uint32_t t) {
    return F == kFmtNvfp4 ? __fdiv_rn(__uint_as_float(a.amax_bits[t]), 2688.0f) : 0.0f;
  };
  float cur_s = tensor_scale(0);
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kEncStages);
    const bool end = ticket >= a.total_tiles;
    const uint32_t next = end ? ticket : atomicAdd(a.counters + 0, 1u) + a.first_ticket;
    if (it >= uint32_t(kEncStages) && !helper_wait(&sh.empty[s], ((it / kEncStages) - 1) & 1u, a))
      break;
    fills_done = it + 1;
    StageMeta m{};
    m.tile = ticket;
    if (end) {
      m.mode = kModeEnd;
      sh.meta[s] = m;
      mbar_arrive(&sh.full[s]);
      break;
    }
    if constexpr (MULTI) {
      if (uint64_t(ticket) < cur_begin || uint64_t(ticket) >= cur_end) {
        cur_t = uint32_t(find_tensor(a.tile_begin, a.ntensors, ticket));
        d = a.tensors[cur_t];
        cur_begin = d.tile_begin;
        cur_end = __ldg(a.tile_begin + cur_t + 1);
        cur_s = tensor_scale(cur_t);
      }
    }
    if (F == kFmtNvfp4 && uint64_t(ticket) == d.tile_begin) a.tscale_out[cur_t] = cur_s;
    const uint64_t base = (uint64_t(ticket) - d.tile_begin) * kEncTile;
    const uint64_t len = d.n - base < uint64_t(kEncTile) ? d.n - base : uint64_t(kEncTile);
    m.tensor = cur_t;
    m.len = uint32_t(len);
    m.tscale = cur_s;
    m.base = base;
    m.first = d.tile_begin;
    m.n = d.n;
    m.master = d.master;
    m.prev_codes = d.prev_codes;
    m.prev_scales = d.prev_scales;
    m.idx = d.idx;
    m.val = d.val;
    m.sidx = d.sidx;
    m.sval = d.sval;
    if (d.bulk_ok && len == uint64_t(kEncTile)) {
      m.mode = kModeBulk;
      sh.meta[s] = m;
      uint8_t* st = stages + size_t(s) * kStageBytes;
      mbar_arrive_expect_tx(&sh.full[s], kStageBytes);
      bulk_g2s(st, d.master + base, kStageMasterBytes, &sh.full[s], pol_stream);
      bulk_g2s_plain(st + kStageMasterBytes, d.prev_codes + base / Fmt<F>::kElemsPerByte,
                     kStageCodeBytes, &sh.full[s]);
      bulk_g2s_plain(st + kStageMasterBytes + kStageCodeBytes, d.prev_scales + base / Fmt<F>::kBlock,
                     Stage<F>::kScaleBytes, &sh.full[s]);
    } else {
      m.mode = kModeGeneric;
      sh.meta[s] = m;
      mbar_arrive(&sh.full[s]);
    }
    ticket = next;
  }
  for (uint32_t f = fills_done > uint32_t(kEncStages) ? fills_done - kEncStages : 0u; f < fills_done; ++f)
    mbar_wait_bounded(&sh.full[f % kEncStages], (f / kEncStages) & 1u, a.wait_limit_ns);
  __threadfence();
  const uint32_t finished = atomicAdd(a.counters + 1, 1u);
  if (finished == gridDim.x - 1) {
    atomicExch(a.counters + 0, 0u);
    atomicExch(a.counters + 1, 0u);
  }
}

// ---------------------------------------------------------- look-back warp

// Copy a parked tile's code entries to positions prefix_c + k (16-byte index
// and 4-byte code stores after a head of up to 3 entries) and its scale
// entries to positions prefix_s + k. Positions past the segment's capacity
// are never written (they only arise after a wait gave up).
template <int F>
__device__ __forceinline__ void copy_out(const ParkedMeta& pm, uint32_t prefix_c, uint32_t prefix_s,
                                         const uint32_t* ring, const uint16_t* sring, int lane) {
  constexpr uint32_t kRingMask = Stage<F>::kRingMask;
  const uint32_t agg = pm.agg_c;
  const uint32_t base = uint32_t(pm.code_base);
  const bool vec = (reinterpret_cast<uintptr_t>(pm.idx) % 16u == 0) &&
                   (reinterpret_cast<uintptr_t>(pm.val) % 4u == 0) &&
                   uint64_t(prefix_c) + agg <= pm.code_cap;
  uint32_t head = vec ? ((4u - (prefix_c & 3u)) & 3u) : agg;
  if (head > agg) head = agg;
  const uint32_t body = vec ? ((agg - head) & ~3u) : 0u;
  for (uint32_t k = uint32_t(lane); k < head; k += 32) {
    const uint32_t ent = ring[(pm.ring_start + k) & kRingMask];
    const uint64_t pos = uint64_t(prefix_c) + k;
    if (pos < pm.code_cap) {
      pm.idx[pos] = base + (ent & 0xFFFFu);
      pm.val[pos] = uint8_t(ent >> 16);
    }
  }
  for (uint32_t k = head + uint32_t(lane) * 4u; k < head + body; k += 128u) {
    uint32_t e[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) e[q] = ring[(pm.ring_start + k + uint32_t(q)) & kRingMask];
    const uint64_t pos = uint64_t(prefix_c) + k;
    *reinterpret_cast<uint4*>(pm.idx + pos) =
        make_uint4(base + (e[0] & 0xFFFFu), base + (e[1] & 0xFFFFu), base + (e[2] & 0xFFFFu),
                   base + (e[3] & 0xFFFFu));
    *reinterpret_cast<uint32_t*>(pm.val + pos) =
        ((e[0] >> 16) & 0xFFu) | (((e[1] >> 16) & 0xFFu) << 8) | (((e[2] >> 16) & 0xFFu) << 16) |
        (((e[3] >> 16) & 0xFFu) << 24);
  }
  for (uint32_t k = head + body + uint32_t(lane); k < agg; k += 32) {
    const uint32_t ent = ring[(pm.ring_start + k) & kRingMask];
    const uint64_t pos = uint64_t(prefix_c) + k;
    if (pos < pm.code_cap) {
      pm.idx[pos] = base + (ent & 0xFFFFu);
      pm.val[pos] = uint8_t(ent >> 16);
    }
  }
  const uint64_t nblocks = pm.scale_cap;
  const uint32_t block_base = uint32_t(pm.scale_base);
  for (uint32_t k = uint32_t(lane); k < pm.agg_s; k += 32) {
    const uint32_t ent = sring[k];
    const uint64_t pos = uint64_t(prefix_s) + k;
    if (pos < nblocks) {
      pm.sidx[pos] = block_base + (ent & 0xFFu);
      pm.sval[pos] = uint8_t(ent >> 8);
    }
  }
}

template <int F>
__device__ __forceinline__ void lookback_loop(const MxLaunch& a, MxShared& sh, const uint32_t* ring,
                                              int w, int lane, bool multi) {
  for (uint32_t i = uint32_t(w);;) {
    const bool ok = helper_wait(&sh.agg_ready[i % kPendSlots], (i / kPendSlots) & 1u, a);
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    int more = 0;
    if (lane == 0) {
      for (int b = 1; b < kLookbackBatch; ++b) {
        const uint32_t ii = i + uint32_t(b * kEncLookbackWarps);
        if (!mbar_test_wait(&sh.agg_ready[ii % kPendSlots], (ii / kPendSlots) & 1u)) break;
        more = b;
      }
    }
    more = __shfl_sync(0xFFFFFFFFu, more, 0);
    int nb = 0;
    bool end = false;
    // NVFP4 measured faster with 2 look-back words per lane than with the
    // pipeline's default (14.12 against 14.22 ms on the 8.03B step)
    constexpr int kW = F == kFmtNvfp4 ? 2 : kLookbackPerLane;
    uint64_t win[kLookbackBatch][kW];
#pragma unroll
    for (int b = 0; b < kLookbackBatch; ++b) {
      if (b > more || end) continue;
      const uint32_t ii = i + uint32_t(b * kEncLookbackWarps);
      const int q = int(ii % kPendSlots);
      if (b > 0) mbar_test_wait(&sh.agg_ready[q], (ii / kPendSlots) & 1u);  // acquire for every lane
      const ParkedMeta& pm = sh.parked[q];
      if (pm.last == 2u) {
        end = true;
        continue;
      }
      if (pm.tile != pm.first)
        load_window<StatusPacked, MxLaunch, kW>(a, int64_t(pm.tile) - 1, pm.first, lane, win[b]);
      nb = b + 1;
    }
#pragma unroll
    for (int b = 0; b < kLookbackBatch; ++b) {
      if (b >= nb) continue;
      const uint32_t ii = i + uint32_t(b * kEncLookbackWarps);
      const int q = int(ii % kPendSlots);
      const ParkedMeta pm = sh.parked[q];
      const uint64_t agg = uint64_t(pm.agg_c) | (uint64_t(pm.agg_s) << 32);
      const uint64_t prefix =
          resolve_prefix<StatusPacked, MxLaunch, 32, kW>(a, pm.tile, pm.first, agg, lane, win[b]);
      const uint32_t prefix_c = uint32_t(prefix), prefix_s = uint32_t(prefix >> 32);
      if (lane == 0 && pm.last == 1u) {
        const uint32_t t = multi ? pm.tensor : 0u;
        a.counts_out[2 * t] = uint64_t(prefix_c) + pm.agg_c;
        a.counts_out[2 * t + 1] = uint64_t(prefix_s) + pm.agg_s;
      }
      copy_out<F>(pm, prefix_c, prefix_s, ring, sh.sring[q], lane);
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        *reinterpret_cast<volatile uint32_t*>(&sh.ring_tail) = pm.ring_start + pm.agg_c;
        mbar_arrive(&sh.slot_free[q]);
      }
    }
    if (end) break;
    i += uint32_t(nb * kEncLookbackWarps);
  }
}

// ------------------------------------------------------------ compute warps
// Per tile each compute thread handles kMxRounds rounds of kMxPerThread
// consecutive elements, so a 32-element block spans 4 consecutive lanes.
constexpr int kMxPerThread = 8;
constexpr int kMxRounds = kEncTile / (kEncThreads * kMxPerThread);  // 2
static_assert(kMxRounds == 2, "two rounds pack into the 16-bit fields of one word");

// Largest magnitude of 8 values; NaN if any of them is NaN.
__device__ __forceinline__ float abs_max_nan(float a, float b) {
  float r;
  asm("{\n\t.reg .f32 x, y;\n\tabs.f32 x, %1;\n\tabs.f32 y, %2;\n\t"
      "max.NaN.f32 %0, x, y;\n\t}" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// E8M0 scale byte of the block this thread's 8 elements belong to (lanes
// 4b .. 4b+3 hold block b), for an element format whose largest normal has
// exponent EMAX. The block maximum is a non-negative float or NaN (max.NaN
// propagates NaN), so its bit pattern's exponent field E is 255 exactly for
// a non-finite block. All 32 lanes must call.
template <uint32_t EMAX>
__device__ __forceinline__ uint32_t block_scale8(const float4& a, const float4& b) {
  float m = max_nan(max_nan(abs_max_nan(a.x, a.y), abs_max_nan(a.z, a.w)),
                    max_nan(abs_max_nan(b.x, b.y), abs_max_nan(b.z, b.w)));
  m = max_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  m = max_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  const uint32_t e = __float_as_uint(m) >> 23;  // sign is clear
  return e == 255u ? 0xFFu : (e > EMAX ? e - EMAX : 0u);
}

// ------------------------------------------------------------ NVFP4 pieces
// Every step is one FP32 operation rounded to nearest even, in this order.

// E4M3 code of a non-negative finite u: round to nearest even, values past
// 448 clamped to 448 (the saturating hardware convert).
__device__ __forceinline__ uint32_t e4m3_of(float u) {
  return cvt_e4m3x2(0.0f, u) & 0xFFu;
}

// Value of an E4M3 code (exact: E4M3 -> f16 -> f32).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(uint16_t(c)));
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(uint16_t(h2 & 0xFFFFu)));
  return f;
}

// Block scale byte of the 16-element block this thread's 8 elements belong
// to (lanes 2b, 2b+1 hold block b) under tensor scale ts: 0x7F for a block
// holding a NaN or an infinity, 0 when ts is 0, else E4M3((amax / 6) / ts).
// All 32 lanes must call.
__device__ __forceinline__ uint32_t nv_block_scale8(const float4& a, const float4& b, float ts) {
  float m = max_nan(max_nan(abs_max_nan(a.x, a.y), abs_max_nan(a.z, a.w)),
                    max_nan(abs_max_nan(b.x, b.y), abs_max_nan(b.z, b.w)));
  m = max_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  if ((__float_as_uint(m) >> 23) == 255u) return 0x7Fu;
  if (ts == 0.0f) return 0u;
  return e4m3_of(__fdiv_rn(__fdiv_rn(m, 6.0f), ts));
}

// Codes of 8 elements under block scale byte d and tensor scale ts: the
// E2M1 of v * (1 / (dec(d) * ts)); all 0 when the block has no usable scale.
__device__ __forceinline__ uint32_t nv_codes8(const float4& a, const float4& b, uint32_t d, float ts) {
  if (d == 0x7Fu || d == 0u) return 0u;
  const float x = __fmul_rn(e4m3_value(d), ts);
  if (x == 0.0f) return 0u;
  const float r = __frcp_rn(x);
  if (!isfinite(r)) return 0u;
  uint32_t q;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(q)
      : "f"(__fmul_rn(a.x, r)), "f"(__fmul_rn(a.y, r)), "f"(__fmul_rn(a.z, r)),
        "f"(__fmul_rn(a.w, r)), "f"(__fmul_rn(b.x, r)), "f"(__fmul_rn(b.y, r)),
        "f"(__fmul_rn(b.z, r)), "f"(__fmul_rn(b.w, r)));
  return q;
}

// Four change flags in byte order (bit b = byte b) from the 0x80 bytes of
// nonzero_bytes: the same multiply as gather_flags8 with one word.
__device__ __forceinline__ uint32_t gather_flags4(uint32_t z) {
  return (((z >> 7) * 0x00204081u) >> 21) & 0xFu;
}

// One 0x80 per byte of x that is non-zero (x = new ^ old codes).
__device__ __forceinline__ uint32_t nonzero_bytes(uint32_t x) {
  return (((x & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | x) & 0x80808080u;
}

// Eight change flags in element order (bit e = element e) from the 0x80
// bytes of nonzero_bytes for elements 0-3 (z0) and 4-7 (z1). After the
// shifts the flags sit at bits 8e (e < 4) and 8(e - 4) + 4; multiplying by
// 1 + 2^7 + 2^14 + 2^21 copies bit p to p, p+7, p+14 and p+21, and for these
// eight p all copies land on distinct bits (so nothing carries), with the
// copy of element e's flag at bit 21 + e.
__device__ __forceinline__ uint32_t gather_flags8(uint32_t z0, uint32_t z1) {
  return ((((z0 >> 7) | (z1 >> 3)) * 0x00204081u) >> 21) & 0xFFu;
}

// A thread's 8-element group of a tail or unaligned tile, read from global
// memory: elements past the end read as +0 (no effect on the block maximum,
// code 0) and bytes past the end are never reported.
struct GroupIn {
  float4 v0, v1;  // the group's 8 master values
  uint2 pc;       // its previous code bytes
  uint32_t ps;    // the previous scale of its block (leader lanes only)
};

template <int F>
__device__ __forceinline__ GroupIn load_group_inline(const float* master, const uint8_t* prev_codes,
                                                     const uint8_t* prev_scales, uint64_t base,
                                                     uint32_t len, uint32_t li, uint32_t lb,
                                                     bool leader) {
  constexpr uint32_t kGroupBytes = kMxPerThread / Fmt<F>::kElemsPerByte;
  constexpr uint32_t kBlock = Fmt<F>::kBlock;
  float mm[kMxPerThread];
#pragma unroll
  for (int e = 0; e < kMxPerThread; ++e) mm[e] = li + e < len ? master[base + li + e] : 0.0f;
  uint32_t pp[2] = {0u, 0u};
  const uint64_t cb = (base + li) / Fmt<F>::kElemsPerByte;  // first code byte
#pragma unroll
  for (int e = 0; e < int(kGroupBytes); ++e) {
    const bool valid = li + uint32_t(e) * Fmt<F>::kElemsPerByte < len;
    pp[e >> 2] |= (valid ? uint32_t(prev_codes[cb + e]) : 0u) << (8 * (e & 3));
  }
  GroupIn g;
  g.v0 = make_float4(mm[0], mm[1], mm[2], mm[3]);
  g.v1 = make_float4(mm[4], mm[5], mm[6], mm[7]);
  g.pc = make_uint2(pp[0], pp[1]);
  g.ps = (leader && lb * kBlock < len) ? uint32_t(prev_scales[(base / kBlock) + lb]) : 0u;
  return g;
}

// The same, out of line (the FP4 formats measured faster with it out of their
// hot loop: NVFP4 14.61 against 15.03 ms on the 8.03B step; E4M3 slower).
template <int F>
__device__ __noinline__ GroupIn load_group_generic(const float* master, const uint8_t* prev_codes,
                                                   const uint8_t* prev_scales, uint64_t base,
                                                   uint32_t len, uint32_t li, uint32_t lb,
                                                   bool leader) {
  return load_group_inline<F>(master, prev_codes, prev_scales, base, len, li, lb, leader);
}

template <int F, bool MULTI>
__device__ __forceinline__ void compute_loop(const MxLaunch& a, MxShared& sh, uint8_t* stages,
                                             uint32_t* ring, int tid, int lane, int warp) {
  constexpr uint32_t kStageBytes = Stage<F>::kBytes, kStageCodeBytes = Stage<F>::kCodeBytes;
  constexpr int kEncStages = Stage<F>::kStages;
  constexpr uint32_t kEncRing = Stage<F>::kRing, kRingMask = Stage<F>::kRingMask;
  constexpr bool kFp4 = F != kFmtE4M3;  // two codes per byte
  constexpr uint32_t kBlock = Fmt<F>::kBlock;
  constexpr int kLanesPerBlock = int(kBlock) / kMxPerThread;  // 4 or 2
  // code bytes per 8-element group, and change flags per round
  constexpr uint32_t kGroupBytes = kMxPerThread / Fmt<F>::kElemsPerByte;
  uint32_t posted = 0, ring_head = 0;
  bool failed = false;
  const bool leader = (lane & (kLanesPerBlock - 1)) == 0;  // lane that owns its block's scale
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kEncStages);
    failed |= !wait_or_flag(&sh.full[s], (it / kEncStages) & 1u, a);
    const StageMeta m = sh.meta[s];
    const bool live = m.mode != kModeEnd;
    const bool bulk = m.mode == kModeBulk;
    const uint64_t base = m.base;
    const uint32_t len = m.len;
    const uint8_t* stage = stages + size_t(s) * kStageBytes;

    // ---- quantize + compare: 8 consecutive elements per thread per round
    uint32_t nc[kMxRounds][2];  // new code bytes, byte 0 in the low byte of word 0 (FP4: word 0 only)
    uint32_t ns = 0;            // byte j: new scale of this thread's block in round j
    uint32_t flags = 0;         // bit 8j + e: code byte e of round j changed
    uint32_t sflags = 0;        // bit j: the block of round j changed its scale (leaders only)
    // MXFP8 compiles this loop apart for a staged (full, aligned) tile and for
    // the generic one; the FP4 formats measured faster with one body that tests
    // the mode at run time (MXFP4 8.86 against 9.03 ms on the 8.03B step)
    auto quantize = [&](auto bulk_tag) {
      constexpr bool kBulk = decltype(bulk_tag)::value;
#pragma unroll
      for (int j = 0; j < kMxRounds; ++j) {
        const uint32_t slot = uint32_t(j * kEncThreads + tid);  // 8-element group within the tile
        const uint32_t li = slot * kMxPerThread;
        const uint32_t lb = slot / kLanesPerBlock;              // block within the tile
        float4 v0, v1;
        uint2 pc = make_uint2(0u, 0u);
        uint32_t ps = 0;
        if constexpr (kBulk) {
          const float4* sm = reinterpret_cast<const float4*>(stage);
          v0 = sm[2 * slot];
          v1 = sm[2 * slot + 1];
          if constexpr (kFp4)
            pc.x = reinterpret_cast<const uint32_t*>(stage + kStageMasterBytes)[slot];
          else
            pc = reinterpret_cast<const uint2*>(stage + kStageMasterBytes)[slot];
          if (leader) ps = stage[kStageMasterBytes + kStageCodeBytes + lb];
        } else {
          GroupIn g;
          if constexpr (kFp4)
            g = load_group_generic<F>(m.master, m.prev_codes, m.prev_scales, base, len, li, lb, leader);
          else
            g = load_group_inline<F>(m.master, m.prev_codes, m.prev_scales, base, len, li, lb, leader);
          v0 = g.v0;
          v1 = g.v1;
          pc = g.pc;
          ps = g.ps;
        }
        uint32_t sb;
        if constexpr (F == kFmtNvfp4)
          sb = nv_block_scale8(v0, v1, m.tscale);
        else
          sb = block_scale8<Fmt<F>::kEmax>(v0, v1);
        uint32_t f4;
        if constexpr (kFp4) {
          if constexpr (F == kFmtNvfp4)
            nc[j][0] = nv_codes8(v0, v1, sb, m.tscale);
          else
            nc[j][0] = fp4_codes8(v0, v1, sb);
          nc[j][1] = 0u;
          uint32_t z = nonzero_bytes(nc[j][0] ^ pc.x);
          if constexpr (!kBulk) {
            // keep only the code bytes inside the tile
            const uint32_t nb = li >= len ? 0u : (len - li >= 8u ? 4u : (len - li + 1u) / 2u);
            z &= nb >= 4u ? 0xFFFFFFFFu : (1u << (8 * nb)) - 1u;
          }
          f4 = gather_flags4(z);
        } else {
          nc[j][0] = mx_codes4(v0, sb);
          nc[j][1] = mx_codes4(v1, sb);
          uint32_t z0 = nonzero_bytes(nc[j][0] ^ pc.x), z1 = nonzero_bytes(nc[j][1] ^ pc.y);
          if constexpr (!kBulk) {
            // keep only elements inside the tile
            const uint32_t nvalid = li >= len ? 0u : (len - li >= 8u ? 8u : len - li);
            const uint64_t keep =  // one 0xFF byte per valid element
                nvalid >= 8u ? ~uint64_t(0) : (uint64_t(1) << (8 * nvalid)) - 1u;
            z0 &= uint32_t(keep);
            z1 &= uint32_t(keep >> 32);
          }
          f4 = gather_flags8(z0, z1);
        }
        ns |= sb << (8 * j);
        flags |= f4 << (8 * j);
        if (leader && (kBulk || lb * kBlock < len) && sb != ps) sflags |= 1u << j;
      }
    };
    if constexpr (F == kFmtE4M3) {
      if (bulk) quantize(std::true_type{}); else quantize(std::false_type{});
    } else {
#pragma unroll
      for (int j = 0; j < kMxRounds; ++j) {
        const uint32_t slot = uint32_t(j * kEncThreads + tid);  // 8-element group within the tile
        const uint32_t li = slot * kMxPerThread;
        const uint32_t lb = slot / kLanesPerBlock;              // block within the tile
        float4 v0, v1;
        uint2 pc = make_uint2(0u, 0u);
        uint32_t ps = 0;
        if (bulk) {
          const float4* sm = reinterpret_cast<const float4*>(stage);
          v0 = sm[2 * slot];
          v1 = sm[2 * slot + 1];
          if constexpr (kFp4)
            pc.x = reinterpret_cast<const uint32_t*>(stage + kStageMasterBytes)[slot];
          else
            pc = reinterpret_cast<const uint2*>(stage + kStageMasterBytes)[slot];
          if (leader) ps = stage[kStageMasterBytes + kStageCodeBytes + lb];
        } else {
          GroupIn g;
          if constexpr (kFp4)
            g = load_group_generic<F>(m.master, m.prev_codes, m.prev_scales, base, len, li, lb, leader);
          else
            g = load_group_inline<F>(m.master, m.prev_codes, m.prev_scales, base, len, li, lb, leader);
          v0 = g.v0;
          v1 = g.v1;
          pc = g.pc;
          ps = g.ps;
        }
        uint32_t sb;
        if constexpr (F == kFmtNvfp4)
          sb = nv_block_scale8(v0, v1, m.tscale);
        else
          sb = block_scale8<Fmt<F>::kEmax>(v0, v1);
        uint32_t f4;
        if constexpr (kFp4) {
          if constexpr (F == kFmtNvfp4)
            nc[j][0] = nv_codes8(v0, v1, sb, m.tscale);
          else
            nc[j][0] = fp4_codes8(v0, v1, sb);
          nc[j][1] = 0u;
          uint32_t z = nonzero_bytes(nc[j][0] ^ pc.x);
          if (!bulk) {
            // keep only the code bytes inside the tile
            const uint32_t nb = li >= len ? 0u : (len - li >= 8u ? 4u : (len - li + 1u) / 2u);
            z &= nb >= 4u ? 0xFFFFFFFFu : (1u << (8 * nb)) - 1u;
          }
          f4 = gather_flags4(z);
        } else {
          nc[j][0] = mx_codes4(v0, sb);
          nc[j][1] = mx_codes4(v1, sb);
          uint32_t z0 = nonzero_bytes(nc[j][0] ^ pc.x), z1 = nonzero_bytes(nc[j][1] ^ pc.y);
          if (!bulk) {
            // keep only elements inside the tile
            const uint32_t nvalid = li >= len ? 0u : (len - li >= 8u ? 8u : len - li);
            const uint64_t keep =  // one 0xFF byte per valid element
                nvalid >= 8u ? ~uint64_t(0) : (uint64_t(1) << (8 * nvalid)) - 1u;
            z0 &= uint32_t(keep);
            z1 &= uint32_t(keep >> 32);
          }
          f4 = gather_flags8(z0, z1);
        }
        ns |= sb << (8 * j);
        flags |= f4 << (8 * j);
        if (leader && lb * kBlock < len && sb != ps) sflags |= 1u << j;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);

    // ---- refresh the previous view now
    auto refresh = [&](auto bulk_tag) {
      constexpr bool kBulk = decltype(bulk_tag)::value;
#pragma unroll
      for (int j = 0; j < kMxRounds; ++j) {
        const uint32_t f = (flags >> (8 * j)) & 0xFFu;
        const uint32_t li = uint32_t(j * kEncThreads + tid) * kMxPerThread;
        if (f != 0u) {
          const uint64_t cb = (base + li) / Fmt<F>::kElemsPerByte;  // first code byte
          if constexpr (kBulk) {
            if constexpr (kFp4)
              *reinterpret_cast<uint32_t*>(m.prev_codes + cb) = nc[j][0];
            else
              *reinterpret_cast<uint2*>(m.prev_codes + cb) = make_uint2(nc[j][0], nc[j][1]);
          } else {
#pragma unroll
            for (int e = 0; e < int(kGroupBytes); ++e)
              if ((f >> e) & 1u) m.prev_codes[cb + e] = uint8_t(nc[j][e >> 2] >> (8 * (e & 3)));
          }
        }
        if ((sflags >> j) & 1u) m.prev_scales[base / kBlock + li / kBlock] = uint8_t(ns >> (8 * j));
      }
    };
    if constexpr (F == kFmtE4M3) {
      if (bulk) refresh(std::true_type{}); else refresh(std::false_type{});
    } else {
#pragma unroll
      for (int j = 0; j < kMxRounds; ++j) {
        const uint32_t f = (flags >> (8 * j)) & 0xFFu;
        const uint32_t li = uint32_t(j * kEncThreads + tid) * kMxPerThread;
        if (f != 0u) {
          const uint64_t cb = (base + li) / Fmt<F>::kElemsPerByte;  // first code byte
          if (bulk) {
            if constexpr (kFp4)
              *reinterpret_cast<uint32_t*>(m.prev_codes + cb) = nc[j][0];
            else
              *reinterpret_cast<uint2*>(m.prev_codes + cb) = make_uint2(nc[j][0], nc[j][1]);
          } else {
#pragma unroll
            for (int e = 0; e < int(kGroupBytes); ++e)
              if ((f >> e) & 1u) m.prev_codes[cb + e] = uint8_t(nc[j][e >> 2] >> (8 * (e & 3)));
          }
        }
        if ((sflags >> j) & 1u) m.prev_scales[base / kBlock + li / kBlock] = uint8_t(ns >> (8 * j));
      }
    }

    // ---- rank. Codes: one warp scan of the two per-round counts in 16-bit
    // fields (a field never exceeds 32 x 8 = 256). Scales: one ballot per round.
    const uint32_t cnts = uint32_t(__popc(flags & 0xFFu)) | (uint32_t(__popc(flags & 0xFF00u)) << 16);
    uint32_t incl = cnts;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const uint32_t excl = incl - cnts;
    const uint32_t lt = lanemask_lt();
    const uint32_t bal0 = __ballot_sync(0xFFFFFFFFu, sflags & 1u);
    const uint32_t bal1 = __ballot_sync(0xFFFFFFFFu, sflags & 2u);
    const uint32_t stot = uint32_t(__popc(bal0)) | (uint32_t(__popc(bal1)) << 8);
    const uint32_t srank = uint32_t(__popc(bal0 & lt)) | (uint32_t(__popc(bal1 & lt)) << 8);
    const int pc = int(it & 1u);
    if (lane == 31) sh.warp_tot[pc][warp] = incl;
    if (lane == 0) sh.warp_stot[pc][warp] = stot;
    if (compute_barrier_or(failed || !live)) break;

    // across warps, in tile order (round-major, then warp): codes in 16-bit
    // fields (at most 8 x 256 = 2048), scales in bytes (at most 8 x 8 = 64)
    const uint32_t t = lane < kWarps ? sh.warp_tot[pc][lane] : 0u;
    const uint32_t ts = lane < kWarps ? sh.warp_stot[pc][lane] : 0u;
    uint32_t sc = t, ss = ts;
#pragma unroll
    for (int o = 1; o < kWarps; o <<= 1) {
      const uint32_t vc = __shfl_up_sync(0xFFFFFFFFu, sc, o);
      const uint32_t vs = __shfl_up_sync(0xFFFFFFFFu, ss, o);
      if (lane >= o) { sc += vc; ss += vs; }
    }
    const uint32_t bc = __shfl_sync(0xFFFFFFFFu, sc - t, warp);   // warps before this one
    const uint32_t bs = __shfl_sync(0xFFFFFFFFu, ss - ts, warp);
    const uint32_t ac = __shfl_sync(0xFFFFFFFFu, sc, kWarps - 1);  // all warps
    const uint32_t as = __shfl_sync(0xFFFFFFFFu, ss, kWarps - 1);
    const uint32_t tot0 = ac & 0xFFFFu, tot1 = ac >> 16;
    const uint32_t round_off0 = (bc & 0xFFFFu) + (excl & 0xFFFFu);
    const uint32_t round_off1 = tot0 + (bc >> 16) + (excl >> 16);
    const uint32_t agg_c = tot0 + tot1;
    const uint32_t stot0 = as & 0xFFu;
    const uint32_t agg_s = stot0 + ((as >> 8) & 0xFFu);
    if (tid == 0) {
      const uint64_t v = uint64_t(agg_c) | (uint64_t(agg_s) << 32);
      st_relaxed_u64(a.status + m.tile,
                     StatusPacked::make(uint64_t(m.tile) == m.first ? kFlagPrefix : kFlagAggregate,
                                        0u, v));
    }

    // ---- room: the parked slot must be free and the ring must hold agg_c more
    const int q = int(posted % kPendSlots);
    if (posted >= uint32_t(kPendSlots))
      failed |= !wait_or_flag(&sh.slot_free[q], ((posted - kPendSlots) / kPendSlots) & 1u, a);
    failed |= !wait_ring_room<64>(&sh.ring_tail, ring_head, agg_c, uint32_t(kEncRing), a);

    // ---- park the compacted tile
#pragma unroll
    for (int j = 0; j < kMxRounds; ++j) {
      uint32_t f = (flags >> (8 * j)) & 0xFFu;
      if (f == 0u) continue;
      const uint32_t li = uint32_t(j * kEncThreads + tid) * kMxPerThread;
      uint32_t r = ring_head + (j == 0 ? round_off0 : round_off1);
      do {
        const uint32_t e = uint32_t(__ffs(f)) - 1u;
        f &= f - 1u;
        const uint32_t word = (e & 4u) ? nc[j][1] : nc[j][0];
        ring[r & kRingMask] =
            (li / Fmt<F>::kElemsPerByte + e) | (((word >> (8 * (e & 3))) & 0xFFu) << 16);
        ++r;
      } while (f != 0u);
    }
#pragma unroll
    for (int j = 0; j < kMxRounds; ++j) {
      if (!((sflags >> j) & 1u)) continue;
      const uint32_t pos = (j > 0 ? stot0 : 0u) + ((bs >> (8 * j)) & 0xFFu) + ((srank >> (8 * j)) & 0xFFu);
      const uint32_t lb = uint32_t(j * kEncThreads + tid) / kLanesPerBlock;
      sh.sring[q][pos] = uint16_t(lb | (((ns >> (8 * j)) & 0xFFu) << 8));
    }
    if (tid == 0) {
      ParkedMeta pm;
      pm.tile = m.tile;
      pm.tensor = m.tensor;
      pm.agg_c = agg_c;
      pm.agg_s = agg_s;
      pm.last = (base + len == m.n) ? 1u : 0u;
      pm.ring_start = ring_head;
      pm.first = m.first;
      pm.n = m.n;
      pm.base = base;
      pm.code_base = base / Fmt<F>::kElemsPerByte;
      pm.code_cap = (m.n + Fmt<F>::kElemsPerByte - 1) / Fmt<F>::kElemsPerByte;
      pm.scale_base = base / kBlock;
      pm.scale_cap = (m.n + kBlock - 1) / kBlock;
      pm.idx = m.idx;
      pm.val = m.val;
      pm.sidx = m.sidx;
      pm.sval = m.sval;
      sh.parked[q] = pm;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.agg_ready[q]);
    ++posted;
    ring_head += agg_c;
  }
  for (uint32_t e = posted > uint32_t(kPendSlots) ? posted - kPendSlots : 0u; e < posted; ++e)
    wait_or_flag(&sh.slot_free[e % kPendSlots], (e / kPendSlots) & 1u, a);
  compute_barrier();
  for (int k = 0; k < kEncLookbackWarps; ++k) {
    const uint32_t i = posted + uint32_t(k);
    const int q = int(i % kPendSlots);
    if (tid == 0) {
      ParkedMeta pm{};
      pm.last = 2u;
      sh.parked[q] = pm;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.agg_ready[q]);
  }
}

// Resident CTAs per SM the register budget is sized for: the FP4 formats'
// smaller stages and ring leave shared memory for more CTAs than E4M3's.
#ifndef PULSE_MX4_MIN_BLOCKS
#define PULSE_MX4_MIN_BLOCKS 3
#endif
template <int F>
constexpr int mx_min_blocks() {
  return F == kFmtE4M3 ? kEncMinBlocks : PULSE_MX4_MIN_BLOCKS;
}

template <int F, bool MULTI>
__global__ void __launch_bounds__(kEncBlockThreads, mx_min_blocks<F>())
    encode_mx_kernel(const __grid_constant__ MxLaunch a) {
  constexpr uint32_t kStageBytes = Stage<F>::kBytes;
  constexpr int kEncStages = Stage<F>::kStages;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ MxShared sh;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 127) & ~uintptr_t(127));
  uint32_t* ring = reinterpret_cast<uint32_t*>(stages + size_t(kEncStages) * kStageBytes);

  if constexpr (MULTI) {
    if (blockIdx.x == 0) {
      for (int t = tid; t < a.ntensors; t += kEncBlockThreads) {
        if (a.tensors[t].n == 0) {
          a.counts_out[2 * t] = 0;
          a.counts_out[2 * t + 1] = 0;
        }
      }
    }
  }
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kEncStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kWarps);
      sh.meta[s] = StageMeta{};
      sh.meta[s].mode = kModeEnd;
    }
#pragma unroll
    for (int q = 0; q < kPendSlots; ++q) {
      mbar_init(&sh.agg_ready[q], kWarps);
      mbar_init(&sh.slot_free[q], 1);
      sh.parked[q] = ParkedMeta{};
      sh.parked[q].last = 2u;
    }
    sh.ring_tail = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp < kWarps) {
    compute_loop<F, MULTI>(a, sh, stages, ring, tid, lane, warp);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_loop<F, MULTI>(a, sh, stages);
  } else {
    lookback_loop<F>(a, sh, ring, warp - kFirstLookbackWarp, lane, MULTI);
  }
}

template <int F, bool MULTI>
int encode_mx_blocks_per_sm() {
  static int cached = [] {
    cudaFuncSetAttribute(encode_mx_kernel<F, MULTI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         int(Stage<F>::kDynSmem));
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, encode_mx_kernel<F, MULTI>,
                                                      kEncBlockThreads, Stage<F>::kDynSmem) != cudaSuccess ||
        b < 1)
      b = 1;
    return b;
  }();
  return cached;
}

// ------------------------------------------------------------ quantize
// The MX view of one tensor (initial state of the trainer's previous view
// and of a receiver), with the encode's arithmetic: 8 consecutive elements
// per thread, so block b of a warp's 256 elements is lanes 4b .. 4b+3.
constexpr int kQuantThreads = 256;

template <int F>
__global__ void __launch_bounds__(kQuantThreads)
    mx_quantize_kernel(const float* __restrict__ master, uint64_t n, uint8_t* __restrict__ codes,
                       uint8_t* __restrict__ scales, const uint32_t* __restrict__ amax_bits,
                       float* __restrict__ tscale_out) {
  constexpr uint32_t kGroupBytes = kMxPerThread / Fmt<F>::kElemsPerByte;
  constexpr uint32_t kBlock = Fmt<F>::kBlock;
  constexpr int kLanesPerBlock = int(kBlock) / kMxPerThread;
  const float ts = F == kFmtNvfp4 ? __fdiv_rn(__uint_as_float(*amax_bits), 2688.0f) : 0.0f;
  if (F == kFmtNvfp4 && blockIdx.x == 0 && threadIdx.x == 0) *tscale_out = ts;
  const bool vec = (reinterpret_cast<uintptr_t>(master) % 16u == 0) &&
                   (reinterpret_cast<uintptr_t>(codes) % kGroupBytes == 0);
  const uint64_t groups = (n + kMxPerThread - 1) / kMxPerThread;
  const uint64_t stride = uint64_t(gridDim.x) * kQuantThreads;
  // every lane of a warp runs the same number of iterations (shuffles below)
  const uint64_t warp_first = uint64_t(blockIdx.x) * kQuantThreads + (threadIdx.x & ~31u);
  const int lane = threadIdx.x & 31;
  for (uint64_t g0 = warp_first; g0 < groups; g0 += stride) {
    const uint64_t i = (g0 + lane) * kMxPerThread;
    const bool full = vec && i + kMxPerThread <= n;
    float v[kMxPerThread];
    if (full) {
      const float4 a = *reinterpret_cast<const float4*>(master + i);
      const float4 b = *reinterpret_cast<const float4*>(master + i + 4);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
      for (int e = 0; e < kMxPerThread; ++e) v[e] = i + e < n ? master[i + e] : 0.0f;
    }
    const float4 a = make_float4(v[0], v[1], v[2], v[3]);
    const float4 b = make_float4(v[4], v[5], v[6], v[7]);
    uint32_t sb, c0, c1;
    if constexpr (F == kFmtNvfp4)
      sb = nv_block_scale8(a, b, ts);
    else
      sb = block_scale8<Fmt<F>::kEmax>(a, b);
    if constexpr (F == kFmtNvfp4) {
      c0 = nv_codes8(a, b, sb, ts);
      c1 = 0u;
    } else if constexpr (F == kFmtE2M1) {
      c0 = fp4_codes8(a, b, sb);
      c1 = 0u;
    } else {
      c0 = mx_codes4(a, sb);
      c1 = mx_codes4(b, sb);
    }
    const uint64_t cb = i / Fmt<F>::kElemsPerByte;  // first code byte
    if (full) {
      if constexpr (F != kFmtE4M3)
        *reinterpret_cast<uint32_t*>(codes + cb) = c0;
      else
        *reinterpret_cast<uint2*>(codes + cb) = make_uint2(c0, c1);
    } else {
      for (int e = 0; e < int(kGroupBytes); ++e)
        if (i + uint64_t(e) * Fmt<F>::kElemsPerByte < n)
          codes[cb + e] = uint8_t((e < 4 ? c0 : c1) >> (8 * (e & 3)));
    }
    if ((lane & (kLanesPerBlock - 1)) == 0 && i < n) scales[i / kBlock] = uint8_t(sb);
  }
}

// ------------------------------------------------------------ tensor maxima
// NVFP4's tensor scale needs each tensor's largest finite magnitude before
// any block is encoded: one pass over the master, 4096-element tiles, a
// block maximum per tile and one atomicMax per tile on the bit pattern (a
// non-negative float orders like its bits). amax_bits is zeroed beforehand.
constexpr int kAmaxThreads = 256;

// Largest finite magnitude of every tensor (bit pattern of a non-negative
// float, so unsigned order is float order). A CTA walks tiles blockIdx.x,
// blockIdx.x + grid, ...; each thread keeps a running maximum while the tiles
// stay in one tensor and a warp folds it into amax_bits[t] with one atomicMax
// when the tensor changes and at the end. A full, aligned tile is read with
// all four 16-byte loads of a thread in flight at once.
template <bool MULTI>
__global__ void __launch_bounds__(kAmaxThreads)
    mx_amax_kernel(const MxTensorDesc one, const MxTensorDesc* tensors, const uint64_t* tile_begin,
                   int ntensors, uint64_t total_tiles, uint32_t* amax_bits) {
  constexpr int kLoads = kEncTile / (4 * kAmaxThreads);  // float4 loads per thread per tile
  static_assert(kLoads * 4 * kAmaxThreads == kEncTile, "a tile is whole float4 rounds");
  const int tid = threadIdx.x, lane = tid & 31;
  int cur = MULTI ? -1 : 0;
  uint64_t cur_begin = 1, cur_end = 0;
  MxTensorDesc d = one;
  float m = 0.0f;  // this thread's maximum over the tiles of tensor `cur` seen so far
  auto take = [&](float v) {
    const float x = fabsf(v);
    if (x <= 3.40282347e38f) m = fmaxf(m, x);  // finite values only (NaN fails the test)
  };
  auto flush = [&]() {  // uniform over the CTA: every thread walks the same tiles
    const uint32_t wm = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m));
    if (lane == 0 && cur >= 0 && wm != 0u) atomicMax(amax_bits + cur, wm);
    m = 0.0f;
  };
  for (uint64_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
    if constexpr (MULTI) {
      if (tile < cur_begin || tile >= cur_end) {
        flush();
        cur = find_tensor(tile_begin, ntensors, tile);
        d = tensors[cur];
        cur_begin = d.tile_begin;
        cur_end = tile_begin[cur + 1];
      }
    }
    const uint64_t base = (tile - d.tile_begin) * kEncTile;
    const uint32_t len = uint32_t(d.n - base < uint64_t(kEncTile) ? d.n - base : uint64_t(kEncTile));
    const float* src = d.master + base;
    if (len == uint32_t(kEncTile) && (reinterpret_cast<uintptr_t>(src) % 16u) == 0) {
      uint4 q[kLoads];
#pragma unroll
      for (int r = 0; r < kLoads; ++r) q[r] = ld_stream_u4_ro(src + (r * kAmaxThreads + tid) * 4);
#pragma unroll
      for (int r = 0; r < kLoads; ++r) {
        take(__uint_as_float(q[r].x));
        take(__uint_as_float(q[r].y));
        take(__uint_as_float(q[r].z));
        take(__uint_as_float(q[r].w));
      }
    } else {
      for (uint32_t k = uint32_t(tid); k < len; k += kAmaxThreads) take(src[k]);
    }
  }
  flush();
}

}  // namespace

int encode_mx_grid_size(int device, int format) {
  int a, b;
  if (format == kFmtNvfp4) {
    a = encode_mx_blocks_per_sm<kFmtNvfp4, true>();
    b = encode_mx_blocks_per_sm<kFmtNvfp4, false>();
  } else if (format == kFmtE2M1) {
    a = encode_mx_blocks_per_sm<kFmtE2M1, true>();
    b = encode_mx_blocks_per_sm<kFmtE2M1, false>();
  } else {
    a = encode_mx_blocks_per_sm<kFmtE4M3, true>();
    b = encode_mx_blocks_per_sm<kFmtE4M3, false>();
  }
  return sm_count(device) * (a < b ? a : b);
}

namespace {
template <int F>
cudaError_t launch_encode_mx_t(const MxLaunch& a, bool multi, int grid, cudaStream_t stream) {
  if (multi) {
    encode_mx_blocks_per_sm<F, true>();
    encode_mx_kernel<F, true><<<grid, kEncBlockThreads, Stage<F>::kDynSmem, stream>>>(a);
  } else {
    encode_mx_blocks_per_sm<F, false>();
    encode_mx_kernel<F, false><<<grid, kEncBlockThreads, Stage<F>::kDynSmem, stream>>>(a);
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_encode_mx(const MxLaunch& a, int format, bool multi, int grid,
                             cudaStream_t stream) {
  if (format == kFmtNvfp4) return launch_encode_mx_t<kFmtNvfp4>(a, multi, grid, stream);
  return format == kFmtE2M1 ? launch_encode_mx_t<kFmtE2M1>(a, multi, grid, stream)
                            : launch_encode_mx_t<kFmtE4M3>(a, multi, grid, stream);
}

cudaError_t launch_mx_amax(const MxLaunch& a, bool multi, uint32_t* amax_bits, cudaStream_t stream) {
  if (a.total_tiles == 0) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t cap = uint64_t(sm_count(dev)) * 8u;
  const unsigned grid = unsigned(a.total_tiles < cap ? a.total_tiles : cap);
  if (multi)
    mx_amax_kernel<true><<<grid, kAmaxThreads, 0, stream>>>(a.one, a.tensors, a.tile_begin,
                                                             a.ntensors, a.total_tiles, amax_bits);
  else
    mx_amax_kernel<false><<<grid, kAmaxThreads, 0, stream>>>(a.one, a.tensors, a.tile_begin,
                                                              a.ntensors, a.total_tiles, amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_mx_quantize(int format, const float* master, uint64_t n, uint8_t* codes,
                               uint8_t* scales, const uint32_t* amax_bits, float* tscale_out,
                               cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t warps = (n + 32 * kMxPerThread - 1) / (32 * kMxPerThread);
  const uint64_t blocks = (warps + kQuantThreads / 32 - 1) / (kQuantThreads / 32);
  const uint64_t cap = uint64_t(sm_count(dev)) * 8u;
  const int grid = int(blocks < cap ? blocks : cap);
  if (grid == 0) return cudaSuccess;
  if (format == kFmtNvfp4)
    mx_quantize_kernel<kFmtNvfp4><<<grid, kQuantThreads, 0, stream>>>(master, n, codes, scales,
                                                                      amax_bits, tscale_out);
  else if (format == kFmtE2M1)
    mx_quantize_kernel<kFmtE2M1><<<grid, kQuantThreads, 0, stream>>>(master, n, codes, scales,
                                                                     amax_bits, tscale_out);
  else
    mx_quantize_kernel<kFmtE4M3><<<grid, kQuantThreads, 0, stream>>>(master, n, codes, scales,
                                                                     amax_bits, tscale_out);
  return cudaGetLastError();
}

}  // namespace pulse
