// encode.cu -- fused cast + compare + order-preserving compaction.
//
// Trainer-side step of compute-visible weight sync: project the FP32 master
// to its BF16 view, compare with the previous view bit for bit, and emit the
// changed positions with their new absolute values in ascending order
// ("Taking Reinforcement Learning Cross Datacenter", talk 10:49-11:08; PULSE
// summary, section "Metodologia: PULSE -- 1. PULSESync"), refreshing the
// previous view in place.
//
// One launch covers one tensor or a whole model. Persistent, warp-specialized
// CTAs:
//  * producer warp: takes tile tickets from a global counter (so a tile's
//    predecessors always belong to CTAs that are already running) and fills
//    a kEncStages-deep shared-memory ring with bulk copies (cp.async.bulk,
//    completion counted in mbarrier transaction bytes);
//  * 8 compute warps: per 4096-element tile, cast + compare 4 consecutive
//    elements per thread per round, write changed BF16 values back to prev
//    at once (8-byte groups), rank changed elements with warp ballots and a
//    scan of the (round, warp) counts (one CTA barrier per tile), publish the
//    tile's count immediately, and park the tile's compacted patch (12-bit
//    local index + value, 4 bytes per entry) in a shared-memory entry ring;
//  * kEncLookbackWarps look-back warps: each takes a different parked tile,
//    resolves its global offset with a single-pass decoupled look-back
//    (Merrill & Garland, "Single-pass Parallel Prefix Scan with Decoupled
//    Look-back", 2016) reading kEncLookbackPerLane x 32 predecessor words per
//    round trip, publishes the inclusive prefix, copies the parked entries to
//    the patch with contiguous coalesced stores, and frees the slot. An L2
//    round trip to the status words costs microseconds while HBM is
//    saturated, so up to kPendSlots tiles per CTA wait in the ring while the
//    compute warps stream on.
// Every wait is bounded; a wait that gives up records PULSE_ERR_TIMEOUT and
// the kernel still finishes with all writes inside the caller's buffers.
#include "encode_common.cuh"

namespace pulse {
namespace {

using namespace enc;

// Look-back words per lane and round trip. A dense tile's look-back sits on
// its CTA's critical path, where 4 words a lane measured much slower than 2
// (2^28 flat at 40 / 70 % density: 0.75 / 1.03 ms against 0.64 / 0.88) for
// 0.7 % at 8 %; the sparser kernels of the pipeline take the default of 4.
#ifndef PULSE_BF16_LOOKBACK
#define PULSE_BF16_LOOKBACK 2
#endif
constexpr int kWindow = PULSE_BF16_LOOKBACK;

constexpr uint32_t kStageMasterBytes = kEncTile * 4;
constexpr uint32_t kStagePrevBytes = kEncTile * 2;
constexpr uint32_t kStageBytes = kStageMasterBytes + kStagePrevBytes;
constexpr size_t kDynSmem = size_t(kEncStages) * kStageBytes + size_t(kEncRing) * 4 + 128;

// Everything the compute warps need about a tile, written by the producer
// (which reads the tensor descriptor anyway) so the compute path touches no
// global descriptor memory.
struct StageMeta {
  uint32_t tile;    // global tile id
  uint32_t tensor;  // tensor index (0 in single-tensor mode)
  uint32_t mode;
  uint32_t len;     // elements in the tile
  uint64_t base;    // first element of the tile within its tensor
  uint64_t first;   // first global tile of the tensor
  uint64_t n;       // elements of the tensor
  const float* master;
  uint16_t* prev;
  uint32_t* idx;
  uint16_t* val;
};

struct ParkedMeta {
  uint32_t tile;
  uint32_t tensor;
  uint32_t agg;     // changed elements in the tile
  uint32_t last;    // 1: last tile of its tensor; 2: no more tiles for this look-back warp
  uint64_t first;   // first global tile of the tensor
  uint64_t n;       // elements of the tensor
  uint32_t ring_start;  // ring slot of the tile's first entry
  uint32_t ring_end;    // entries parked by the CTA up to the tile's last
  uint32_t base;    // first element of the tile within its tensor
  uint32_t* idx;
  uint16_t* val;
};

struct __align__(16) EncodeShared {
  uint64_t full[kEncStages];       // producer -> compute: stage filled
  uint64_t empty[kEncStages];      // compute -> producer: stage consumed
  uint64_t agg_ready[kPendSlots];  // compute -> look-back: tile parked and counted
  uint64_t slot_free[kPendSlots];  // look-back -> compute: tile copied out
  StageMeta meta[kEncStages];
  ParkedMeta parked[kPendSlots];
  uint32_t warp_tot[2][kWarps];  // per warp: changed elements per round, one byte each
  uint32_t ring_tail;            // ring entries before this position are copied out
};
static_assert(kEncLookbackWarps == 1, "parked tiles are freed in order by one look-back warp");

template <bool MULTI>
__device__ __forceinline__ const TensorDesc& desc_of(const EncodeLaunch& a, uint32_t t) {
  if constexpr (MULTI) return a.tensors[t];
  else return a.one;
}

// ------------------------------------------------------------ producer warp
// One thread. The next tile ticket is requested one fill ahead, so the
// atomic's round trip overlaps the wait for a free stage; consecutive tickets
// usually fall in the same tensor, so its descriptor is kept in registers and
// the tile -> tensor search runs only when a ticket leaves it.
template <bool MULTI>
__device__ __forceinline__ void producer_loop(const EncodeLaunch& a, EncodeShared& sh,
                                              uint8_t* stages) {
  const uint64_t pol_stream = l2_policy_evict_first();
  uint32_t ticket_fills_done = 0;  // stage fills issued (the END marker included)
  uint32_t ticket = atomicAdd(a.counters + 0, 1u) + a.first_ticket;
  uint32_t cur_t = 0;                      // cached tensor (multi-tensor mode)
  uint64_t cur_begin = 1, cur_end = 0;     // its global tile range; empty until loaded
  TensorDesc d = a.one;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kEncStages);
    const bool end = ticket >= a.total_tiles;
    const uint32_t next = end ? ticket : atomicAdd(a.counters + 0, 1u) + a.first_ticket;
    if (it >= uint32_t(kEncStages) && !helper_wait(&sh.empty[s], ((it / kEncStages) - 1) & 1u, a))
      break;
    ticket_fills_done = it + 1;
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
      }
    }
    const uint64_t base = (uint64_t(ticket) - d.tile_begin) * kEncTile;
    const uint64_t len = d.n - base < uint64_t(kEncTile) ? d.n - base : uint64_t(kEncTile);
    m.tensor = cur_t;
    m.len = uint32_t(len);
    m.base = base;
    m.first = d.tile_begin;
    m.n = d.n;
    m.master = d.master;
    m.prev = d.prev;
    m.idx = d.idx;
    m.val = d.val;
    if (d.bulk_ok && len == uint64_t(kEncTile)) {
      m.mode = kModeBulk;
      sh.meta[s] = m;
      uint8_t* st = stages + size_t(s) * kStageBytes;
      mbar_arrive_expect_tx(&sh.full[s], kStageBytes);
      bulk_g2s(st, d.master + base, kStageMasterBytes, &sh.full[s], pol_stream);
      // prev is written back soon after, so it keeps the default L2 policy
      bulk_g2s_plain(st + kStageMasterBytes, d.prev + base, kStagePrevBytes, &sh.full[s]);
    } else {
      m.mode = kModeGeneric;  // tail or unaligned tile: compute threads load from global
      sh.meta[s] = m;
      mbar_arrive(&sh.full[s]);
    }
    ticket = next;
  }
  // No bulk copy may still be in flight when the CTA exits: wait (bounded)
  // for the last fill of every stage.
  const uint32_t fills = ticket_fills_done;
  for (uint32_t f = fills > uint32_t(kEncStages) ? fills - kEncStages : 0u; f < fills; ++f)
    mbar_wait_bounded(&sh.full[f % kEncStages], (f / kEncStages) & 1u, a.wait_limit_ns);
  // The last CTA to stop taking tickets rewinds the ticket and finish
  // counters for the next launch on this workspace.
  __threadfence();
  const uint32_t finished = atomicAdd(a.counters + 1, 1u);
  if (finished == gridDim.x - 1) {
    atomicExch(a.counters + 0, 0u);
    atomicExch(a.counters + 1, 0u);
  }
}

// ---------------------------------------------------------- look-back warps
// Look-back warp w handles parked tiles w, w + W, w + 2W, ... of its CTA
// (W = kEncLookbackWarps), each in its own slot. It takes every such tile
// that is already counted, up to kLookbackBatch, issues all their look-back
// windows at once (one L2 round trip for the batch), then for each tile:
// resolves its global offset, publishes its inclusive prefix, copies its
// parked entries to the patch (entry k to position offset + k: contiguous,
// coalesced stores) and frees the slot.
// Copy a parked tile's entries to the patch: entry k goes to position
// prefix + k. A head of up to 3 entries brings the position to a multiple of
// 4; then each lane moves 4 consecutive entries with one 16-byte index store
// and one 8-byte value store; the tail goes one entry at a time. Positions at
// or past n are never written (they only arise after a wait gave up).
__device__ __forceinline__ void copy_out(const ParkedMeta& pm, uint32_t prefix,
                                         const uint32_t* ring, int lane) {
  const uint32_t agg = pm.agg;
  const bool vec = (reinterpret_cast<uintptr_t>(pm.idx) % 16u == 0) &&
                   (reinterpret_cast<uintptr_t>(pm.val) % 8u == 0) &&
                   uint64_t(prefix) + agg <= pm.n;
  uint32_t head = vec ? ((4u - (prefix & 3u)) & 3u) : agg;
  if (head > agg) head = agg;
  const uint32_t body = vec ? ((agg - head) & ~3u) : 0u;
  for (uint32_t k = uint32_t(lane); k < head; k += 32) {
    const uint32_t ent = ring[ring_slot(pm.ring_start + k)];
    const uint64_t pos = uint64_t(prefix) + k;
    if (pos < pm.n) {
      pm.idx[pos] = pm.base + (ent & 0xFFFFu);
      pm.val[pos] = uint16_t(ent >> 16);
    }
  }
  for (uint32_t k = head + uint32_t(lane) * 4u; k < head + body; k += 128u) {
    uint32_t e[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) e[q] = ring[ring_slot(pm.ring_start + k + uint32_t(q))];
    const uint64_t pos = uint64_t(prefix) + k;  // a multiple of 4
    *reinterpret_cast<uint4*>(pm.idx + pos) =
        make_uint4(pm.base + (e[0] & 0xFFFFu), pm.base + (e[1] & 0xFFFFu),
                   pm.base + (e[2] & 0xFFFFu), pm.base + (e[3] & 0xFFFFu));
    *reinterpret_cast<uint2*>(pm.val + pos) =
        make_uint2((e[0] >> 16) | (e[1] & 0xFFFF0000u), (e[2] >> 16) | (e[3] & 0xFFFF0000u));
  }
  for (uint32_t k = head + body + uint32_t(lane); k < agg; k += 32) {
    const uint32_t ent = ring[ring_slot(pm.ring_start + k)];
    const uint64_t pos = uint64_t(prefix) + k;
    if (pos < pm.n) {
      pm.idx[pos] = pm.base + (ent & 0xFFFFu);
      pm.val[pos] = uint16_t(ent >> 16);
    }
  }
}

__device__ __forceinline__ void lookback_loop(const EncodeLaunch& a, EncodeShared& sh,
                                              const uint32_t* ring, int w, int lane, bool multi) {
  for (uint32_t i = uint32_t(w);;) {
    const bool ok = helper_wait(&sh.agg_ready[i % kPendSlots], (i / kPendSlots) & 1u, a);
    // the warp leaves together: everything below uses full-warp collectives
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    // how many more of this warp's tiles are already parked (lane 0 decides)
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
    uint64_t win[kLookbackBatch][kWindow];
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
        load_window<StatusEpoch, EncodeLaunch, kWindow>(a, int64_t(pm.tile) - 1, pm.first, lane, win[b]);
      nb = b + 1;
    }
#pragma unroll
    for (int b = 0; b < kLookbackBatch; ++b) {
      if (b >= nb) continue;
      const uint32_t ii = i + uint32_t(b * kEncLookbackWarps);
      const int q = int(ii % kPendSlots);
      const ParkedMeta pm = sh.parked[q];
      const uint32_t prefix = resolve_prefix<StatusEpoch, EncodeLaunch, 32, kWindow>(
          a, pm.tile, pm.first, pm.agg, lane, win[b]);
      if (lane == 0 && pm.last == 1u) a.counts_out[multi ? pm.tensor : 0] = uint64_t(prefix) + pm.agg;
      copy_out(pm, prefix, ring, lane);
      __syncwarp();
      if (lane == 0) {
        // tiles are copied out in order: everything before this tile's end is free
        __threadfence_block();
        *reinterpret_cast<volatile uint32_t*>(&sh.ring_tail) = pm.ring_end;
        mbar_arrive(&sh.slot_free[q]);
      }
    }
    if (end) break;
    i += uint32_t(nb * kEncLookbackWarps);
  }
}

// ------------------------------------------------------------ compute warps
// Four consecutive elements from element li of a tail or unaligned tile, read
// from global memory: elements past the end read as +0 with a +0 view, which
// never counts as a change. Out of line: the bulk path is the hot one, and
// this one, inlined at every round of both passes, only added to its code.
struct RoundIn {
  float4 mv;
  uint2 pv;
};

__device__ __noinline__ RoundIn load_round_generic(const float* master, const uint16_t* prev,
                                                   uint64_t base, uint32_t len, uint32_t li) {
  float mm[4];
  uint32_t pp[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const bool valid = li + e < len;
    mm[e] = valid ? master[base + li + e] : 0.0f;
    pp[e] = valid ? uint32_t(prev[base + li + e]) : 0u;
  }
  RoundIn r;
  r.mv = make_float4(mm[0], mm[1], mm[2], mm[3]);
  r.pv = make_uint2(pp[0] | (pp[1] << 16), pp[2] | (pp[3] << 16));
  return r;
}

template <bool MULTI>
__device__ __forceinline__ void compute_loop(const EncodeLaunch& a, EncodeShared& sh,
                                             uint8_t* stages, uint32_t* ring, int tid, int lane,
                                             int warp) {
  // uniform across the compute threads
  uint32_t posted = 0, ring_head = 0;  // ring_head: entries parked so far
  uint32_t ring_pos = 0;               // its ring slot
  bool failed = false;  // this thread saw a wait give up
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kEncStages);
    failed |= !wait_or_flag(&sh.full[s], (it / kEncStages) & 1u, a);
    const StageMeta m = sh.meta[s];
    const bool live = m.mode != kModeEnd;
    const uint64_t base = m.base;
    const uint32_t len = m.len;

    // ---- cast + compare: 4 consecutive elements per thread per round
    uint32_t nb[kEncRounds][2];  // new BF16 values, two per word (low half = lower index)
    uint32_t flags = 0;          // bit (j*4 + e): element e of round j changed
    uint32_t nan_seen = 0;
    const float4* sm = reinterpret_cast<const float4*>(stages + size_t(s) * kStageBytes);
    const uint2* sp = reinterpret_cast<const uint2*>(stages + size_t(s) * kStageBytes + kStageMasterBytes);
    // tail or unaligned tile: elements past the end read as +0 with a +0 view,
    // which never counts as a change (len is 0 for the end marker)
    auto load_round = [&](int j, float4& mv, uint2& pv) {
      if (m.mode == kModeBulk) {
        mv = sm[j * kEncThreads + tid];
        pv = sp[j * kEncThreads + tid];
      } else {
        const RoundIn r = load_round_generic(m.master, m.prev, base, len,
                                             uint32_t(j * kEncThreads + tid) * 4u);
        mv = r.mv;
        pv = r.pv;
      }
    };
    auto compare_round = [&](int j, const uint2& pv) {
      const uint32_t d01 = nb[j][0] ^ pv.x, d23 = nb[j][1] ^ pv.y;  // bitwise, two at a time
      return uint32_t((d01 << 16) != 0u) | (uint32_t(d01 > 0xFFFFu) << 1) |
             (uint32_t((d23 << 16) != 0u) << 2) | (uint32_t(d23 > 0xFFFFu) << 3);
    };
#pragma unroll
    for (int j = 0; j < kEncRounds; ++j) {
      float4 mv;
      uint2 pv;
      load_round(j, mv, pv);
      nb[j][0] = cvt_bf16x2_rn(mv.x, mv.y);
      nb[j][1] = cvt_bf16x2_rn(mv.z, mv.w);
      nan_seen |= any_nan4(mv.x, mv.y, mv.z, mv.w);
      flags |= compare_round(j, pv) << (4 * j);
    }
    if (nan_seen) {
      // rare: redo this thread's rounds with NaN mapped to the canonical 0x7FC0
      flags = 0;
#pragma unroll
      for (int j = 0; j < kEncRounds; ++j) {
        float4 mv;
        uint2 pv;
        load_round(j, mv, pv);
        nb[j][0] = canon_nan_pair(cvt_bf16x2_rn(mv.x, mv.y), mv.x, mv.y);
        nb[j][1] = canon_nan_pair(cvt_bf16x2_rn(mv.z, mv.w), mv.z, mv.w);
        flags |= compare_round(j, pv) << (4 * j);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);  // this warp is done with stage s

    // ---- refresh prev now: it does not depend on the tile's global offset
#pragma unroll
    for (int j = 0; j < kEncRounds; ++j) {
      const uint32_t f = (flags >> (j * 4)) & 0xFu;
      if (f == 0u) continue;
      const uint32_t li = uint32_t(j * kEncThreads + tid) * 4u;
      if (m.mode == kModeBulk) {
        *reinterpret_cast<uint2*>(m.prev + base + li) = make_uint2(nb[j][0], nb[j][1]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((f >> e) & 1u) m.prev[base + li + e] = uint16_t((nb[j][e >> 1] >> ((e & 1) * 16)) & 0xFFFFu);
      }
    }

    // ---- rank the changed elements. Within a warp: one scan of the four
    // per-round counts packed into bytes (a byte never exceeds 32 x 4 = 128).
    uint32_t cnts = 0;
#pragma unroll
    for (int j = 0; j < kEncRounds; ++j) cnts |= uint32_t(__popc((flags >> (4 * j)) & 0xFu)) << (8 * j);
    uint32_t incl = cnts;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const uint32_t excl = incl - cnts;
    const int pc = int(it & 1u);
    if (lane == 31) sh.warp_tot[pc][warp] = incl;
    // the one CTA barrier of the iteration; it also decides, for every compute
    // warp at once, whether the loop ends
    if (compute_barrier_or(failed || !live)) break;
    // Across warps, in tile order (round-major, then warp): every warp scans
    // the 8 packed warp totals, widened to 16-bit fields (rounds 0/2 and 1/3;
    // a field never exceeds 8 x 128 = 1024).
    const uint32_t t = lane < kWarps ? sh.warp_tot[pc][lane] : 0u;
    const uint32_t t02 = t & 0x00FF00FFu, t13 = (t >> 8) & 0x00FF00FFu;
    uint32_t s02 = t02, s13 = t13;
#pragma unroll
    for (int o = 1; o < kWarps; o <<= 1) {
      const uint32_t v02 = __shfl_up_sync(0xFFFFFFFFu, s02, o);
      const uint32_t v13 = __shfl_up_sync(0xFFFFFFFFu, s13, o);
      if (lane >= o) { s02 += v02; s13 += v13; }
    }
    const uint32_t b02 = __shfl_sync(0xFFFFFFFFu, s02 - t02, warp);  // warps before this one
    const uint32_t b13 = __shfl_sync(0xFFFFFFFFu, s13 - t13, warp);
    const uint32_t a02 = __shfl_sync(0xFFFFFFFFu, s02, kWarps - 1);   // all warps
    const uint32_t a13 = __shfl_sync(0xFFFFFFFFu, s13, kWarps - 1);
    const uint32_t tot0 = a02 & 0xFFFFu, tot1 = a13 & 0xFFFFu, tot2 = a02 >> 16, tot3 = a13 >> 16;
    uint32_t round_off[kEncRounds];  // this thread's first entry in each round, within the tile
    round_off[0] = (b02 & 0xFFFFu) + (excl & 0xFFu);
    round_off[1] = tot0 + (b13 & 0xFFFFu) + ((excl >> 8) & 0xFFu);
    round_off[2] = tot0 + tot1 + (b02 >> 16) + ((excl >> 16) & 0xFFu);
    round_off[3] = tot0 + tot1 + tot2 + (b13 >> 16) + (excl >> 24);
    const uint32_t agg = tot0 + tot1 + tot2 + tot3;
    if (tid == 0) {
      // publish the count at once; a tensor's first tile is its own prefix
      st_relaxed_u64(a.status + m.tile,
                     make_status(uint64_t(m.tile) == m.first ? kFlagPrefix : kFlagAggregate,
                                 a.epoch, agg));
    }

    // ---- room for the tile: its parked slot must have been copied out (the
    // look-back warp frees slots in order) and the ring must hold agg more
    // entries. Each thread checks for itself; no CTA barrier is needed.
    const int q = int(posted % kPendSlots);
    if (posted >= uint32_t(kPendSlots))
      failed |= !wait_or_flag(&sh.slot_free[q], ((posted - kPendSlots) / kPendSlots) & 1u, a);
    failed |= !wait_ring_room<64>(&sh.ring_tail, ring_head, agg, uint32_t(kEncRing), a);

    // ---- park the compacted tile: (local index | value << 16) per entry,
    // visiting only the set flag bits
#pragma unroll
    for (int j = 0; j < kEncRounds; ++j) {
      uint32_t f = (flags >> (j * 4)) & 0xFu;
      if (f == 0u) continue;
      const uint32_t li = uint32_t(j * kEncThreads + tid) * 4u;
      uint32_t r = ring_pos + round_off[j];
      do {
        const uint32_t e = uint32_t(__ffs(f)) - 1u;
        f &= f - 1u;
        const uint32_t word = (e & 2u) ? nb[j][1] : nb[j][0];
        const uint32_t value = (e & 1u) ? (word >> 16) : (word & 0xFFFFu);
        ring[ring_slot(r)] = (li + e) | (value << 16);
        ++r;
      } while (f != 0u);
    }
    if (tid == 0) {
      ParkedMeta pm;
      pm.tile = m.tile;
      pm.tensor = m.tensor;
      pm.agg = agg;
      pm.last = (base + len == m.n) ? 1u : 0u;
      pm.first = m.first;
      pm.n = m.n;
      pm.ring_start = ring_pos;
      pm.ring_end = ring_head + agg;
      pm.base = uint32_t(base);
      pm.idx = m.idx;
      pm.val = m.val;
      sh.parked[q] = pm;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.agg_ready[q]);  // 8 arrivals: every warp's entries are in
    ++posted;
    ring_head += agg;
    ring_pos = ring_slot(ring_pos + agg);
  }
  // no more tiles (the compute warps left the loop together): wait until
  // every parked tile is copied out, then send each look-back warp its end
  // marker
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

template <bool MULTI>
__global__ void __launch_bounds__(kEncBlockThreads, kEncMinBlocks)
    encode_kernel(const __grid_constant__ EncodeLaunch a) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ EncodeShared sh;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 127) & ~uintptr_t(127));
  uint32_t* ring = reinterpret_cast<uint32_t*>(stages + size_t(kEncStages) * kStageBytes);

  if constexpr (MULTI) {
    // tensors with no elements have no tiles: their count is 0
    if (blockIdx.x == 0) {
      for (int t = tid; t < a.ntensors; t += kEncBlockThreads)
        if (a.tensors[t].n == 0) a.counts_out[t] = 0;
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
  __syncthreads();  // the last CTA-wide barrier: roles split below

  if (warp < kWarps) {
    compute_loop<MULTI>(a, sh, stages, ring, tid, lane, warp);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_loop<MULTI>(a, sh, stages);
  } else {
    lookback_loop(a, sh, ring, warp - kFirstLookbackWarp, lane, MULTI);
  }
}

template <bool MULTI>
int encode_blocks_per_sm() {
  static int cached = [] {
    cudaFuncSetAttribute(encode_kernel<MULTI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         int(kDynSmem));
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, encode_kernel<MULTI>, kEncBlockThreads,
                                                      kDynSmem) != cudaSuccess || b < 1)
      b = 1;
    return b;
  }();
  return cached;
}

}  // namespace

int encode_grid_size(int device) {
  const int per_sm = encode_blocks_per_sm<true>() < encode_blocks_per_sm<false>()
                         ? encode_blocks_per_sm<true>()
                         : encode_blocks_per_sm<false>();
  return sm_count(device) * per_sm;
}

cudaError_t launch_encode(const EncodeLaunch& a, bool multi, int grid, cudaStream_t stream) {
  if (multi) {
    encode_blocks_per_sm<true>();
    encode_kernel<true><<<grid, kEncBlockThreads, kDynSmem, stream>>>(a);
  } else {
    encode_blocks_per_sm<false>();
    encode_kernel<false><<<grid, kEncBlockThreads, kDynSmem, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace pulse
