// compose.cu -- patch-chain composition for a sidecar that catches up over
// several missing versions ("Taking Reinforcement Learning Cross Datacenter",
// talk 16:40-17:04: if the engine is behind but can catch up, the sidecar
// applies the missing transitions). Patches carry absolute values (PULSE
// summary, "1. PULSESync"), so patch A followed by patch B equals one patch:
// the union of their indices, each with the value of the later patch that
// lists it. compose(A, B) builds it in ascending order.
//
// Merge-path design (Green, McColl, Bader, "GPU Merge Path", 2012) with an
// order-preserving compaction:
//  * partition kernel: one thread per output tile finds, by binary search on
//    the merge path, how many entries of A precede the tile's first merged
//    position (stable merge, A before B on an equal index), and the tile's
//    segment;
//  * compose kernel: persistent, warp-specialized CTAs with the encode
//    kernels' layout. The producer warp takes tile tickets and stages the
//    tile's four ranges (A and B indices and values) in a 2-stage
//    shared-memory ring: the 16-byte-aligned body of each range by bulk copy
//    (cp.async.bulk, counted in mbarrier transaction bytes), the ragged ends
//    with plain loads. The 8 compute warps merge kCmpPerThread positions per
//    thread (a merge-path search in shared memory), keep a position unless
//    the next merged position has the same index (of the pair A-entry,
//    B-entry of a shared index only B's is kept), rank the kept entries, and
//    park them in a shared-memory ring. The look-back warp resolves each
//    parked tile's output offset with a decoupled look-back and copies its
//    entries out with contiguous vector stores.
#include "encode_common.cuh"

namespace pulse {
namespace {

// Parked tiles per CTA and tiles resolved per look-back round trip (the
// values this kernel was tuned with).
constexpr int kCmpSlots = 8;
constexpr int kCmpBatch = 4;
constexpr int kCmpWindow = 2;  // look-back words per lane and round trip

#ifndef PULSE_CMP_PER_THREAD
#define PULSE_CMP_PER_THREAD 8
#endif
constexpr int kCmpThreads = kEncThreads;                // compute threads
constexpr int kCmpPerThread = PULSE_CMP_PER_THREAD;
constexpr int kCmpTile = kCmpThreads * kCmpPerThread;  // merged positions per tile
constexpr int kCmpWarps = kCmpThreads / 32;
static_assert(kCmpWarps == enc::kWarps, "the compute warps of the shared CTA layout");
constexpr int kSlack = 32;  // entries of room for 16-byte-aligned range ends (and one more index)
#ifndef PULSE_CMP_STAGES
#define PULSE_CMP_STAGES 2
#endif
// Stage ring depth (measured: 2 stages at 3 CTAs per SM beat 3 stages at 2).
constexpr int kCmpStages = PULSE_CMP_STAGES;
constexpr uint32_t kCmpRing = 4096;              // parked entries per CTA
constexpr uint32_t kCmpRingMask = kCmpRing - 1;
static_assert(kCmpRing >= uint32_t(kCmpTile), "the ring holds a whole tile");
static_assert(kEncLookbackWarps == 1, "parked tiles are copied out in order by one look-back warp");

struct CmpLaunch {
  const CmpSegment* segs;  // multi-segment mode: device array
  CmpSegment one;          // single-segment mode
  const uint64_t* tile_begin;
  int nsegs;
  uint64_t total_tiles;
  const uint32_t* splits;  // per tile: A entries before the tile's first merged position
  const uint32_t* tile_seg;  // per tile: its segment (multi-segment mode)
  uint64_t* status;
  uint32_t* counters;
  uint64_t* counts_out;
  uint32_t epoch;
  uint64_t wait_limit_ns;
};

template <bool MULTI>
__device__ __forceinline__ const CmpSegment& seg_of(const CmpLaunch& a, int t) {
  if constexpr (MULTI) return a.segs[t];
  else return a.one;
}

// Number of A entries among the first d merged entries (A before B on ties).
__device__ __forceinline__ uint64_t merge_split_global(const uint32_t* A, uint64_t ka,
                                                       const uint32_t* B, uint64_t kb,
                                                       uint64_t d) {
  uint64_t lo = d > kb ? d - kb : 0, hi = d < ka ? d : ka;
  while (lo < hi) {
    const uint64_t mid = (lo + hi) >> 1;
    if (A[mid] <= B[d - 1 - mid]) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ uint32_t merge_split_shared(const uint32_t* A, uint32_t na,
                                                       const uint32_t* B, uint32_t nb,
                                                       uint32_t d) {
  uint32_t lo = d > nb ? d - nb : 0, hi = d < na ? d : na;
  while (lo < hi) {
    const uint32_t mid = (lo + hi) >> 1;
    if (A[mid] <= B[d - 1 - mid]) lo = mid + 1; else hi = mid;
  }
  return lo;
}

template <bool MULTI>
__global__ void __launch_bounds__(256)
    compose_partition_kernel(const CmpLaunch a, uint32_t* splits, uint32_t* tile_seg) {
  const uint64_t g = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= a.total_tiles) return;
  int t = 0;
  if constexpr (MULTI) {
    t = enc::find_tensor(a.tile_begin, a.nsegs, g);
    tile_seg[g] = uint32_t(t);
  }
  const CmpSegment& s = seg_of<MULTI>(a, t);
  const uint64_t d = (g - s.tile_begin) * kCmpTile;
  splits[g] = uint32_t(merge_split_global(s.idx_a, s.count_a, s.idx_b, s.count_b, d));
}


// ------------------------------------------------------------ shared state
template <class V>
struct CmpGeom {
  static constexpr uint32_t kIdxBytes = (kCmpTile + kSlack) * 4;
  static constexpr uint32_t kValBytes = ((kCmpTile + kSlack) * sizeof(V) + 15) / 16 * 16;
  static constexpr uint32_t kStageBytes = 2 * kIdxBytes + 2 * kValBytes;
  // stage regions: A idx, B idx, A val, B val
  static constexpr uint32_t kOffIdxA = 0;
  static constexpr uint32_t kOffIdxB = kIdxBytes;
  static constexpr uint32_t kOffValA = 2 * kIdxBytes;
  static constexpr uint32_t kOffValB = 2 * kIdxBytes + kValBytes;
  static constexpr size_t kDynSmem = size_t(kCmpStages) * kStageBytes +
                                     size_t(kCmpRing) * (4 + sizeof(V)) + 128;
};

struct CmpStageMeta {
  uint32_t tile;
  uint32_t seg;
  uint32_t mode;
  uint32_t na, nb;
  uint32_t head[4];      // entries before the range start in each region (A/B idx, A/B val)
  uint32_t ext_a;        // 1: A's entry right after the tile is staged at sA[na]
  uint32_t ext_b;        // 1: B's entry right after the tile is staged at sB[nb]
  uint32_t last;         // last tile of its segment
  uint64_t first;        // first global tile of the segment
  uint64_t i0, j0;       // first A and B entries of the tile
  uint64_t total;        // merged positions of the segment
  const uint32_t* idx_a;
  const void* val_a;
  const uint32_t* idx_b;
  const void* val_b;
  uint32_t* idx_out;
  void* val_out;
};

struct CmpParked {
  uint32_t tile;
  uint32_t seg;
  uint32_t agg;
  uint32_t last;  // 1: last tile of its segment; 2: no more tiles
  uint32_t ring_start;
  uint64_t first;
  uint64_t total;
  uint32_t* idx_out;
  void* val_out;
};

struct __align__(16) CmpShared {
  uint64_t full[kCmpStages];
  uint64_t empty[kCmpStages];
  uint64_t agg_ready[kCmpSlots];
  uint64_t slot_free[kCmpSlots];
  CmpStageMeta meta[kCmpStages];
  CmpParked parked[kCmpSlots];
  uint32_t warp_tot[2][kCmpWarps];
  uint32_t ring_tail;
};

// Plain loads of `count` elements [first, first + count) of a range into its
// stage region (only where a range ends inside the array's last, partial
// 16-byte chunk; at most 15 bytes).
template <class E>
__device__ __forceinline__ void load_ragged(uint8_t* region, uint64_t aligned_first_elem,
                                            const E* src, uint64_t first, uint64_t count) {
  E* dst = reinterpret_cast<E*>(region);
  for (uint64_t k = 0; k < count; ++k) dst[first + k - aligned_first_elem] = src[first + k];
}

// Stage range [e0, e1) of an array of c elements of type E into `region`.
// The bulk copy runs from the 16-byte boundary at or below e0 to the one at
// or above e1 when that stays inside the array, else to the one below e1
// (then *ragged_from = that boundary and the rest needs plain loads).
// Returns the bulk bytes; *head = entries between the start boundary and e0.
template <class E>
__device__ __forceinline__ uint32_t stage_range(uint8_t* region, const E* src, uint64_t e0,
                                                uint64_t e1, uint64_t c, uint32_t* head,
                                                uint64_t* ragged_from, uint64_t* bar,
                                                uint64_t pol, bool issue) {
  constexpr uint64_t kPer = 16 / sizeof(E);  // elements per 16 bytes
  const uint64_t a0 = e0 / kPer * kPer;
  uint64_t a1 = (e1 + kPer - 1) / kPer * kPer;
  if (a1 > c) a1 = e1 / kPer * kPer;
  *head = uint32_t(e0 - a0);
  *ragged_from = a1 > e0 ? a1 : e0;
  uint32_t bytes = 0;
  if (a1 > a0) {
    bytes = uint32_t((a1 - a0) * sizeof(E));
    if (issue) bulk_g2s(region, src + a0, bytes, bar, pol);
  }
  return bytes;
}

// ------------------------------------------------------------ producer warp
template <class V, bool MULTI>
__device__ __forceinline__ void cmp_producer(const CmpLaunch& a, CmpShared& sh, uint8_t* stages) {
  using G = CmpGeom<V>;
  const uint64_t pol = l2_policy_evict_first();
  uint32_t fills_done = 0;
  // Tickets run two ahead of the tile being staged and their split words and
  // segment one ahead, so neither the ticket atomic nor those loads wait in
  // line with the bulk copies.
  auto fetch = [&](uint32_t tk, uint32_t& s0, uint32_t& s1, uint32_t& sg) {
    s0 = s1 = sg = 0;
    if (tk < a.total_tiles) {
      s0 = a.splits[tk];
      if (uint64_t(tk) + 1 < a.total_tiles) s1 = a.splits[tk + 1];
      if (MULTI) sg = a.tile_seg[tk];
    }
  };
  uint32_t ticket = atomicAdd(a.counters + 0, 1u);
  uint32_t cs0, cs1, cseg;
  fetch(ticket, cs0, cs1, cseg);
  uint32_t ticket1 = ticket < a.total_tiles ? atomicAdd(a.counters + 0, 1u) : ticket;
  uint32_t ticket2 = ticket1 < a.total_tiles ? atomicAdd(a.counters + 0, 1u) : ticket1;
  uint32_t ns0, ns1, nseg;
  fetch(ticket1, ns0, ns1, nseg);
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kCmpStages);
    const bool end = ticket >= a.total_tiles;
    if (it >= uint32_t(kCmpStages) &&
        !enc::helper_wait(&sh.empty[s], ((it / kCmpStages) - 1) & 1u, a))
      break;
    fills_done = it + 1;
    CmpStageMeta m{};
    m.tile = ticket;
    if (end) {
      m.mode = enc::kModeEnd;
      sh.meta[s] = m;
      mbar_arrive(&sh.full[s]);
      mbar_arrive(&sh.full[s]);
      break;
    }
    const uint64_t g = ticket;
    const int t = MULTI ? int(cseg) : 0;
    const CmpSegment& sg = seg_of<MULTI>(a, t);
    const uint64_t total = sg.count_a + sg.count_b;
    const uint64_t d0 = (g - sg.tile_begin) * kCmpTile;
    const uint64_t d1 = d0 + kCmpTile < total ? d0 + kCmpTile : total;
    const bool last = d1 == total;
    const uint64_t i0 = cs0;
    const uint64_t i1 = last ? sg.count_a : cs1;
    const uint64_t j0 = d0 - i0, j1 = d1 - i1;
    // stage one index past each range when it exists: the merged position
    // after the tile is the smaller of the two
    const uint64_t xa = i1 < sg.count_a ? 1 : 0, xb = j1 < sg.count_b ? 1 : 0;
    m.ext_a = uint32_t(xa);
    m.ext_b = uint32_t(xb);
    m.seg = uint32_t(t);
    m.na = uint32_t(i1 - i0);
    m.nb = uint32_t(j1 - j0);
    m.last = last ? 1u : 0u;
    m.first = sg.tile_begin;
    m.i0 = i0;
    m.j0 = j0;
    m.total = total;
    m.idx_a = sg.idx_a;
    m.val_a = sg.val_a;
    m.idx_b = sg.idx_b;
    m.val_b = sg.val_b;
    m.idx_out = sg.idx_out;
    m.val_out = sg.val_out;
    const V* va = static_cast<const V*>(sg.val_a);
    const V* vb = static_cast<const V*>(sg.val_b);
    const bool bulk = (reinterpret_cast<uintptr_t>(sg.idx_a) % 16u == 0) &&
                      (reinterpret_cast<uintptr_t>(sg.idx_b) % 16u == 0) &&
                      (reinterpret_cast<uintptr_t>(va) % 16u == 0) &&
                      (reinterpret_cast<uintptr_t>(vb) % 16u == 0);
    uint8_t* st = stages + size_t(s) * G::kStageBytes;
    if (bulk) {
      m.mode = enc::kModeBulk;
      uint64_t rf[4];
      uint32_t bytes = 0;
      bytes += stage_range(st + G::kOffIdxA, sg.idx_a, i0, i1 + xa, sg.count_a, &m.head[0], &rf[0],
                           nullptr, pol, false);
      bytes += stage_range(st + G::kOffIdxB, sg.idx_b, j0, j1 + xb, sg.count_b, &m.head[1], &rf[1],
                           nullptr, pol, false);
      bytes += stage_range(st + G::kOffValA, va, i0, i1, sg.count_a, &m.head[2], &rf[2], nullptr,
                           pol, false);
      bytes += stage_range(st + G::kOffValB, vb, j0, j1, sg.count_b, &m.head[3], &rf[3], nullptr,
                           pol, false);
      sh.meta[s] = m;
      mbar_arrive_expect_tx(&sh.full[s], bytes);  // first of the two arrivals
      uint32_t h;
      uint64_t r;
      stage_range(st + G::kOffIdxA, sg.idx_a, i0, i1 + xa, sg.count_a, &h, &r, &sh.full[s], pol, true);
      stage_range(st + G::kOffIdxB, sg.idx_b, j0, j1 + xb, sg.count_b, &h, &r, &sh.full[s], pol, true);
      stage_range(st + G::kOffValA, va, i0, i1, sg.count_a, &h, &r, &sh.full[s], pol, true);
      stage_range(st + G::kOffValB, vb, j0, j1, sg.count_b, &h, &r, &sh.full[s], pol, true);
      // ranges that end inside their array's last partial 16-byte chunk
      constexpr uint64_t kPi = 4, kPv = 16 / sizeof(V);
      if (rf[0] < i1 + xa) load_ragged(st + G::kOffIdxA, i0 / kPi * kPi, sg.idx_a, rf[0], i1 + xa - rf[0]);
      if (rf[1] < j1 + xb) load_ragged(st + G::kOffIdxB, j0 / kPi * kPi, sg.idx_b, rf[1], j1 + xb - rf[1]);
      if (rf[2] < i1) load_ragged(st + G::kOffValA, i0 / kPv * kPv, va, rf[2], i1 - rf[2]);
      if (rf[3] < j1) load_ragged(st + G::kOffValB, j0 / kPv * kPv, vb, rf[3], j1 - rf[3]);
      mbar_arrive(&sh.full[s]);  // second arrival: plain stores done
    } else {
      m.mode = enc::kModeGeneric;  // compute warps stage the ranges themselves
      sh.meta[s] = m;
      mbar_arrive(&sh.full[s]);
      mbar_arrive(&sh.full[s]);
    }
    // advance the ticket pipeline
    ticket = ticket1;
    cs0 = ns0;
    cs1 = ns1;
    cseg = nseg;
    ticket1 = ticket2;
    fetch(ticket1, ns0, ns1, nseg);
    ticket2 = ticket2 < a.total_tiles ? atomicAdd(a.counters + 0, 1u) : ticket2;
  }
  for (uint32_t f = fills_done > uint32_t(kCmpStages) ? fills_done - kCmpStages : 0u; f < fills_done; ++f)
    mbar_wait_bounded(&sh.full[f % kCmpStages], (f / kCmpStages) & 1u, a.wait_limit_ns);
  __threadfence();
  const uint32_t finished = atomicAdd(a.counters + 1, 1u);
  if (finished == gridDim.x - 1) {
    atomicExch(a.counters + 0, 0u);
    atomicExch(a.counters + 1, 0u);
  }
}

// ---------------------------------------------------------- look-back warp
template <class V>
__device__ __forceinline__ void cmp_copy_out(const CmpParked& pm, uint32_t prefix,
                                             const uint32_t* ring_idx, const V* ring_val,
                                             int lane) {
  const uint32_t agg = pm.agg;
  V* val_out = static_cast<V*>(pm.val_out);
  const bool vec = (reinterpret_cast<uintptr_t>(pm.idx_out) % 16u == 0) &&
                   (reinterpret_cast<uintptr_t>(val_out) % (4 * sizeof(V)) == 0) &&
                   uint64_t(prefix) + agg <= pm.total;
  uint32_t head = vec ? ((4u - (prefix & 3u)) & 3u) : agg;
  if (head > agg) head = agg;
  const uint32_t body = vec ? ((agg - head) & ~3u) : 0u;
  auto one = [&](uint32_t k) {
    const uint64_t pos = uint64_t(prefix) + k;
    if (pos < pm.total) {
      const uint32_t r = (pm.ring_start + k) & kCmpRingMask;
      pm.idx_out[pos] = ring_idx[r];
      val_out[pos] = ring_val[r];
    }
  };
  for (uint32_t k = uint32_t(lane); k < head; k += 32) one(k);
  for (uint32_t k = head + uint32_t(lane) * 4u; k < head + body; k += 128u) {
    uint32_t e[4];
    uint32_t v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t r = (pm.ring_start + k + uint32_t(q)) & kCmpRingMask;
      e[q] = ring_idx[r];
      v[q] = ring_val[r];
    }
    const uint64_t pos = uint64_t(prefix) + k;
    *reinterpret_cast<uint4*>(pm.idx_out + pos) = make_uint4(e[0], e[1], e[2], e[3]);
    if constexpr (sizeof(V) == 2) {
      *reinterpret_cast<uint2*>(val_out + pos) = make_uint2(v[0] | (v[1] << 16), v[2] | (v[3] << 16));
    } else {
      *reinterpret_cast<uint32_t*>(val_out + pos) = v[0] | (v[1] << 8) | (v[2] << 16) | (v[3] << 24);
    }
  }
  for (uint32_t k = head + body + uint32_t(lane); k < agg; k += 32) one(k);
}

template <class V, bool MULTI>
__device__ __forceinline__ void cmp_lookback(const CmpLaunch& a, CmpShared& sh,
                                             const uint32_t* ring_idx, const V* ring_val,
                                             int lane) {
  using namespace enc;
  for (uint32_t i = 0;;) {
    const bool ok = helper_wait(&sh.agg_ready[i % kCmpSlots], (i / kCmpSlots) & 1u, a);
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    int more = 0;
    if (lane == 0) {
      for (int b = 1; b < kCmpBatch; ++b) {
        const uint32_t ii = i + uint32_t(b);
        if (!mbar_test_wait(&sh.agg_ready[ii % kCmpSlots], (ii / kCmpSlots) & 1u)) break;
        more = b;
      }
    }
    more = __shfl_sync(0xFFFFFFFFu, more, 0);
    int nb = 0;
    bool end = false;
    uint64_t win[kCmpBatch][kCmpWindow];
#pragma unroll
    for (int b = 0; b < kCmpBatch; ++b) {
      if (b > more || end) continue;
      const uint32_t ii = i + uint32_t(b);
      const int q = int(ii % kCmpSlots);
      if (b > 0) mbar_test_wait(&sh.agg_ready[q], (ii / kCmpSlots) & 1u);  // acquire for every lane
      const CmpParked& pm = sh.parked[q];
      if (pm.last == 2u) {
        end = true;
        continue;
      }
      if (pm.tile != pm.first)
        load_window<StatusEpoch, CmpLaunch, kCmpWindow>(a, int64_t(pm.tile) - 1, pm.first, lane, win[b]);
      nb = b + 1;
    }
#pragma unroll
    for (int b = 0; b < kCmpBatch; ++b) {
      if (b >= nb) continue;
      const uint32_t ii = i + uint32_t(b);
      const int q = int(ii % kCmpSlots);
      const CmpParked pm = sh.parked[q];
      const uint32_t prefix = resolve_prefix<StatusEpoch, CmpLaunch, 32, kCmpWindow>(
          a, pm.tile, pm.first, pm.agg, lane, win[b]);
      if (lane == 0 && pm.last == 1u) a.counts_out[MULTI ? pm.seg : 0] = uint64_t(prefix) + pm.agg;
      cmp_copy_out<V>(pm, prefix, ring_idx, ring_val, lane);
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        *reinterpret_cast<volatile uint32_t*>(&sh.ring_tail) = pm.ring_start + pm.agg;
        mbar_arrive(&sh.slot_free[q]);
      }
    }
    if (end) break;
    i += uint32_t(nb);
  }
}

// ------------------------------------------------------------ compute warps
template <class V>
__device__ __forceinline__ void cmp_compute(const CmpLaunch& a, CmpShared& sh, uint8_t* stages,
                                            uint32_t* ring_idx, V* ring_val, int tid, int lane,
                                            int warp) {
  using namespace enc;
  using G = CmpGeom<V>;
  uint32_t posted = 0, ring_head = 0;
  bool failed = false;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kCmpStages);
    failed |= !wait_or_flag(&sh.full[s], (it / kCmpStages) & 1u, a);
    const CmpStageMeta m = sh.meta[s];
    const bool live = m.mode != kModeEnd;
    uint8_t* st = stages + size_t(s) * G::kStageBytes;
    uint32_t ha = m.head[0], hb = m.head[1], hva = m.head[2], hvb = m.head[3];
    if (m.mode == kModeGeneric) {
      // unaligned patch arrays: the compute warps stage the ranges themselves
      uint32_t* ia = reinterpret_cast<uint32_t*>(st + G::kOffIdxA);
      uint32_t* ib = reinterpret_cast<uint32_t*>(st + G::kOffIdxB);
      V* va = reinterpret_cast<V*>(st + G::kOffValA);
      V* vb = reinterpret_cast<V*>(st + G::kOffValB);
      for (uint32_t k = tid; k < m.na + m.ext_a; k += kCmpThreads) {
        ia[k] = m.idx_a[m.i0 + k];
        if (k < m.na) va[k] = static_cast<const V*>(m.val_a)[m.i0 + k];
      }
      for (uint32_t k = tid; k < m.nb + m.ext_b; k += kCmpThreads) {
        ib[k] = m.idx_b[m.j0 + k];
        if (k < m.nb) vb[k] = static_cast<const V*>(m.val_b)[m.j0 + k];
      }
      ha = hb = hva = hvb = 0;
      compute_barrier();
    }
    const uint32_t* sA = reinterpret_cast<const uint32_t*>(st + G::kOffIdxA) + ha;
    const uint32_t* sB = reinterpret_cast<const uint32_t*>(st + G::kOffIdxB) + hb;
    const V* vA = reinterpret_cast<const V*>(st + G::kOffValA) + hva;
    const V* vB = reinterpret_cast<const V*>(st + G::kOffValB) + hvb;
    const uint32_t na = live ? m.na : 0u, nb = live ? m.nb : 0u;

    // ---- merge kCmpPerThread positions; a position is dropped when the next
    // merged position has the same index
    const uint32_t n = na + nb;
    const uint32_t dd = uint32_t(tid) * kCmpPerThread;
    uint32_t mi[kCmpPerThread];
    uint32_t mv[kCmpPerThread];
    uint32_t keep = 0;
    if (dd < n) {
      // keys of the next unconsumed A and B entries; an exhausted side reads
      // as 0xFFFFFFFF, which no index reaches (n < 2^32)
      constexpr uint32_t kInf = 0xFFFFFFFFu;
      uint32_t x = merge_split_shared(sA, na, sB, nb, dd);
      uint32_t y = dd - x;
      uint32_t ak = x < na ? sA[x] : kInf, bk = y < nb ? sB[y] : kInf;
      const uint32_t cnt_here = n - dd < uint32_t(kCmpPerThread) ? n - dd : uint32_t(kCmpPerThread);
#pragma unroll
      for (int e = 0; e < kCmpPerThread; ++e) {
        if (uint32_t(e) < cnt_here) {
          const bool take_a = ak <= bk;  // A first on an equal index
          mi[e] = take_a ? ak : bk;
          mv[e] = take_a ? uint32_t(vA[x]) : uint32_t(vB[y]);
          if (take_a) {
            ++x;
            ak = x < na ? sA[x] : kInf;
          } else {
            ++y;
            bk = y < nb ? sB[y] : kInf;
          }
        }
      }
      // the merged position after this thread's last: the smaller remaining
      // key, or past the tile the smaller of the staged next entries
      uint32_t after = ak < bk ? ak : bk;
      bool has_after = after != kInf;
      if (!has_after) {
        if (m.ext_a) { after = sA[na]; has_after = true; }
        if (m.ext_b && (!has_after || sB[nb] < after)) { after = sB[nb]; has_after = true; }
      }
#pragma unroll
      for (int e = 0; e < kCmpPerThread; ++e) {
        if (uint32_t(e) < cnt_here) {
          const bool last = uint32_t(e) + 1 == cnt_here;
          const uint32_t nxt = last ? after : mi[e + 1 < kCmpPerThread ? e + 1 : e];
          const bool dup = last ? (has_after && after == mi[e]) : nxt == mi[e];
          if (!dup) keep |= 1u << e;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);

    // ---- rank
    const uint32_t cnt = uint32_t(__popc(keep));
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const int pc = int(it & 1u);
    if (lane == 31) sh.warp_tot[pc][warp] = incl;
    if (compute_barrier_or(failed || !live)) break;
    const uint32_t tw = lane < kCmpWarps ? sh.warp_tot[pc][lane] : 0u;
    uint32_t sw = tw;
#pragma unroll
    for (int o = 1; o < kCmpWarps; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, sw, o);
      if (lane >= o) sw += v;
    }
    const uint32_t before = __shfl_sync(0xFFFFFFFFu, sw - tw, warp);
    const uint32_t agg = __shfl_sync(0xFFFFFFFFu, sw, kCmpWarps - 1);
    const uint32_t excl = before + incl - cnt;
    if (tid == 0)
      st_relaxed_u64(a.status + m.tile,
                     make_status(uint64_t(m.tile) == m.first ? kFlagPrefix : kFlagAggregate, a.epoch, agg));

    // ---- room: the parked slot must be free and the ring must hold agg more
    const int q = int(posted % kCmpSlots);
    if (posted >= uint32_t(kCmpSlots))
      failed |= !wait_or_flag(&sh.slot_free[q], ((posted - kCmpSlots) / kCmpSlots) & 1u, a);
    failed |= !wait_ring_room<64>(&sh.ring_tail, ring_head, agg, kCmpRing, a);

    // ---- park the kept entries
    uint32_t r = ring_head + excl;
#pragma unroll
    for (int e = 0; e < kCmpPerThread; ++e) {
      if ((keep >> e) & 1u) {
        ring_idx[r & kCmpRingMask] = mi[e];
        ring_val[r & kCmpRingMask] = V(mv[e]);
        ++r;
      }
    }
    if (tid == 0) {
      CmpParked pm;
      pm.tile = m.tile;
      pm.seg = m.seg;
      pm.agg = agg;
      pm.last = m.last;
      pm.ring_start = ring_head;
      pm.first = m.first;
      pm.total = m.total;
      pm.idx_out = m.idx_out;
      pm.val_out = m.val_out;
      sh.parked[q] = pm;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.agg_ready[q]);
    ++posted;
    ring_head += agg;
  }
  for (uint32_t e = posted > uint32_t(kCmpSlots) ? posted - kCmpSlots : 0u; e < posted; ++e)
    wait_or_flag(&sh.slot_free[e % kCmpSlots], (e / kCmpSlots) & 1u, a);
  compute_barrier();
  const int q = int(posted % kCmpSlots);
  if (tid == 0) {
    CmpParked pm{};
    pm.last = 2u;
    sh.parked[q] = pm;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&sh.agg_ready[q]);
}

template <class V, bool MULTI>
__global__ void __launch_bounds__(kEncBlockThreads, kEncMinBlocks)
    compose_kernel(const __grid_constant__ CmpLaunch a) {
  using G = CmpGeom<V>;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ CmpShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 127) & ~uintptr_t(127));
  uint32_t* ring_idx = reinterpret_cast<uint32_t*>(stages + size_t(kCmpStages) * G::kStageBytes);
  V* ring_val = reinterpret_cast<V*>(ring_idx + kCmpRing);
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kCmpStages; ++s) {
      mbar_init(&sh.full[s], 2);  // producer: bulk bytes expected + plain stores done
      mbar_init(&sh.empty[s], kCmpWarps);
      sh.meta[s] = CmpStageMeta{};
      sh.meta[s].mode = enc::kModeEnd;
    }
#pragma unroll
    for (int q = 0; q < kCmpSlots; ++q) {
      mbar_init(&sh.agg_ready[q], kCmpWarps);
      mbar_init(&sh.slot_free[q], 1);
      sh.parked[q] = CmpParked{};
      sh.parked[q].last = 2u;
    }
    sh.ring_tail = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp < kCmpWarps) {
    cmp_compute<V>(a, sh, stages, ring_idx, ring_val, tid, lane, warp);
  } else if (warp == enc::kProducerWarp) {
    if (lane == 0) cmp_producer<V, MULTI>(a, sh, stages);
  } else {
    cmp_lookback<V, MULTI>(a, sh, ring_idx, ring_val, lane);
  }
}

template <class V, bool MULTI>
int compose_blocks_per_sm() {
  static int cached = [] {
    cudaFuncSetAttribute(compose_kernel<V, MULTI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         int(CmpGeom<V>::kDynSmem));
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, compose_kernel<V, MULTI>, kEncBlockThreads,
                                                      CmpGeom<V>::kDynSmem) != cudaSuccess || b < 1)
      b = 1;
    return b;
  }();
  return cached;
}

template <class V, bool MULTI>
void launch_compose_t(const CmpLaunch& a, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t cap = uint64_t(sm_count(dev)) * uint64_t(compose_blocks_per_sm<V, MULTI>());
  const unsigned grid = unsigned(a.total_tiles < cap ? a.total_tiles : cap);
  compose_kernel<V, MULTI><<<grid, kEncBlockThreads, CmpGeom<V>::kDynSmem, stream>>>(a);
}

}  // namespace

uint64_t compose_tiles(uint64_t entries) { return (entries + kCmpTile - 1) / kCmpTile; }

cudaError_t launch_compose(const CmpSegment* segs_dev, const CmpSegment& one,
                           const uint64_t* tile_begin_dev, int nsegs, uint64_t total_tiles,
                           uint32_t* splits, uint32_t* tile_seg, uint64_t* status,
                           uint32_t* counters,
                           uint64_t* counts_out, uint32_t epoch, uint64_t wait_limit_ns,
                           int value_bytes, cudaStream_t stream) {
  if (total_tiles == 0) return cudaSuccess;
  CmpLaunch a{};
  a.segs = segs_dev;
  a.one = one;
  a.tile_begin = tile_begin_dev;
  a.nsegs = nsegs;
  a.total_tiles = total_tiles;
  a.splits = splits;
  a.tile_seg = tile_seg;
  a.status = status;
  a.counters = counters;
  a.counts_out = counts_out;
  a.epoch = epoch;
  a.wait_limit_ns = wait_limit_ns;
  const bool multi = segs_dev != nullptr;
  const unsigned pgrid = unsigned((total_tiles + 255) / 256);
  if (multi) compose_partition_kernel<true><<<pgrid, 256, 0, stream>>>(a, splits, tile_seg);
  else compose_partition_kernel<false><<<pgrid, 256, 0, stream>>>(a, splits, tile_seg);
  if (value_bytes == 2) {
    if (multi) launch_compose_t<uint16_t, true>(a, stream);
    else launch_compose_t<uint16_t, false>(a, stream);
  } else {
    if (multi) launch_compose_t<uint8_t, true>(a, stream);
    else launch_compose_t<uint8_t, false>(a, stream);
  }
  return cudaGetLastError();
}

}  // namespace pulse
