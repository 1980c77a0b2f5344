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
//    position (stable merge, A before B on an equal index);
//  * compose kernel: one CTA per tile of kCmpTile merged positions, in ticket
//    order. The CTA stages its A and B ranges in shared memory, each thread
//    merges 8 positions (its own merge-path search in shared memory), keeps a
//    position unless the next merged position has the same index (the pair
//    A-entry, B-entry of a shared index keeps only B's), ranks the kept
//    entries with a block scan, finds its output offset with a decoupled
//    look-back over per-tile status words, and writes them out.
#include "encode_common.cuh"

namespace pulse {
namespace {

#ifndef PULSE_CMP_PER_THREAD
#define PULSE_CMP_PER_THREAD 8
#endif
#ifndef PULSE_CMP_MIN_BLOCKS
#define PULSE_CMP_MIN_BLOCKS 6
#endif
constexpr int kCmpThreads = 256;
constexpr int kCmpPerThread = PULSE_CMP_PER_THREAD;
constexpr int kCmpTile = kCmpThreads * kCmpPerThread;  // merged positions per tile
constexpr int kCmpWarps = kCmpThreads / 32;

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

template <class V>
struct __align__(16) CmpShared {
  uint32_t ia[kCmpTile];   // staged A indices (then: merged indices)
  uint32_t ib[kCmpTile];   // staged B indices
  V va[kCmpTile];
  V vb[kCmpTile];
  uint32_t warp_tot[kCmpWarps];
  uint32_t ticket;
  uint32_t next_idx;       // index of the first merged position after the tile
  uint32_t has_next;
  uint32_t prefix;
};

template <class V, bool MULTI>
__global__ void __launch_bounds__(kCmpThreads, PULSE_CMP_MIN_BLOCKS)
    compose_kernel(const __grid_constant__ CmpLaunch a) {
  __shared__ CmpShared<V> sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) sh.ticket = atomicAdd(a.counters + 0, 1u);
  __syncthreads();
  const uint64_t g = sh.ticket;  // tiles are taken in ticket order: predecessors already run

  int t = 0;
  if constexpr (MULTI) t = int(a.tile_seg[g]);
  const CmpSegment& s = seg_of<MULTI>(a, t);
  const uint64_t first = s.tile_begin;
  const uint64_t total = s.count_a + s.count_b;
  const uint64_t d0 = (g - first) * kCmpTile;
  const uint64_t d1 = d0 + kCmpTile < total ? d0 + kCmpTile : total;
  const bool last_tile = d1 == total;
  const uint64_t i0 = a.splits[g];
  const uint64_t i1 = last_tile ? s.count_a : a.splits[g + 1];
  const uint64_t j0 = d0 - i0, j1 = d1 - i1;
  const uint32_t na = uint32_t(i1 - i0), nb = uint32_t(j1 - j0);
  const V* val_a = static_cast<const V*>(s.val_a);
  const V* val_b = static_cast<const V*>(s.val_b);

  // ---- stage the tile's A and B ranges
  for (uint32_t k = tid; k < na; k += kCmpThreads) {
    sh.ia[k] = s.idx_a[i0 + k];
    sh.va[k] = val_a[i0 + k];
  }
  for (uint32_t k = tid; k < nb; k += kCmpThreads) {
    sh.ib[k] = s.idx_b[j0 + k];
    sh.vb[k] = val_b[j0 + k];
  }
  if (tid == 0) {
    // the merged position right after the tile: the smaller of the next A
    // and next B index (equal indices give the same value either way)
    uint32_t nx = 0xFFFFFFFFu, has = 0;
    if (i1 < s.count_a) { nx = s.idx_a[i1]; has = 1; }
    if (j1 < s.count_b) { const uint32_t v = s.idx_b[j1]; if (!has || v < nx) nx = v; has = 1; }
    sh.next_idx = nx;
    sh.has_next = has;
  }
  __syncthreads();

  // ---- merge kCmpPerThread positions per thread; a position is dropped when
  // the next merged position has the same index. The position after a
  // thread's last one is the smaller of the next unconsumed A and B entries
  // (or, past the tile, the first position of the next tile).
  const uint32_t n = na + nb;
  const uint32_t dd = uint32_t(tid) * kCmpPerThread;
  uint32_t mi[kCmpPerThread];
  V mv[kCmpPerThread];
  uint32_t keep = 0;  // bit e: merged position dd + e is kept
  if (dd < n) {
    uint32_t x = merge_split_shared(sh.ia, na, sh.ib, nb, dd);
    uint32_t y = dd - x;
#pragma unroll
    for (int e = 0; e < kCmpPerThread; ++e) {
      if (dd + e < n) {
        const bool take_a = y >= nb || (x < na && sh.ia[x] <= sh.ib[y]);
        mi[e] = take_a ? sh.ia[x] : sh.ib[y];
        mv[e] = take_a ? sh.va[x] : sh.vb[y];
        x += take_a ? 1u : 0u;
        y += take_a ? 0u : 1u;
      }
    }
    uint32_t after = sh.next_idx;
    bool has_after = sh.has_next != 0;
    if (x < na || y < nb) {
      after = (y >= nb || (x < na && sh.ia[x] <= sh.ib[y])) ? sh.ia[x] : sh.ib[y];
      has_after = true;
    }
#pragma unroll
    for (int e = 0; e < kCmpPerThread; ++e) {
      if (dd + e < n) {
        const bool last = e + 1 == kCmpPerThread || dd + e + 1 == n;
        const bool dup = last ? (has_after && after == mi[e]) : mi[e + 1 < kCmpPerThread ? e + 1 : e] == mi[e];
        if (!dup) keep |= 1u << e;
      }
    }
  }
  const uint32_t cnt = uint32_t(__popc(keep));

  // ---- block scan of kept counts
  uint32_t incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) sh.warp_tot[warp] = incl;
  __syncthreads();
  uint32_t before = 0, agg = 0;
#pragma unroll
  for (int w = 0; w < kCmpWarps; ++w) {
    const uint32_t v = sh.warp_tot[w];
    before += w < warp ? v : 0u;
    agg += v;
  }
  const uint32_t excl = before + incl - cnt;

  // ---- tile offset: decoupled look-back by warp 0
  if (warp == 0) {
    if (lane == 0)
      st_relaxed_u64(a.status + g, make_status(g == first ? kFlagPrefix : kFlagAggregate, a.epoch, agg));
    uint64_t win[enc::kLookbackPerLane];
    uint32_t prefix = 0;
    if (g != first) {
      enc::load_window<enc::StatusEpoch>(a, int64_t(g) - 1, first, lane, win);
      prefix = enc::resolve_prefix<enc::StatusEpoch>(a, g, first, agg, lane, win);
    }
    if (lane == 0) {
      sh.prefix = prefix;
      if (last_tile) a.counts_out[MULTI ? t : 0] = uint64_t(prefix) + agg;
    }
  }
  __syncthreads();
  const uint64_t base = uint64_t(sh.prefix) + excl;
  uint32_t r = 0;
#pragma unroll
  for (int e = 0; e < kCmpPerThread; ++e) {
    if ((keep >> e) & 1u) {
      const uint64_t pos = base + r;
      if (pos < total) {  // only fails after a wait gave up
        s.idx_out[pos] = mi[e];
        static_cast<V*>(s.val_out)[pos] = mv[e];
      }
      ++r;
    }
  }

  // the last CTA to finish rewinds the ticket and finish counters
  if (tid == 0) {
    __threadfence();
    const uint32_t done = atomicAdd(a.counters + 1, 1u);
    if (done == gridDim.x - 1) {
      atomicExch(a.counters + 0, 0u);
      atomicExch(a.counters + 1, 0u);
    }
  }
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
  const unsigned grid = unsigned(total_tiles);
  if (value_bytes == 2) {
    if (multi) compose_kernel<uint16_t, true><<<grid, kCmpThreads, 0, stream>>>(a);
    else compose_kernel<uint16_t, false><<<grid, kCmpThreads, 0, stream>>>(a);
  } else {
    if (multi) compose_kernel<uint8_t, true><<<grid, kCmpThreads, 0, stream>>>(a);
    else compose_kernel<uint8_t, false><<<grid, kCmpThreads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace pulse
