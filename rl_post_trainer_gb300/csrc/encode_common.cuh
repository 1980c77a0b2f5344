// encode_common.cuh -- pieces shared by the persistent encode kernels (the
// BF16 view in encode.cu, the MXFP8 view in encode_mx.cu): CTA roles, the
// compute warps' named barrier, bounded waits, and the single-pass decoupled
// look-back (Merrill & Garland, "Single-pass Parallel Prefix Scan with
// Decoupled Look-back", 2016) over a status word per tile.
//
// Both kernels have the same CTA layout: kEncThreads compute threads (8
// warps), one producer warp, kEncLookbackWarps look-back warps; tiles of
// kEncTile elements are handed out by a global ticket counter.
#pragma once

#include "pulse_device.cuh"
#include "pulse_internal.h"

namespace pulse {
namespace enc {

constexpr int kWarps = kEncThreads / 32;  // compute warps
constexpr int kProducerWarp = kWarps;
constexpr int kFirstLookbackWarp = kWarps + 1;
static_assert(kEncRounds == 4, "four rounds pack into the bytes of one word");
static_assert(kWarps == 8, "the cross-warp scan runs over 8 lanes");
constexpr int kLookbackPerLane = kEncLookbackPerLane;
constexpr int kLookbackBatch = kEncLookbackBatch;
// parked-tile slots: a multiple of the look-back warps (slot p is always
// handled by look-back warp p % kEncLookbackWarps), at least kEncParked
constexpr int kPendSlots =
    ((kEncParked > kEncLookbackWarps ? kEncParked : kEncLookbackWarps) + kEncLookbackWarps - 1) /
    kEncLookbackWarps * kEncLookbackWarps;
constexpr int kComputeBarrier = 1;  // named barrier of the compute warps
// Ring slot of position r < 2 * kEncRing (a ring start below kEncRing plus
// at most one tile): a mask for a power-of-two ring, else one subtraction.
__device__ __forceinline__ uint32_t ring_slot(uint32_t r) {
  if constexpr ((kEncRing & (kEncRing - 1)) == 0) return r & uint32_t(kEncRing - 1);
  else return r >= uint32_t(kEncRing) ? r - uint32_t(kEncRing) : r;
}

enum : uint32_t { kModeEnd = 0, kModeBulk = 1, kModeGeneric = 2 };

__device__ __forceinline__ int find_tensor(const uint64_t* tile_begin, int ntensors, uint64_t g) {
  // largest t with tile_begin[t] <= g; tile_begin[ntensors] = total > g
  int lo = 0, hi = ntensors;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(tile_begin + mid) <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void bulk_g2s_plain(void* smem_dst, const void* gmem_src,
                                               uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void compute_barrier() {
  asm volatile("bar.sync %0, %1;" ::"n"(kComputeBarrier), "n"(kEncThreads) : "memory");
}

// Named barrier of the compute warps that also ORs a predicate across them:
// every loop-exit decision goes through it, so the 8 compute warps always
// leave their loop together and no named barrier is ever left short.
__device__ __forceinline__ bool compute_barrier_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(v)), "n"(kComputeBarrier), "n"(kEncThreads)
      : "memory");
  return r != 0;
}

// Bounded wait for the producer and look-back warps. The hardware suspends
// the waiting warp between tries, so waiting warps leave the issue slots to
// the compute warps. Same failure contract as wait_or_flag below.
template <class L>
__device__ __forceinline__ bool helper_wait(uint64_t* bar, uint32_t parity, const L& a) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 28); ++it) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if ((it & 15u) == 15u) {
      if (ld_volatile_u32(a.counters + 2) & kErrTimeout) return false;
      if (global_timer_ns() - t0 > a.wait_limit_ns) break;
    }
  }
  record_error(a.counters + 2, kErrTimeout);
  return false;
}

// Bounded mbarrier wait. Returns false if it gave up (the error is recorded);
// once any wait of the launch has given up, later waits give up at once, so
// a failed launch ends quickly. Callers stop after a failed wait; every
// write they may still make stays in bounds.
template <class L>
__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, const L& a) {
  // the hardware suspends the warp for up to 20 us per try
#pragma unroll 1
  for (int i = 0; i < 4; ++i)
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  if (ld_volatile_u32(a.counters + 2) & kErrTimeout) return false;
  if (mbar_wait_bounded(bar, parity, a.wait_limit_ns)) return true;
  record_error(a.counters + 2, kErrTimeout);
  return false;
}

// Bounded wait of a compute thread for room in its CTA's entry ring: until
// head + need - tail <= cap, with tail advanced by the copy-out warp. The
// spin reads only shared memory; the clock and the launch's error word (which
// shares an L2 sector with the tile tickets) are read every 64th turn, so a
// dense tile's waiting threads do not keep that sector busy for every CTA.
// Returns false if it gave up (the error is recorded).
template <unsigned kSleepNs, class L>
__device__ __forceinline__ bool wait_ring_room(const uint32_t* tail, uint32_t head, uint32_t need,
                                               uint32_t cap, const L& a) {
  const volatile uint32_t* t = tail;
  if (head + need - *t <= cap) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t spin = 0; head + need - *t > cap; ++spin) {
    __nanosleep(kSleepNs);
    if ((spin & 63u) == 63u &&
        (global_timer_ns() - t0 > a.wait_limit_ns || (ld_volatile_u32(a.counters + 2) & kErrTimeout))) {
      record_error(a.counters + 2, kErrTimeout);
      return false;
    }
  }
  return true;
}

template <class T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// ------------------------------------------------------------ status words
// StatusEpoch: the BF16 kernel's word, [flag 2 | launch epoch 30 | count 32];
// words of other launches read as unpublished, so nothing is cleared between
// launches.
struct StatusEpoch {
  using value_t = uint32_t;
  static __device__ __forceinline__ uint32_t flag(uint64_t w, uint32_t epoch) {
    return status_flag(w, epoch);
  }
  static __device__ __forceinline__ value_t value(uint64_t w) { return status_value(w); }
  static __device__ __forceinline__ uint64_t make(uint32_t flag, uint32_t epoch, value_t v) {
    return make_status(flag, epoch, v);
  }
};

// StatusPacked: [flag 2 | value 62] with two counts in the value (low 32
// bits and the 30 bits above them) that add field by field as long as
// neither overflows. No epoch: the status words are cleared before every
// launch.
struct StatusPacked {
  using value_t = uint64_t;
  static constexpr uint64_t kValueMask = (uint64_t(1) << 62) - 1u;
  static __device__ __forceinline__ uint32_t flag(uint64_t w, uint32_t) { return uint32_t(w >> 62); }
  static __device__ __forceinline__ value_t value(uint64_t w) { return w & kValueMask; }
  static __device__ __forceinline__ uint64_t make(uint32_t flag, uint32_t, value_t v) {
    return (uint64_t(flag) << 62) | (v & kValueMask);
  }
};

// Issue the loads of one look-back window: the W x 32 status words before
// `pos`, nearest first; words before the tensor's first tile read as an
// inclusive prefix of 0.
template <class S, class L, int W = kLookbackPerLane>
__device__ __forceinline__ void load_window(const L& a, int64_t pos, uint64_t first, int lane,
                                            uint64_t (&w)[W]) {
#pragma unroll
  for (int q = 0; q < W; ++q) {
    const int64_t tile = pos - (lane * W + q);
    w[q] = tile >= int64_t(first) ? ld_relaxed_u64(a.status + tile)
                                  : S::make(kFlagPrefix, a.epoch, 0u);
  }
}

// Look-back warp: exclusive prefix of tile g within its tensor (its own
// aggregate is already published). Reads W x 32 predecessor words per round
// trip, nearest first; waits only on unpublished words that lie before the
// nearest inclusive prefix; publishes g's inclusive prefix. `w` holds the
// first window (load_window at g - 1), already in flight. kSleepNs: pause
// between polls of unpublished words.
template <class S, class L, unsigned kSleepNs = 32, int W = kLookbackPerLane>
__device__ __forceinline__ typename S::value_t resolve_prefix(const L& a, uint64_t g,
                                                              uint64_t first,
                                                              typename S::value_t agg, int lane,
                                                              uint64_t (&w)[W]) {
  constexpr int kLookbackPerLane = W;
  using V = typename S::value_t;
  uint64_t* st = a.status;
  if (g == first) return V(0);  // published as an inclusive prefix already
  constexpr int kNone = 1 << 30;
  V prefix = 0;
  int64_t pos = int64_t(g) - 1;
  bool gave_up = false;
  for (bool first_window = true;; first_window = false) {
    if (!first_window) load_window<S, L, W>(a, pos, first, lane, w);
    int dp = kNone;  // window distance of the nearest inclusive prefix
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 0;; ++spin) {
      int my_p = kNone, my_x = kNone;
#pragma unroll
      for (int q = kLookbackPerLane - 1; q >= 0; --q) {
        const uint32_t f = S::flag(w[q], a.epoch);
        if (f == kFlagPrefix) my_p = lane * kLookbackPerLane + q;
        if (f == 0u) my_x = lane * kLookbackPerLane + q;
      }
      dp = __reduce_min_sync(0xFFFFFFFFu, my_p);
      const int dx = __reduce_min_sync(0xFFFFFFFFu, my_x);
      if (dx == kNone || dx > dp) break;  // every word up to the nearest prefix is published
      if (gave_up || (spin & 63u) == 63u) {
        const bool late = gave_up || spin > (1u << 26) ||
                          global_timer_ns() - t0 > a.wait_limit_ns ||
                          (ld_volatile_u32(a.counters + 2) & kErrTimeout);
        if (__any_sync(0xFFFFFFFFu, late)) {
          // give up: unpublished words read as an inclusive prefix of 0, which
          // keeps every offset at or below the true one (writes stay in bounds)
          if (lane == 0) record_error(a.counters + 2, kErrTimeout);
          gave_up = true;
#pragma unroll
          for (int q = 0; q < kLookbackPerLane; ++q)
            if (S::flag(w[q], a.epoch) == 0u) w[q] = S::make(kFlagPrefix, a.epoch, 0u);
          continue;
        }
      }
      __nanosleep(kSleepNs);
#pragma unroll
      for (int q = 0; q < kLookbackPerLane; ++q) {
        if (S::flag(w[q], a.epoch) == 0u)
          w[q] = ld_relaxed_u64(st + (pos - (lane * kLookbackPerLane + q)));
      }
    }
    V sum = 0;
#pragma unroll
    for (int q = 0; q < kLookbackPerLane; ++q)
      if (lane * kLookbackPerLane + q <= dp) sum += S::value(w[q]);
    prefix += warp_sum(sum);
    if (dp != kNone) break;
    pos -= 32 * kLookbackPerLane;
  }
  if (lane == 0) st_relaxed_u64(st + g, S::make(kFlagPrefix, a.epoch, prefix + agg));
  return prefix;
}

}  // namespace enc
}  // namespace pulse
