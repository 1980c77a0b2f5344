// loco.cu -- the PULSELoCo sender step and the receiver's accumulation.
//
// PULSE summary (arXiv 2602.03839), "Metodologia: PULSE -- 2. PULSELoCo":
// workers run H local Adam steps from a shared global checkpoint and form a
// pseudo-gradient (the parameter change); the compute-visibility gate is
// applied to these FP32 pseudo-gradients and only entries that would change
// the BF16 representation are synchronised; the others are kept in an FP32
// error-feedback buffer and revisited in the next round.
//
// Per element: d = local - global; u = d + err (each rounded once, no fused
// multiply-add; a NaN u is the quiet NaN 0x7FC00000); u passes iff the BF16
// view of global + u differs bitwise from the BF16 view of global (RNE,
// every NaN -> 0x7FC0); a passing entry is emitted as (index, u) in
// ascending order and its error becomes +0, a failing entry keeps u as its
// error.
//
// Kernel: the encode kernels' persistent warp-specialized CTA. The producer
// warp bulk-copies each 2048-element tile of global, local and err into a
// 2-stage shared-memory ring; 8 compute warps evaluate the gate (4 elements
// per thread per round, 2 rounds), store the new error straight to global
// memory, rank the passing entries and park them (11-bit local index + FP32
// value) in a shared ring; the look-back warp resolves each parked tile's
// output offset (decoupled look-back) and copies the entries out.
#include "encode_common.cuh"

namespace pulse {
namespace {

using namespace enc;

constexpr int kLocoRounds = 2;
constexpr int kLocoTile = kEncThreads * kLocoRounds * 4;  // 2048 elements
constexpr uint32_t kLocoRing = 4096;                       // parked entries per CTA
constexpr uint32_t kLocoRingMask = kLocoRing - 1;
constexpr uint32_t kArrBytes = kLocoTile * 4;               // one FP32 array per tile
constexpr uint32_t kStageBytes = 3 * kArrBytes;             // global, local, err
constexpr size_t kDynSmem = size_t(kEncStages) * kStageBytes + size_t(kLocoRing) * 6 + 128;
static_assert(kLocoRing >= uint32_t(kLocoTile), "the ring holds a whole tile");
static_assert(kEncLookbackWarps == 1, "parked tiles are copied out in order by one look-back warp");

struct LocoStageMeta {
  uint32_t tile;
  uint32_t tensor;
  uint32_t mode;
  uint32_t len;
  uint64_t base;
  uint64_t first;
  uint64_t n;
  const float* global;
  const float* local;
  float* err;
  uint32_t* idx;
  float* val;
};

struct LocoParked {
  uint32_t tile;
  uint32_t tensor;
  uint32_t agg;
  uint32_t last;  // 1: last tile of its tensor; 2: no more tiles
  uint32_t ring_start;
  uint64_t first;
  uint64_t n;
  uint64_t base;
  uint32_t* idx;
  float* val;
};

struct __align__(16) LocoShared {
  uint64_t full[kEncStages];
  uint64_t empty[kEncStages];
  uint64_t agg_ready[kPendSlots];
  uint64_t slot_free[kPendSlots];
  LocoStageMeta meta[kEncStages];
  LocoParked parked[kPendSlots];
  uint32_t warp_tot[2][kWarps];
  uint32_t ring_tail;
};

// BF16 views of a pair with every NaN read as 0x7FC0.
__device__ __forceinline__ uint32_t view2(float lo, float hi) {
  uint32_t b = cvt_bf16x2_rn(lo, hi);
  if (any_nan2(lo, hi)) b = canon_nan_pair(b, lo, hi);
  return b;
}

// ------------------------------------------------------------ producer warp
template <bool MULTI>
__device__ __forceinline__ void loco_producer(const LocoLaunch& a, LocoShared& sh, uint8_t* stages) {
  const uint64_t pol = l2_policy_evict_first();
  uint32_t fills_done = 0;
  uint32_t ticket = atomicAdd(a.counters + 0, 1u) + a.first_ticket;
  uint32_t cur_t = 0;
  uint64_t cur_begin = 1, cur_end = 0;
  LocoTensorDesc d = a.one;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kEncStages);
    const bool end = ticket >= a.total_tiles;
    const uint32_t next = end ? ticket : atomicAdd(a.counters + 0, 1u) + a.first_ticket;
    if (it >= uint32_t(kEncStages) && !helper_wait(&sh.empty[s], ((it / kEncStages) - 1) & 1u, a))
      break;
    fills_done = it + 1;
    LocoStageMeta m{};
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
    const uint64_t base = (uint64_t(ticket) - d.tile_begin) * kLocoTile;
    const uint64_t len = d.n - base < uint64_t(kLocoTile) ? d.n - base : uint64_t(kLocoTile);
    m.tensor = cur_t;
    m.len = uint32_t(len);
    m.base = base;
    m.first = d.tile_begin;
    m.n = d.n;
    m.global = d.global;
    m.local = d.local;
    m.err = d.err;
    m.idx = d.idx;
    m.val = d.val;
    if (d.bulk_ok && len == uint64_t(kLocoTile)) {
      m.mode = kModeBulk;
      sh.meta[s] = m;
      uint8_t* st = stages + size_t(s) * kStageBytes;
      mbar_arrive_expect_tx(&sh.full[s], kStageBytes);
      bulk_g2s(st, d.global + base, kArrBytes, &sh.full[s], pol);
      bulk_g2s(st + kArrBytes, d.local + base, kArrBytes, &sh.full[s], pol);
      // err is rewritten by the compute warps right after: default L2 policy
      bulk_g2s_plain(st + 2 * kArrBytes, d.err + base, kArrBytes, &sh.full[s]);
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
__device__ __forceinline__ void loco_copy_out(const LocoParked& pm, uint32_t prefix,
                                              const uint16_t* ring_idx, const float* ring_val,
                                              int lane) {
  const uint32_t agg = pm.agg;
  const uint32_t base = uint32_t(pm.base);
  const bool vec = (reinterpret_cast<uintptr_t>(pm.idx) % 16u == 0) &&
                   (reinterpret_cast<uintptr_t>(pm.val) % 16u == 0) &&
                   uint64_t(prefix) + agg <= pm.n;
  uint32_t head = vec ? ((4u - (prefix & 3u)) & 3u) : agg;
  if (head > agg) head = agg;
  const uint32_t body = vec ? ((agg - head) & ~3u) : 0u;
  auto one = [&](uint32_t k) {
    const uint64_t pos = uint64_t(prefix) + k;
    if (pos < pm.n) {
      const uint32_t r = (pm.ring_start + k) & kLocoRingMask;
      pm.idx[pos] = base + ring_idx[r];
      pm.val[pos] = ring_val[r];
    }
  };
  for (uint32_t k = uint32_t(lane); k < head; k += 32) one(k);
  for (uint32_t k = head + uint32_t(lane) * 4u; k < head + body; k += 128u) {
    uint32_t e[4];
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t r = (pm.ring_start + k + uint32_t(q)) & kLocoRingMask;
      e[q] = base + ring_idx[r];
      v[q] = ring_val[r];
    }
    const uint64_t pos = uint64_t(prefix) + k;
    *reinterpret_cast<uint4*>(pm.idx + pos) = make_uint4(e[0], e[1], e[2], e[3]);
    *reinterpret_cast<float4*>(pm.val + pos) = make_float4(v[0], v[1], v[2], v[3]);
  }
  for (uint32_t k = head + body + uint32_t(lane); k < agg; k += 32) one(k);
}

__device__ __forceinline__ void loco_lookback(const LocoLaunch& a, LocoShared& sh,
                                              const uint16_t* ring_idx, const float* ring_val,
                                              int lane, bool multi) {
  for (uint32_t i = 0;;) {
    const bool ok = helper_wait(&sh.agg_ready[i % kPendSlots], (i / kPendSlots) & 1u, a);
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    int more = 0;
    if (lane == 0) {
      for (int b = 1; b < kLookbackBatch; ++b) {
        const uint32_t ii = i + uint32_t(b);
        if (!mbar_test_wait(&sh.agg_ready[ii % kPendSlots], (ii / kPendSlots) & 1u)) break;
        more = b;
      }
    }
    more = __shfl_sync(0xFFFFFFFFu, more, 0);
    int nb = 0;
    bool end = false;
    uint64_t win[kLookbackBatch][kLookbackPerLane];
#pragma unroll
    for (int b = 0; b < kLookbackBatch; ++b) {
      if (b > more || end) continue;
      const uint32_t ii = i + uint32_t(b);
      const int q = int(ii % kPendSlots);
      if (b > 0) mbar_test_wait(&sh.agg_ready[q], (ii / kPendSlots) & 1u);  // acquire for every lane
      const LocoParked& pm = sh.parked[q];
      if (pm.last == 2u) {
        end = true;
        continue;
      }
      if (pm.tile != pm.first) load_window<StatusEpoch>(a, int64_t(pm.tile) - 1, pm.first, lane, win[b]);
      nb = b + 1;
    }
#pragma unroll
    for (int b = 0; b < kLookbackBatch; ++b) {
      if (b >= nb) continue;
      const uint32_t ii = i + uint32_t(b);
      const int q = int(ii % kPendSlots);
      const LocoParked pm = sh.parked[q];
      const uint32_t prefix = resolve_prefix<StatusEpoch>(a, pm.tile, pm.first, pm.agg, lane, win[b]);
      if (lane == 0 && pm.last == 1u) a.counts_out[multi ? pm.tensor : 0] = uint64_t(prefix) + pm.agg;
      loco_copy_out(pm, prefix, ring_idx, ring_val, lane);
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
__device__ __forceinline__ void loco_compute(const LocoLaunch& a, LocoShared& sh, uint8_t* stages,
                                             uint16_t* ring_idx, float* ring_val, int tid, int lane,
                                             int warp) {
  uint32_t posted = 0, ring_head = 0;
  bool failed = false;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kEncStages);
    failed |= !wait_or_flag(&sh.full[s], (it / kEncStages) & 1u, a);
    const LocoStageMeta m = sh.meta[s];
    const bool live = m.mode != kModeEnd;
    const bool bulk = m.mode == kModeBulk;
    const uint64_t base = m.base;
    const uint32_t len = m.len;
    const uint8_t* st = stages + size_t(s) * kStageBytes;

    float u[kLocoRounds][4];
    uint32_t flags = 0;  // bit 4j + e: element e of round j passes
#pragma unroll
    for (int j = 0; j < kLocoRounds; ++j) {
      const uint32_t li = uint32_t(j * kEncThreads + tid) * 4u;
      float4 g4, w4, e4;
      if (bulk) {
        g4 = reinterpret_cast<const float4*>(st)[j * kEncThreads + tid];
        w4 = reinterpret_cast<const float4*>(st + kArrBytes)[j * kEncThreads + tid];
        e4 = reinterpret_cast<const float4*>(st + 2 * kArrBytes)[j * kEncThreads + tid];
      } else {
        float gg[4], ww[4], ee[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool valid = li + e < len;
          gg[e] = valid ? m.global[base + li + e] : 0.0f;
          ww[e] = valid ? m.local[base + li + e] : 0.0f;
          ee[e] = valid ? m.err[base + li + e] : 0.0f;
        }
        g4 = make_float4(gg[0], gg[1], gg[2], gg[3]);
        w4 = make_float4(ww[0], ww[1], ww[2], ww[3]);
        e4 = make_float4(ee[0], ee[1], ee[2], ee[3]);
      }
      u[j][0] = __fadd_rn(__fsub_rn(w4.x, g4.x), e4.x);
      u[j][1] = __fadd_rn(__fsub_rn(w4.y, g4.y), e4.y);
      u[j][2] = __fadd_rn(__fsub_rn(w4.z, g4.z), e4.z);
      u[j][3] = __fadd_rn(__fsub_rn(w4.w, g4.w), e4.w);
      if (any_nan4(u[j][0], u[j][1], u[j][2], u[j][3])) {
        // rare: a NaN sum is stored and sent as the quiet NaN 0x7FC00000
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (u[j][e] != u[j][e]) u[j][e] = __uint_as_float(0x7FC00000u);
      }
      const uint32_t s01 = view2(__fadd_rn(g4.x, u[j][0]), __fadd_rn(g4.y, u[j][1]));
      const uint32_t s23 = view2(__fadd_rn(g4.z, u[j][2]), __fadd_rn(g4.w, u[j][3]));
      const uint32_t d01 = s01 ^ view2(g4.x, g4.y), d23 = s23 ^ view2(g4.z, g4.w);
      uint32_t f = uint32_t((d01 & 0xFFFFu) != 0u) | (uint32_t(d01 > 0xFFFFu) << 1) |
                   (uint32_t((d23 & 0xFFFFu) != 0u) << 2) | (uint32_t(d23 > 0xFFFFu) << 3);
      if (!bulk) {
        const uint32_t nvalid = li >= len ? 0u : (len - li >= 4u ? 4u : len - li);
        f &= (1u << nvalid) - 1u;
      }
      flags |= f << (4 * j);
      // the new error: +0 where the entry is sent, u elsewhere
      const float4 e_new = make_float4((f & 1u) ? 0.0f : u[j][0], (f & 2u) ? 0.0f : u[j][1],
                                       (f & 4u) ? 0.0f : u[j][2], (f & 8u) ? 0.0f : u[j][3]);
      if (bulk) {
        *reinterpret_cast<float4*>(m.err + base + li) = e_new;
      } else if (live) {
        const float ev[4] = {e_new.x, e_new.y, e_new.z, e_new.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (li + e < len) m.err[base + li + e] = ev[e];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);

    // ---- rank: two per-round counts in bytes (at most 32 x 4 = 128)
    const uint32_t cnts = uint32_t(__popc(flags & 0xFu)) | (uint32_t(__popc(flags & 0xF0u)) << 8);
    uint32_t incl = cnts;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    const uint32_t excl = incl - cnts;
    const int pc = int(it & 1u);
    if (lane == 31) sh.warp_tot[pc][warp] = incl;
    if (compute_barrier_or(failed || !live)) break;
    // across warps, round-major: widened to 16-bit fields (at most 8 x 128)
    const uint32_t t = lane < kWarps ? sh.warp_tot[pc][lane] : 0u;
    const uint32_t tw = (t & 0xFFu) | ((t & 0xFF00u) << 8);
    uint32_t sw = tw;
#pragma unroll
    for (int o = 1; o < kWarps; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, sw, o);
      if (lane >= o) sw += v;
    }
    const uint32_t bw = __shfl_sync(0xFFFFFFFFu, sw - tw, warp);
    const uint32_t aw = __shfl_sync(0xFFFFFFFFu, sw, kWarps - 1);
    const uint32_t tot0 = aw & 0xFFFFu, tot1 = aw >> 16;
    const uint32_t off0 = (bw & 0xFFFFu) + (excl & 0xFFu);
    const uint32_t off1 = tot0 + (bw >> 16) + ((excl >> 8) & 0xFFu);
    const uint32_t agg = tot0 + tot1;
    if (tid == 0)
      st_relaxed_u64(a.status + m.tile,
                     make_status(uint64_t(m.tile) == m.first ? kFlagPrefix : kFlagAggregate, a.epoch, agg));

    // ---- room for the tile
    const int q = int(posted % kPendSlots);
    if (posted >= uint32_t(kPendSlots))
      failed |= !wait_or_flag(&sh.slot_free[q], ((posted - kPendSlots) / kPendSlots) & 1u, a);
    failed |= !wait_ring_room<64>(&sh.ring_tail, ring_head, agg, kLocoRing, a);

    // ---- park the passing entries
#pragma unroll
    for (int j = 0; j < kLocoRounds; ++j) {
      uint32_t f = (flags >> (4 * j)) & 0xFu;
      if (f == 0u) continue;
      const uint32_t li = uint32_t(j * kEncThreads + tid) * 4u;
      uint32_t r = ring_head + (j == 0 ? off0 : off1);
      do {
        const uint32_t e = uint32_t(__ffs(f)) - 1u;
        f &= f - 1u;
        ring_idx[r & kLocoRingMask] = uint16_t(li + e);
        ring_val[r & kLocoRingMask] = e == 0 ? u[j][0] : e == 1 ? u[j][1] : e == 2 ? u[j][2] : u[j][3];
        ++r;
      } while (f != 0u);
    }
    if (tid == 0) {
      LocoParked pm;
      pm.tile = m.tile;
      pm.tensor = m.tensor;
      pm.agg = agg;
      pm.last = (base + len == m.n) ? 1u : 0u;
      pm.ring_start = ring_head;
      pm.first = m.first;
      pm.n = m.n;
      pm.base = base;
      pm.idx = m.idx;
      pm.val = m.val;
      sh.parked[q] = pm;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.agg_ready[q]);
    ++posted;
    ring_head += agg;
  }
  for (uint32_t e = posted > uint32_t(kPendSlots) ? posted - kPendSlots : 0u; e < posted; ++e)
    wait_or_flag(&sh.slot_free[e % kPendSlots], (e / kPendSlots) & 1u, a);
  compute_barrier();
  const int q = int(posted % kPendSlots);
  if (tid == 0) {
    LocoParked pm{};
    pm.last = 2u;
    sh.parked[q] = pm;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&sh.agg_ready[q]);
}

template <bool MULTI>
__global__ void __launch_bounds__(kEncBlockThreads, kEncMinBlocks)
    loco_gate_kernel(const __grid_constant__ LocoLaunch a) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ LocoShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 127) & ~uintptr_t(127));
  float* ring_val = reinterpret_cast<float*>(stages + size_t(kEncStages) * kStageBytes);
  uint16_t* ring_idx = reinterpret_cast<uint16_t*>(ring_val + kLocoRing);
  if constexpr (MULTI) {
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
      sh.meta[s] = LocoStageMeta{};
      sh.meta[s].mode = kModeEnd;
    }
#pragma unroll
    for (int q = 0; q < kPendSlots; ++q) {
      mbar_init(&sh.agg_ready[q], kWarps);
      mbar_init(&sh.slot_free[q], 1);
      sh.parked[q] = LocoParked{};
      sh.parked[q].last = 2u;
    }
    sh.ring_tail = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp < kWarps) {
    loco_compute(a, sh, stages, ring_idx, ring_val, tid, lane, warp);
  } else if (warp == kProducerWarp) {
    if (lane == 0) loco_producer<MULTI>(a, sh, stages);
  } else {
    loco_lookback(a, sh, ring_idx, ring_val, lane, MULTI);
  }
}

template <bool MULTI>
int loco_blocks_per_sm() {
  static int cached = [] {
    cudaFuncSetAttribute(loco_gate_kernel<MULTI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         int(kDynSmem));
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, loco_gate_kernel<MULTI>, kEncBlockThreads,
                                                      kDynSmem) != cudaSuccess || b < 1)
      b = 1;
    return b;
  }();
  return cached;
}

// ------------------------------------------------------------ accumulate
// acc[idx[j]] += val[j] (FP32) over one patch segment; an index of a single
// patch appears once, so no two threads touch the same element, and a thread's
// entries are distinct elements: all of its acc loads are issued before any
// of its stores (one memory round trip per tile instead of one per entry).
constexpr int kAccThreads = 256;
#ifndef PULSE_ACC_PER_THREAD
#define PULSE_ACC_PER_THREAD 8  // 9.8 ms on the 8.03B step against 10.3-10.4 with 2 or 4
#endif
constexpr int kAccPerThread = PULSE_ACC_PER_THREAD;
constexpr int kAccTile = kAccThreads * kAccPerThread;

__device__ __forceinline__ void acc_tile(float* acc, uint64_t n, const uint32_t* idx,
                                         const float* val, uint64_t count, uint64_t tile,
                                         uint32_t* err) {
  const uint64_t b = tile * kAccTile + threadIdx.x;
  uint32_t ii[kAccPerThread];
  float vv[kAccPerThread], av[kAccPerThread];
  bool ok[kAccPerThread];
#pragma unroll
  for (int k = 0; k < kAccPerThread; ++k) {
    const uint64_t j = b + uint64_t(k) * kAccThreads;
    ii[k] = j < count ? __ldcs(idx + j) : 0u;
    vv[k] = j < count ? __ldcs(val + j) : 0.0f;
  }
#pragma unroll
  for (int k = 0; k < kAccPerThread; ++k) {
    const uint64_t j = b + uint64_t(k) * kAccThreads;
    ok[k] = j < count && uint64_t(ii[k]) < n;
    if (j < count && !ok[k]) record_error(err, kErrIndex);
    av[k] = ok[k] ? acc[ii[k]] : 0.0f;
  }
#pragma unroll
  for (int k = 0; k < kAccPerThread; ++k)
    if (ok[k]) acc[ii[k]] = __fadd_rn(av[k], vv[k]);
}

__global__ void __launch_bounds__(kAccThreads)
    loco_accumulate_kernel(float* acc, uint64_t n, const uint32_t* idx, const float* val,
                           uint64_t count, uint32_t* err) {
  const uint64_t tiles = (count + kAccTile - 1) / kAccTile;
  for (uint64_t t = blockIdx.x; t < tiles; t += gridDim.x) acc_tile(acc, n, idx, val, count, t, err);
}

// Whole-model accumulate from device-resident counts: every CTA rebuilds the
// tile map (tiles per tensor, prefix over the list) in shared memory.
__global__ void __launch_bounds__(kAccThreads)
    loco_accumulate_multi_kernel(const LocoTensorDesc* tensors, int ntensors,
                                 const uint64_t* counts, uint32_t* err) {
  extern __shared__ uint64_t tile_begin[];  // ntensors + 1
  __shared__ uint64_t warp_tot[kAccThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (ntensors + kAccThreads - 1) / kAccThreads;
  const int t0 = tid * per;
  uint64_t mine = 0;
  for (int t = t0; t < t0 + per && t < ntensors; ++t) {
    uint64_t c = counts[t];
    if (c > tensors[t].n) c = tensors[t].n;
    mine += (c + kAccTile - 1) / kAccTile;
  }
  uint64_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  uint64_t warp_off = 0;
  for (int k = 0; k < warp; ++k) warp_off += warp_tot[k];
  uint64_t run = warp_off + incl - mine;
  for (int t = t0; t < t0 + per && t < ntensors; ++t) {
    tile_begin[t] = run;
    uint64_t c = counts[t];
    if (c > tensors[t].n) c = tensors[t].n;
    run += (c + kAccTile - 1) / kAccTile;
  }
  if (tid == kAccThreads - 1) tile_begin[ntensors] = warp_off + incl;
  __syncthreads();
  if (tid == 0) {
    for (int t = 0; t < ntensors; ++t)
      if (counts[t] > tensors[t].n) record_error(err, kErrIndex);
  }
  const uint64_t total = tile_begin[ntensors];
  for (uint64_t g = blockIdx.x; g < total; g += gridDim.x) {
    int lo = 0, hi = ntensors;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_begin[mid] <= g) lo = mid; else hi = mid - 1;
    }
    const LocoTensorDesc& d = tensors[lo];
    uint64_t c = counts[lo];
    if (c > d.n) c = d.n;
    acc_tile(d.acc, d.n, d.idx, d.val, c, g - tile_begin[lo], err);
  }
}

}  // namespace

uint64_t loco_tiles(uint64_t n) { return (n + kLocoTile - 1) / kLocoTile; }

int loco_grid_size(int device) {
  const int a = loco_blocks_per_sm<true>(), b = loco_blocks_per_sm<false>();
  return sm_count(device) * (a < b ? a : b);
}

cudaError_t launch_loco_gate(const LocoLaunch& a, bool multi, int grid, cudaStream_t stream) {
  if (multi) {
    loco_blocks_per_sm<true>();
    loco_gate_kernel<true><<<grid, kEncBlockThreads, kDynSmem, stream>>>(a);
  } else {
    loco_blocks_per_sm<false>();
    loco_gate_kernel<false><<<grid, kEncBlockThreads, kDynSmem, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_loco_accumulate(float* acc, uint64_t n, const uint32_t* idx, const float* val,
                                   uint64_t count, uint32_t* err, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t tiles = (count + kAccTile - 1) / kAccTile;
  const uint64_t cap = uint64_t(sm_count(dev)) * 8u;
  const int grid = int(tiles < cap ? tiles : cap);
  if (grid == 0) return cudaSuccess;
  loco_accumulate_kernel<<<grid, kAccThreads, 0, stream>>>(acc, n, idx, val, count, err);
  return cudaGetLastError();
}

cudaError_t launch_loco_accumulate_multi(const LocoTensorDesc* tensors, int ntensors,
                                         const uint64_t* counts, uint32_t* err, int grid,
                                         cudaStream_t stream) {
  const size_t smem = size_t(ntensors + 1) * sizeof(uint64_t);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(loco_accumulate_multi_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
  }
  loco_accumulate_multi_kernel<<<grid, kAccThreads, smem, stream>>>(tensors, ntensors, counts, err);
  return cudaGetLastError();
}

}  // namespace pulse
