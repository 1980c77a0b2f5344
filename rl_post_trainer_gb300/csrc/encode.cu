// encode.cu -- fused cast + compare + order-preserving compaction.
//
// Trainer-side step of compute-visible weight sync: project the FP32 master
// to its BF16 view, compare with the previous view bit for bit, and emit the
// changed positions with their new absolute values in ascending order
// ("Taking Reinforcement Learning Cross Datacenter", talk 10:49-11:08; PULSE
// summary, section "Metodologia: PULSE -- 1. PULSESync"), refreshing the
// previous view in place.
//
// Kernel structure (one launch covers one tensor or a whole model):
//  * persistent CTAs (SMs x resident CTAs); each takes tiles from a global
//    ticket counter, so every tile's predecessors belong to CTAs that are
//    already running and the look-back below always makes progress;
//  * a kEncStages-deep ring of shared-memory stages filled by bulk copies
//    (cp.async.bulk + mbarrier transaction counts): while a CTA resolves one
//    tile's global offset, the next tiles are already streaming in;
//  * per tile: 4 elements per thread per round, warp ballots give each
//    thread's rank inside its warp, one warp scans the (round, warp) counts,
//    and a single-pass decoupled look-back (Merrill & Garland, "Single-pass
//    Parallel Prefix Scan with Decoupled Look-back", 2016) turns tile counts
//    into global offsets; the look-back warp reads 128 predecessor words per
//    step so the chain keeps up at HBM rates;
//  * epilogue: (index, value) pairs at their global positions, and the new
//    BF16 values written back to prev in 8-byte groups that hold a change.
// Every wait is bounded; a wait that gives up records PULSE_ERR_TIMEOUT and
// the kernel still finishes with all writes inside the caller's buffers.
#include "pulse_device.cuh"
#include "pulse_internal.h"

namespace pulse {
namespace {

constexpr int kWarps = kEncThreads / 32;
constexpr int kPairs = kEncRounds * kWarps;  // (round, warp) pairs in tile order
static_assert(kPairs == 32, "one warp scans the (round, warp) counts");
constexpr int kLookbackPerLane = 4;          // 128 predecessor words per step

constexpr uint32_t kStageMasterBytes = kEncTile * 4;
constexpr uint32_t kStagePrevBytes = kEncTile * 2;
constexpr uint32_t kStageBytes = kStageMasterBytes + kStagePrevBytes;
constexpr size_t kDynSmem = size_t(kEncStages) * kStageBytes + 128;  // +128 for alignment

enum : uint32_t { kModeEnd = 0, kModeBulk = 1, kModeGeneric = 2 };

struct StageMeta {
  uint32_t tile;    // global tile id
  uint32_t tensor;  // tensor index (0 in single-tensor mode)
  uint32_t mode;
  uint32_t pad;
};

struct __align__(16) EncodeShared {
  uint64_t bar[kEncStages];
  StageMeta meta[kEncStages];
  uint32_t pair_count[kPairs];
  uint32_t pair_offset[kPairs];
  uint32_t tile_prefix;
};

__device__ __forceinline__ int find_tensor(const uint64_t* tile_begin, int ntensors, uint64_t g) {
  // largest t with tile_begin[t] <= g; tile_begin[ntensors] = total > g
  int lo = 0, hi = ntensors;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(tile_begin + mid) <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <bool MULTI>
__device__ __forceinline__ const TensorDesc& desc_of(const EncodeLaunch& a, uint32_t t) {
  if constexpr (MULTI) return a.tensors[t];
  else return a.one;
}

__device__ __forceinline__ void bulk_g2s_plain(void* smem_dst, const void* gmem_src,
                                               uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Thread 0: take the next tile ticket and start filling stage s.
template <bool MULTI>
__device__ __forceinline__ void produce(const EncodeLaunch& a, EncodeShared& sh, uint8_t* stages,
                                        int s, uint64_t pol_stream) {
  const uint32_t ticket = atomicAdd(a.counters + 0, 1u) + a.first_ticket;
  StageMeta m;
  m.tile = ticket;
  m.pad = 0;
  if (ticket >= a.total_tiles) {
    m.tensor = 0;
    m.mode = kModeEnd;
    sh.meta[s] = m;
    return;
  }
  const uint32_t t = MULTI ? static_cast<uint32_t>(find_tensor(a.tile_begin, a.ntensors, ticket)) : 0u;
  const TensorDesc& d = desc_of<MULTI>(a, t);
  const uint64_t base = (uint64_t(ticket) - d.tile_begin) * kEncTile;
  const uint64_t len = d.n - base < uint64_t(kEncTile) ? d.n - base : uint64_t(kEncTile);
  m.tensor = t;
  if (d.bulk_ok && len == uint64_t(kEncTile)) {
    m.mode = kModeBulk;
    uint8_t* st = stages + size_t(s) * kStageBytes;
    mbar_arrive_expect_tx(&sh.bar[s], kStageBytes);
    bulk_g2s(st, d.master + base, kStageMasterBytes, &sh.bar[s], pol_stream);
    // prev is written back soon after, so it keeps the default L2 policy
    bulk_g2s_plain(st + kStageMasterBytes, d.prev + base, kStagePrevBytes, &sh.bar[s]);
  } else {
    m.mode = kModeGeneric;  // tail or unaligned tile: threads load from global
    mbar_arrive(&sh.bar[s]);
  }
  sh.meta[s] = m;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Spin (bounded) until the status word of `tile` is published in this epoch.
// On timeout: record the error and report an inclusive prefix of 0, which
// keeps every later offset at or below the true one (in bounds).
__device__ __forceinline__ uint64_t wait_status(const EncodeLaunch& a, uint64_t tile) {
  const uint64_t* p = a.status + tile;
  uint64_t w = ld_relaxed_u64(p);
  if (status_flag(w, a.epoch) != 0u) return w;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 28); ++it) {
    __nanosleep(40);
    w = ld_relaxed_u64(p);
    if (status_flag(w, a.epoch) != 0u) return w;
    if ((it & 63u) == 63u) {
      if (global_timer_ns() - t0 > a.wait_limit_ns ||
          (ld_volatile_u32(a.counters + 2) & kErrTimeout)) {
        break;
      }
    }
  }
  record_error(a.counters + 2, kErrTimeout);
  return make_status(kFlagPrefix, a.epoch, 0u);
}

// Warp 0: publish this tile's count, find its exclusive prefix within the
// tensor, publish the inclusive prefix.
__device__ __forceinline__ uint32_t look_back(const EncodeLaunch& a, uint64_t g, uint64_t first,
                                              uint32_t agg, int lane) {
  uint64_t* st = a.status;
  if (g == first) {
    if (lane == 0) st_relaxed_u64(st + g, make_status(kFlagPrefix, a.epoch, agg));
    return 0u;
  }
  if (lane == 0) st_relaxed_u64(st + g, make_status(kFlagAggregate, a.epoch, agg));
  uint32_t prefix = 0;
  int64_t pos = int64_t(g) - 1;
  for (;;) {
    // issue all window loads first (one round trip), then wait on any word
    // that is not published yet; tiles before the tensor's first tile read
    // as an inclusive prefix of 0
    uint64_t w[kLookbackPerLane];
#pragma unroll
    for (int q = 0; q < kLookbackPerLane; ++q) {
      const int64_t tile = pos - (lane * kLookbackPerLane + q);
      w[q] = tile >= int64_t(first) ? ld_relaxed_u64(st + tile)
                                    : make_status(kFlagPrefix, a.epoch, 0u);
    }
    uint32_t vals[kLookbackPerLane];
    int first_p = kLookbackPerLane;
#pragma unroll
    for (int q = 0; q < kLookbackPerLane; ++q) {
      if (status_flag(w[q], a.epoch) == 0u)
        w[q] = wait_status(a, uint64_t(pos - (lane * kLookbackPerLane + q)));
      vals[q] = status_value(w[q]);
      if (first_p == kLookbackPerLane && status_flag(w[q], a.epoch) == kFlagPrefix) first_p = q;
    }
    const uint32_t has_p = __ballot_sync(0xFFFFFFFFu, first_p < kLookbackPerLane);
    uint32_t s = 0;
    if (has_p) {
      const int lp = __ffs(has_p) - 1;
#pragma unroll
      for (int q = 0; q < kLookbackPerLane; ++q) {
        if (lane < lp || (lane == lp && q <= first_p)) s += vals[q];
      }
      prefix += warp_sum(s);
      break;
    }
#pragma unroll
    for (int q = 0; q < kLookbackPerLane; ++q) s += vals[q];
    prefix += warp_sum(s);
    pos -= 32 * kLookbackPerLane;
  }
  if (lane == 0) st_relaxed_u64(st + g, make_status(kFlagPrefix, a.epoch, prefix + agg));
  return prefix;
}

template <bool MULTI>
__global__ void __launch_bounds__(kEncThreads) encode_kernel(const __grid_constant__ EncodeLaunch a) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ EncodeShared sh;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 127) & ~uintptr_t(127));
  const uint64_t pol_stream = l2_policy_evict_first();

  if constexpr (MULTI) {
    // tensors with no elements have no tiles: their count is 0
    if (blockIdx.x == 0) {
      for (int t = tid; t < a.ntensors; t += kEncThreads)
        if (a.tensors[t].n == 0) a.counts_out[t] = 0;
    }
  }
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kEncStages; ++s) mbar_init(&sh.bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kEncStages; ++s) produce<MULTI>(a, sh, stages, s, pol_stream);
  }
  __syncthreads();

  uint32_t phase = 0;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kEncStages);
    const StageMeta m = sh.meta[s];
    if (m.mode == kModeEnd) break;
    const TensorDesc& d = desc_of<MULTI>(a, m.tensor);
    const uint64_t first_tile = d.tile_begin;
    const uint64_t base = (uint64_t(m.tile) - first_tile) * kEncTile;
    const uint64_t n = d.n;
    const uint32_t len = uint32_t(n - base < uint64_t(kEncTile) ? n - base : uint64_t(kEncTile));

    if (!mbar_wait_bounded(&sh.bar[s], (phase >> s) & 1u, a.wait_limit_ns)) {
      record_error(a.counters + 2, kErrTimeout);
      mbar_wait_bounded(&sh.bar[s], (phase >> s) & 1u, a.wait_limit_ns);
    }
    phase ^= 1u << s;

    // ---- cast + compare: 4 consecutive elements per thread per round
    uint32_t nb[kEncRounds][2];  // new BF16 values, two per word (low = lower index)
    uint32_t flags = 0;          // bit (j*4 + e): element e of round j changed
    const float4* sm = reinterpret_cast<const float4*>(stages + size_t(s) * kStageBytes);
    const uint2* sp = reinterpret_cast<const uint2*>(stages + size_t(s) * kStageBytes + kStageMasterBytes);
#pragma unroll
    for (int j = 0; j < kEncRounds; ++j) {
      const uint32_t li = uint32_t(j * kEncThreads + tid) * 4u;
      uint32_t mu[4], pu[4];
      bool valid[4];
      if (m.mode == kModeBulk) {
        const float4 mv = sm[j * kEncThreads + tid];
        const uint2 pv = sp[j * kEncThreads + tid];
        mu[0] = __float_as_uint(mv.x); mu[1] = __float_as_uint(mv.y);
        mu[2] = __float_as_uint(mv.z); mu[3] = __float_as_uint(mv.w);
        pu[0] = pv.x & 0xFFFFu; pu[1] = pv.x >> 16; pu[2] = pv.y & 0xFFFFu; pu[3] = pv.y >> 16;
        valid[0] = valid[1] = valid[2] = valid[3] = true;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          valid[e] = li + e < len;
          mu[e] = valid[e] ? __float_as_uint(d.master[base + li + e]) : 0u;
          pu[e] = valid[e] ? uint32_t(d.prev[base + li + e]) : 0u;
        }
      }
      uint32_t b[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        b[e] = bf16_rne_bits(mu[e]);
        if (valid[e] && b[e] != pu[e]) flags |= 1u << (j * 4 + e);
      }
      nb[j][0] = b[0] | (b[1] << 16);
      nb[j][1] = b[2] | (b[3] << 16);
    }
    __syncthreads();  // stage s consumed by every thread
    if (tid == 0) produce<MULTI>(a, sh, stages, s, pol_stream);

    // ---- ranks: within warp by ballots, across (round, warp) by one scan
    uint32_t before[kEncRounds];
#pragma unroll
    for (int j = 0; j < kEncRounds; ++j) {
      uint32_t cnt = 0, bef = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, (flags >> (j * 4 + e)) & 1u);
        cnt += __popc(bal);
        bef += __popc(bal & lanemask_lt());
      }
      before[j] = bef;
      if (lane == 0) sh.pair_count[j * kWarps + warp] = cnt;
    }
    __syncthreads();
    if (warp == 0) {
      const uint32_t c = sh.pair_count[lane];
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      sh.pair_offset[lane] = incl - c;
      const uint32_t agg = __shfl_sync(0xFFFFFFFFu, incl, 31);
      const uint32_t prefix = look_back(a, m.tile, first_tile, agg, lane);
      if (lane == 0) {
        sh.tile_prefix = prefix;
        if (base + len == n) a.counts_out[MULTI ? m.tensor : 0] = uint64_t(prefix) + agg;
      }
    }
    __syncthreads();

    // ---- emit the patch entries and refresh prev
    const uint32_t prefix = sh.tile_prefix;
#pragma unroll
    for (int j = 0; j < kEncRounds; ++j) {
      const uint32_t f = (flags >> (j * 4)) & 0xFu;
      if (f == 0u) continue;
      const uint32_t li = uint32_t(j * kEncThreads + tid) * 4u;
      uint32_t pos = prefix + sh.pair_offset[j * kWarps + warp] + before[j];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if ((f >> e) & 1u) {
          d.idx[pos] = uint32_t(base) + li + uint32_t(e);
          d.val[pos] = uint16_t((nb[j][e >> 1] >> ((e & 1) * 16)) & 0xFFFFu);
          ++pos;
        }
      }
      if (m.mode == kModeBulk) {
        *reinterpret_cast<uint2*>(d.prev + base + li) = make_uint2(nb[j][0], nb[j][1]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if ((f >> e) & 1u) d.prev[base + li + e] = uint16_t((nb[j][e >> 1] >> ((e & 1) * 16)) & 0xFFFFu);
      }
    }
  }

  // The last CTA to finish rewinds the ticket and finish counters for the
  // next launch on this workspace.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t finished = atomicAdd(a.counters + 1, 1u);
    if (finished == gridDim.x - 1) {
      atomicExch(a.counters + 0, 0u);
      atomicExch(a.counters + 1, 0u);
    }
  }
}

template <bool MULTI>
int encode_blocks_per_sm() {
  static int cached = [] {
    cudaFuncSetAttribute(encode_kernel<MULTI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         int(kDynSmem));
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, encode_kernel<MULTI>, kEncThreads,
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
    encode_kernel<true><<<grid, kEncThreads, kDynSmem, stream>>>(a);
  } else {
    encode_blocks_per_sm<false>();
    encode_kernel<false><<<grid, kEncThreads, kDynSmem, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace pulse
