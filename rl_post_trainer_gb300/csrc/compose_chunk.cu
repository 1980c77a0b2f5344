// compose_chunk.cu -- k-way composition of a chain of patches over a whole
// model in one pass: the sidecar that is several versions behind ("Taking
// Reinforcement Learning Cross Datacenter", talk 16:40-17:04) can receive
// ONE patch for all the versions it missed. Patch values are absolute (PULSE
// summary, "1. PULSESync"), so the chain equals one patch: every index any
// version lists, with the value of the latest version that lists it, in
// ascending order.
//
// Each tensor is cut into chunks of kCcChunk positions (the chunk-owned
// apply's chunks and its per-version partition). A CTA takes chunks in
// ticket order:
//  * producer warp: one ticket ahead; reads every version's entry range in
//    the chunk (one lane per version) and asks L2 to prefetch the entries;
//  * 8 compute warps: store each version's entries into a shared-memory
//    image of the chunk with atomicMax on (version + 1) << 16 | value, so the
//    latest version wins whatever the order of the stores (no barrier
//    between versions), and set their bits in a presence bitmap; then each
//    thread owns one 32-bit word of the bitmap: popcount, block scan, and
//    the chunk's entries in ascending order are parked in a ring as
//    (chunk-local index | value << 16);
//  * look-back warp: the chunk's output offset within its tensor by the
//    single-pass decoupled look-back (Merrill & Garland 2016) over one status
//    word per chunk, then copies the parked entries out.
// Work per chunk is proportional to its entries plus 256 bitmap words, not
// to a merge of every pair of inputs.
#include "encode_common.cuh"

namespace pulse {
namespace {

using namespace enc;

// Parked chunks per CTA and chunks resolved per look-back round trip: 8 and 4
// (16 and 2, the other kernels' choice, measured 0.4 % slower here).
#ifndef PULSE_CC_PARKED
#define PULSE_CC_PARKED 8
#endif
#ifndef PULSE_CC_LB_BATCH
#define PULSE_CC_LB_BATCH 4
#endif
constexpr int kCcSlots = PULSE_CC_PARKED;
constexpr int kCcBatch = PULSE_CC_LB_BATCH;
constexpr int kCcWindow = 2;  // look-back words per lane and round trip

constexpr int kCcChunk = kApplyChunk;        // positions per chunk
constexpr int kCcWords = kCcChunk / 32;      // bitmap words, one per compute thread
static_assert(kCcWords == kEncThreads, "one bitmap word per compute thread");
static_assert(kCcChunk <= 0x10000, "chunk-local indices fit the ring entry's low half");
constexpr int kCcStages = 3;                 // chunks prepared ahead by the producer
constexpr int kCcGroup = 1;                  // versions whose entries are loaded together
constexpr int kCcPre = 3;                    // entries per thread and version loaded at once
constexpr int kCcMinBlocks = 3;              // resident CTAs per SM
#ifndef PULSE_CC_LB_SLEEP
#define PULSE_CC_LB_SLEEP 256
#endif
constexpr unsigned kCcLookbackSleepNs = PULSE_CC_LB_SLEEP;  // look-back poll pause
// The image holds one word per position with one pad word after every 32,
// so the 32 positions b of the 32 words that a warp's lanes own fall in 32
// different banks when the lanes read them back.
constexpr int kCcImage = kCcChunk + kCcChunk / 32;
__device__ __forceinline__ uint32_t img_at(uint32_t li) { return li + (li >> 5); }

struct CcMeta {
  uint32_t mode;    // kModeEnd, or kModeBulk for a chunk to compose
  uint32_t ticket;  // global chunk index
  uint32_t tensor;
  uint32_t len;     // positions in the chunk
  uint64_t base;    // tensor-local index of the chunk's first position
  uint64_t first;   // the tensor's first chunk
  uint32_t last;    // 1: last chunk of its tensor
  CcOut out;        // the tensor's output segment
  uint32_t e0[kChainMaxVersions], e1[kChainMaxVersions];
  const uint32_t* idx[kChainMaxVersions];
  const uint16_t* val[kChainMaxVersions];
};

#ifndef PULSE_CC_RING
#define PULSE_CC_RING 8192
#endif
constexpr int kCcRing = PULSE_CC_RING;       // parked entries per CTA (at least one chunk)
static_assert(kCcRing >= kCcChunk, "a whole chunk fits the ring");
constexpr uint32_t kCcRingMask = uint32_t(kCcRing) - 1u;
static_assert((kCcRing & (kCcRing - 1)) == 0, "the ring is a power of two");

struct CcParked {
  uint32_t tile;       // ticket (global chunk index)
  uint32_t tensor;
  uint32_t agg;        // entries of the chunk
  uint32_t last;       // 1: last chunk of its tensor; 2: no more chunks
  uint32_t ring_start;
  uint64_t first;
  uint64_t base;
  CcOut out;           // the tensor's output segment
};

struct __align__(16) CcShared {
  uint64_t full[kCcStages];
  uint64_t empty[kCcStages];
  uint64_t agg_ready[kCcSlots];
  uint64_t slot_free[kCcSlots];
  CcMeta meta[kCcStages];
  CcParked parked[kCcSlots];
  uint32_t warp_tot[2][kWarps];
  uint32_t ring_tail;
  uint32_t bits[kCcWords];
  uint32_t image[kCcImage];   // (version + 1) << 16 | value, 0 = empty; padded, see img_at
  uint32_t ring[kCcRing];
};

// ------------------------------------------------------------ producer warp
__device__ __forceinline__ void cc_producer(const CcArgs& a, CcShared& sh, int lane) {
  // Tickets are taken one ahead and each ticket's tensor is loaded when the
  // ticket arrives, so a chunk's own loads (sizes, segment pointers, entry
  // ranges) go out together: one L2 round trip per chunk.
  uint32_t ticket = 0;
  if (lane == 0) ticket = atomicAdd(a.counters + 0, 1u);
  ticket = __shfl_sync(0xFFFFFFFFu, ticket, 0);
  uint32_t t = ticket < a.total_chunks ? a.chunk_tensor[ticket] : 0u;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kCcStages);
    const bool end = ticket >= a.total_chunks;
    uint32_t next = ticket;
    if (lane == 0 && !end) next = atomicAdd(a.counters + 0, 1u);
    next = __shfl_sync(0xFFFFFFFFu, next, 0);
    if (it >= uint32_t(kCcStages)) {
      const bool ok = helper_wait(&sh.empty[s], ((it / kCcStages) - 1) & 1u, a);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
    }
    CcMeta& m = sh.meta[s];
    if (end) {
      if (lane == 0) {
        m.mode = kModeEnd;
        mbar_arrive(&sh.full[s]);
      }
      break;
    }
    const uint64_t g = ticket;
    const uint64_t n = a.tensors[t].n;
    const uint64_t cb = a.chunk_begin[t];
    const uint64_t ce = a.chunk_begin[t + 1];
    uint32_t e0 = 0, e1 = 0, f1 = 0;
    ChainSeg sg{};
    if (lane < a.nversions) {
      const uint32_t* f = a.first + uint64_t(lane) * a.total_chunks;
      sg = a.segs[size_t(lane) * size_t(a.ntensors) + t];
      e0 = f[g];
      if (g + 1 < a.total_chunks) f1 = f[g + 1];
    }
    const uint32_t t_next = next < a.total_chunks ? a.chunk_tensor[next] : 0u;
    CcOut out{};
    if (lane == 0) out = a.outs[t];
    const uint64_t base = (g - cb) * kCcChunk;
    const bool last = g + 1 >= ce;
    if (lane < a.nversions) {
      const uint64_t cnt = sg.count < n ? sg.count : n;
      e1 = last ? uint32_t(cnt) : f1;
      if (e1 < e0) e1 = e0;
      if (e1 > e0) {
        l2_prefetch_range(sg.idx + e0, uint64_t(e1 - e0) * 4u);
        l2_prefetch_range(sg.val + e0, uint64_t(e1 - e0) * 2u);
      }
      m.e0[lane] = e0;
      m.e1[lane] = e1;
      m.idx[lane] = sg.idx;
      m.val[lane] = sg.val;
    }
    if (lane == 0) {
      m.mode = kModeBulk;
      m.ticket = ticket;
      m.tensor = t;
      m.len = uint32_t(n - base < uint64_t(kCcChunk) ? n - base : uint64_t(kCcChunk));
      m.base = base;
      m.first = cb;
      m.last = last ? 1u : 0u;
      m.out = out;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.full[s]);
    ticket = next;
    t = t_next;
  }
  // the last CTA to finish rewinds the ticket and finish counters
  if (lane == 0) {
    __threadfence();
    const uint32_t finished = atomicAdd(a.counters + 1, 1u);
    if (finished == gridDim.x - 1) {
      atomicExch(a.counters + 0, 0u);
      atomicExch(a.counters + 1, 0u);
    }
  }
}

// ---------------------------------------------------------- look-back warp

// Copy a parked chunk's entries to positions prefix + k of its tensor's
// output. Lane l moves entries l, l + 32, l + 64, ...: the ring reads are
// free of bank conflicts and every store instruction of the warp covers 32
// consecutive positions (four in flight per lane). Positions at or past the
// segment's room are never written.
__device__ __forceinline__ void cc_copy_out(const CcParked& pm, uint32_t prefix,
                                            const uint32_t* ring, int lane) {
  const uint32_t agg = pm.agg;
  const uint32_t base = uint32_t(pm.base);
  uint32_t* const oi = pm.out.idx;
  uint16_t* const ov = pm.out.val;
  const uint64_t cap = pm.out.cap;
  const bool inb = uint64_t(prefix) + agg <= cap;
  uint32_t k = uint32_t(lane);
  if (inb) {
    for (; k + 96u < agg; k += 128u) {
      uint32_t e[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) e[q] = ring[(pm.ring_start + k + 32u * q) & kCcRingMask];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint64_t pos = uint64_t(prefix) + k + 32u * q;
        oi[pos] = base + (e[q] & 0xFFFFu);
        ov[pos] = uint16_t(e[q] >> 16);
      }
    }
  }
  for (; k < agg; k += 32u) {
    const uint32_t ent = ring[(pm.ring_start + k) & kCcRingMask];
    const uint64_t pos = uint64_t(prefix) + k;
    if (pos < cap) {
      oi[pos] = base + (ent & 0xFFFFu);
      ov[pos] = uint16_t(ent >> 16);
    }
  }
}

__device__ __forceinline__ void cc_lookback(const CcArgs& a, CcShared& sh, int lane) {
  for (uint32_t i = 0;;) {
    const bool ok = helper_wait(&sh.agg_ready[i % kCcSlots], (i / kCcSlots) & 1u, a);
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    // how many more chunks are already parked (lane 0 decides)
    int more = 0;
    if (lane == 0) {
      for (int b = 1; b < kCcBatch; ++b) {
        const uint32_t ii = i + uint32_t(b);
        if (!mbar_test_wait(&sh.agg_ready[ii % kCcSlots], (ii / kCcSlots) & 1u)) break;
        more = b;
      }
    }
    more = __shfl_sync(0xFFFFFFFFu, more, 0);
    int nb = 0;
    bool end = false;
    uint64_t win[kCcBatch][kCcWindow];
#pragma unroll
    for (int b = 0; b < kCcBatch; ++b) {
      if (b > more || end) continue;
      const uint32_t ii = i + uint32_t(b);
      const int q = int(ii % kCcSlots);
      if (b > 0) mbar_test_wait(&sh.agg_ready[q], (ii / kCcSlots) & 1u);  // acquire for every lane
      const CcParked& pm = sh.parked[q];
      if (pm.last == 2u) {
        end = true;
        continue;
      }
      if (pm.tile != pm.first)
        load_window<StatusEpoch, CcArgs, kCcWindow>(a, int64_t(pm.tile) - 1, pm.first, lane, win[b]);
      nb = b + 1;
    }
#pragma unroll
    for (int b = 0; b < kCcBatch; ++b) {
      if (b >= nb) continue;
      const uint32_t ii = i + uint32_t(b);
      const int q = int(ii % kCcSlots);
      const CcParked pm = sh.parked[q];
      const uint32_t prefix = resolve_prefix<StatusEpoch, CcArgs, kCcLookbackSleepNs, kCcWindow>(
          a, pm.tile, pm.first, pm.agg, lane, win[b]);
      if (lane == 0 && pm.last == 1u) a.counts_out[pm.tensor] = uint64_t(prefix) + pm.agg;
      cc_copy_out(pm, prefix, sh.ring, lane);
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
__device__ __forceinline__ void cc_compute(const CcArgs& a, CcShared& sh, int tid, int lane,
                                           int warp) {
  uint32_t posted = 0, ring_head = 0;
  bool failed = false;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kCcStages);
    failed |= !wait_or_flag(&sh.full[s], (it / kCcStages) & 1u, a);
    // every exit decision goes through a barrier that ORs it over the compute
    // warps, so they always leave together (no named barrier left short)
    if (compute_barrier_or(failed || sh.meta[s].mode == kModeEnd)) break;
    const CcMeta& m = sh.meta[s];
    const uint32_t g = m.ticket, t = m.tensor, len = m.len, last = m.last;
    const uint64_t base = m.base, first = m.first;
    CcOut out{};
    if (tid == 0) out = m.out;  // read before the slot is released
    // ---- the chain's entries into the image; atomicMax orders the versions
    auto put = [&](uint32_t i, uint16_t v, uint32_t stamp) {
      const uint64_t li = uint64_t(i) - base;  // wraps to a huge value below base
      if (li >= len) {
        record_error(a.counters + 2, kErrIndex);
        return;
      }
      atomicMax(&sh.image[img_at(uint32_t(li))], stamp | v);
      atomicOr(&sh.bits[li >> 5], 1u << (li & 31u));
    };
    for (int v0 = 0; v0 < a.nversions; v0 += kCcGroup) {
      uint32_t pi[kCcGroup][kCcPre];
      uint16_t pv[kCcGroup][kCcPre];
#pragma unroll
      for (int u = 0; u < kCcGroup; ++u) {
        const int v = v0 + u;
        const int vc = v < a.nversions ? v : 0;  // every shared read stays in bounds
        const uint32_t e0 = m.e0[vc];
        const uint32_t e1 = v < a.nversions ? m.e1[vc] : e0;
        const uint32_t* ip = m.idx[vc];
        const uint16_t* vp = m.val[vc];
#pragma unroll
        for (int q = 0; q < kCcPre; ++q) {
          const uint32_t j = e0 + uint32_t(q * kEncThreads + tid);
          pi[u][q] = j < e1 ? ip[j] : 0u;
          pv[u][q] = j < e1 ? vp[j] : uint16_t(0);
        }
      }
#pragma unroll
      for (int u = 0; u < kCcGroup; ++u) {
        const int v = v0 + u;
        if (v >= a.nversions) break;  // uniform
        const uint32_t e0 = m.e0[v], e1 = m.e1[v];
        const uint32_t stamp = uint32_t(v + 1) << 16;
#pragma unroll
        for (int q = 0; q < kCcPre; ++q)
          if (e0 + uint32_t(q * kEncThreads + tid) < e1) put(pi[u][q], pv[u][q], stamp);
        // the rest of a crowded chunk, kCcPre loads in flight per thread
        const uint32_t* ip = m.idx[v];
        const uint16_t* vp = m.val[v];
        for (uint32_t j0 = e0 + uint32_t(kCcPre * kEncThreads); j0 < e1;
             j0 += uint32_t(kCcPre * kEncThreads)) {
          uint32_t xi[kCcPre];
          uint16_t xv[kCcPre];
#pragma unroll
          for (int q = 0; q < kCcPre; ++q) {
            const uint32_t j = j0 + uint32_t(q * kEncThreads + tid);
            xi[q] = j < e1 ? ip[j] : 0u;
            xv[q] = j < e1 ? vp[j] : uint16_t(0);
          }
#pragma unroll
          for (int q = 0; q < kCcPre; ++q)
            if (j0 + uint32_t(q * kEncThreads + tid) < e1) put(xi[q], xv[q], stamp);
        }
      }
    }
    compute_barrier();  // every entry of the chunk is in the image
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);  // the slot is read no more

    // ---- this thread's bitmap word: count and scan
    uint32_t word = sh.bits[tid];
    sh.bits[tid] = 0u;  // cleared for the next chunk (set again only after the last barrier)
    const uint32_t c = uint32_t(__popc(word));
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const int pc = int(it & 1u);
    if (lane == 31) sh.warp_tot[pc][warp] = incl;
    compute_barrier();
    const uint32_t wt = lane < kWarps ? sh.warp_tot[pc][lane] : 0u;
    uint32_t sc = wt;
#pragma unroll
    for (int o = 1; o < kWarps; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, sc, o);
      if (lane >= o) sc += y;
    }
    const uint32_t before = __shfl_sync(0xFFFFFFFFu, sc - wt, warp);  // warps before this one
    const uint32_t agg = __shfl_sync(0xFFFFFFFFu, sc, kWarps - 1);    // the chunk's entries
    if (tid == 0)
      st_relaxed_u64(a.status + g, make_status(uint64_t(g) == first ? kFlagPrefix : kFlagAggregate,
                                               a.epoch, agg));

    // ---- room: the parked slot must be free and the ring must hold agg more
    const int q = int(posted % kCcSlots);
    if (posted >= uint32_t(kCcSlots))
      failed |= !wait_or_flag(&sh.slot_free[q], ((posted - kCcSlots) / kCcSlots) & 1u, a);
    failed |= !wait_ring_room<256>(&sh.ring_tail, ring_head, agg, uint32_t(kCcRing), a);

    // ---- park the chunk's entries in ascending order
    uint32_t r = ring_head + before + (incl - c);
    while (word != 0u) {
      const uint32_t b = uint32_t(__ffs(word)) - 1u;
      word &= word - 1u;
      const uint32_t li = uint32_t(tid) * 32u + b;
      const uint32_t at = img_at(li);
      sh.ring[r & kCcRingMask] = li | (sh.image[at] << 16);  // the stamp shifts out
      sh.image[at] = 0u;  // empty again for the next chunk
      ++r;
    }
    if (tid == 0) {
      CcParked pm;
      pm.tile = g;
      pm.tensor = t;
      pm.agg = agg;
      pm.last = last;
      pm.ring_start = ring_head;
      pm.first = first;
      pm.base = base;
      pm.out = out;
      sh.parked[q] = pm;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.agg_ready[q]);
    ++posted;
    ring_head += agg;
    // the next chunk writes the image only after the barrier at the top of
    // the loop, which every thread reaches after parking this one
  }
  for (uint32_t e = posted > uint32_t(kCcSlots) ? posted - kCcSlots : 0u; e < posted; ++e)
    wait_or_flag(&sh.slot_free[e % kCcSlots], (e / kCcSlots) & 1u, a);
  compute_barrier();
  const int q = int(posted % kCcSlots);
  if (tid == 0) {
    CcParked pm{};
    pm.last = 2u;
    sh.parked[q] = pm;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&sh.agg_ready[q]);
}

__global__ void __launch_bounds__(kEncBlockThreads, kCcMinBlocks)
    compose_chunk_kernel(const __grid_constant__ CcArgs a) {
  // the shared state is addressed through the shared window itself (no
  // integer round trip), so every access stays a shared-memory instruction
  extern __shared__ __align__(16) uint8_t cc_smem[];
  CcShared& sh = *reinterpret_cast<CcShared*>(cc_smem);
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kCcStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kWarps);
      sh.meta[s].mode = kModeEnd;
    }
#pragma unroll
    for (int q = 0; q < kCcSlots; ++q) {
      mbar_init(&sh.agg_ready[q], kWarps);
      mbar_init(&sh.slot_free[q], 1);
      sh.parked[q].last = 2u;
    }
    sh.ring_tail = 0;
    fence_mbar_init();
  }
  for (int k = tid; k < kCcWords; k += kEncBlockThreads) sh.bits[k] = 0u;
  for (int k = tid; k < kCcImage; k += kEncBlockThreads) sh.image[k] = 0u;
  __syncthreads();
  if (warp < kWarps) {
    cc_compute(a, sh, tid, lane, warp);
  } else if (warp == kProducerWarp) {
    cc_producer(a, sh, lane);
  } else if (warp == kFirstLookbackWarp) {
    cc_lookback(a, sh, lane);
  }
}

constexpr size_t kCcSmem = sizeof(CcShared);

int compose_chunk_blocks_per_sm() {
  static int cached = [] {
    cudaFuncSetAttribute(compose_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         int(kCcSmem));
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, compose_chunk_kernel, kEncBlockThreads,
                                                      kCcSmem) != cudaSuccess ||
        b < 1)
      b = 1;
    return b;
  }();
  return cached;
}

}  // namespace

cudaError_t launch_compose_chunks(const CcArgs& a, cudaStream_t stream) {
  if (a.total_chunks == 0) return cudaSuccess;
  if (a.nversions < 1 || a.nversions > kChainMaxVersions) return cudaErrorInvalidValue;
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t cap = uint64_t(sm_count(dev)) * uint64_t(compose_chunk_blocks_per_sm());
  const unsigned grid = unsigned(a.total_chunks < cap ? a.total_chunks : cap);
  compose_chunk_kernel<<<grid, kEncBlockThreads, kCcSmem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pulse
