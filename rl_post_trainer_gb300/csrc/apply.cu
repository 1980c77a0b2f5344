// apply.cu -- sampler-side patch apply: w[idx[j]] = val[j], for 2-byte
// values (the BF16 view) and 1-byte values (the MX views' codes and scales),
// and the chained apply that brings w forward by several versions at once.
//
// "Taking Reinforcement Learning Cross Datacenter", talk 11:08-11:30
// (selective overrides reconstruct the served version bitwise) and the PULSE
// summary, section "Metodologia: PULSE -- 1. PULSESync" (the sampler applies
// the sparse patch of absolute values directly to its BF16 weights).
//
// One version: an entry scatter. The patch is read once as a stream and each
// entry is stored with one 2-byte (or 1-byte) store; consecutive entries sit
// on consecutive lanes, so one warp-wide store holds 32 consecutive entries of
// the ascending patch and L2 merges the entries of one 32-byte sector into one
// request. A store that covers part of a sector makes L2 fetch the sector from
// HBM before it is written back (measured: a scatter of 3.25M entries into a
// 2^28-element array read 6k + 30 bytes per touched sector), so the traffic
// is 6k + 64 S bytes for S touched sectors, the read-modify-write minimum of
// a patch that does not cover whole sectors. Against the alternative of
// reading every touched 8192-element chunk whole into shared memory, the
// scatter measured faster at every density from 0.5 % to 70 % (8.03B-param
// patch at 8 %: 4.78 against 5.05 ms; at 1.2 %: 2.01 against 4.13 ms).
#include "pulse_device.cuh"
#include "pulse_internal.h"

namespace pulse {
namespace {

// The scatter's stores carry the evict-first hint: no sector of w is read
// again in the launch (8 % density, 8.03B step: 4.68 against 4.75 ms).
#ifndef PULSE_APPLY_STREAM_STORES
#define PULSE_APPLY_STREAM_STORES 1
#endif
template <bool CHECKED, class V>
__device__ __forceinline__ void scatter1(V* w, uint64_t n, uint32_t i, uint32_t v, uint32_t* err) {
  if (CHECKED && uint64_t(i) >= n) {
    record_error(err, kErrIndex);
    return;
  }
#if PULSE_APPLY_STREAM_STORES
  __stcs(&w[i], V(v));
#else
  w[i] = V(v);
#endif
}

// Apply entries [0, count) of one segment, tile `tile` of kApplyTile entries.
// Entry base + q * kApplyThreads + threadIdx.x goes to thread threadIdx.x:
// consecutive entries sit on consecutive lanes, so one warp-wide store holds
// 32 consecutive entries of the (ascending) patch and L2 receives one
// request per 32-byte sector they touch.
template <bool CHECKED, class V>
__device__ __forceinline__ void apply_tile(V* w, uint64_t n, const uint32_t* idx, const V* val,
                                           uint64_t count, uint64_t tile, uint32_t* err) {
  const uint64_t base = tile * kApplyTile + threadIdx.x;
  uint32_t ii[kApplyPerThread], vv[kApplyPerThread];
#pragma unroll
  for (int q = 0; q < kApplyPerThread; ++q) {
    const uint64_t j = base + uint64_t(q) * kApplyThreads;
    ii[q] = j < count ? __ldcs(idx + j) : 0u;
    vv[q] = j < count ? uint32_t(val[j]) : 0u;
  }
#pragma unroll
  for (int q = 0; q < kApplyPerThread; ++q)
    if (base + uint64_t(q) * kApplyThreads < count) scatter1<CHECKED>(w, n, ii[q], vv[q], err);
}

template <bool CHECKED, class V>
__global__ void __launch_bounds__(kApplyThreads)
    apply_kernel(V* w, uint64_t n, const uint32_t* idx, const V* val, uint64_t count,
                 uint32_t* err) {
  const uint64_t ntiles = (count + kApplyTile - 1) / kApplyTile;
  for (uint64_t t = blockIdx.x; t < ntiles; t += gridDim.x)
    apply_tile<CHECKED>(w, n, idx, val, count, t, err);
}

// Whole-model apply over segments (a TensorDesc for the BF16 view, a
// ByteSegment for each MXFP8 code or scale array; both name their target w,
// its length n and the patch idx / val). The segment lengths live in device
// memory, so the tile map (tiles per segment, prefix over the segment list)
// is rebuilt by every CTA in shared memory at the start of the launch.
template <class Seg>
__global__ void __launch_bounds__(kApplyThreads)
    apply_multi_kernel(const Seg* segs, int nsegs, const uint64_t* counts, uint32_t* err) {
  extern __shared__ uint64_t tile_begin[];  // nsegs + 1
  __shared__ uint64_t warp_tot[kApplyThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (nsegs + kApplyThreads - 1) / kApplyThreads;
  const int t0 = tid * per;
  uint64_t mine = 0;
  for (int t = t0; t < t0 + per && t < nsegs; ++t) {
    uint64_t c = counts[t];
    if (c > segs[t].n) c = segs[t].n;  // a segment never exceeds its target
    mine += (c + kApplyTile - 1) / kApplyTile;
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
  for (int t = t0; t < t0 + per && t < nsegs; ++t) {
    tile_begin[t] = run;
    uint64_t c = counts[t];
    if (c > segs[t].n) c = segs[t].n;
    run += (c + kApplyTile - 1) / kApplyTile;
  }
  if (tid == kApplyThreads - 1) tile_begin[nsegs] = warp_off + incl;
  __syncthreads();
  if (tid == 0) {
    for (int t = 0; t < nsegs; ++t)
      if (counts[t] > segs[t].n) record_error(err, kErrIndex);
  }

  const uint64_t total = tile_begin[nsegs];
  for (uint64_t g = blockIdx.x; g < total; g += gridDim.x) {
    int lo = 0, hi = nsegs;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_begin[mid] <= g) lo = mid; else hi = mid - 1;
    }
    const Seg& d = segs[lo];
    uint64_t c = counts[lo];
    if (c > d.n) c = d.n;
    apply_tile<true>(d.w, d.n, d.idx, d.val, c, g - tile_begin[lo], err);
  }
}

template <class V>
cudaError_t launch_apply_t(V* w, uint64_t n, bool checked, const uint32_t* idx, const V* val,
                           uint64_t count, uint32_t* error_word, cudaStream_t stream) {
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t ntiles = (count + kApplyTile - 1) / kApplyTile;
  const uint64_t cap = uint64_t(sm_count(dev)) * 8u;
  const int grid = int(ntiles < cap ? ntiles : cap);
  if (grid == 0) return cudaSuccess;
  if (checked)
    apply_kernel<true, V><<<grid, kApplyThreads, 0, stream>>>(w, n, idx, val, count, error_word);
  else
    apply_kernel<false, V><<<grid, kApplyThreads, 0, stream>>>(w, n, idx, val, count, error_word);
  return cudaGetLastError();
}

template <class Seg>
cudaError_t launch_apply_multi_t(const Seg* segs, int nsegs, const uint64_t* counts_dev,
                                 uint32_t* error_word, int grid, cudaStream_t stream) {
  const size_t smem = size_t(nsegs + 1) * sizeof(uint64_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(apply_multi_kernel<Seg>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
  }
  apply_multi_kernel<Seg><<<grid, kApplyThreads, smem, stream>>>(segs, nsegs, counts_dev,
                                                                 error_word);
  return cudaGetLastError();
}

// ------------------------------------------------------------ chained apply
// A receiver that is several versions behind applies the patches of versions
// v0 < v1 < ... in order (talk 16:40-17:04, the sidecar catching up). Each
// patch lists absolute values, so applying them in order equals applying
// their composition once; the chained form gets there without composing:
// one pass over w in which every chunk of kChunk elements is loaded once,
// receives the entries of every version in version order (a barrier of the
// storing warps between versions: the later patch wins) and writes its
// changed sectors back once. A partition kernel finds each chunk's first
// entry in every version's (ascending) segment. Entries outside their chunk
// (a segment that is not ascending, or an index past the tensor) are skipped
// and reported as PULSE_ERR_INDEX.
constexpr int kChunk = kApplyChunk;                 // elements per chunk (16 KB of BF16)
constexpr int kChunkSectors = kChunk * 2 / 32;      // 512
constexpr uint32_t kDenseMin = kApplyDenseMin;      // entries from which a chunk goes dense

__device__ __forceinline__ uint32_t lower_bound_u32(const uint32_t* a, uint32_t n, uint32_t key) {
  uint32_t lo = 0, hi = n;
  while (lo < hi) {
    const uint32_t mid = (lo + hi) >> 1;
    if (a[mid] < key) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(256)
    chain_partition_kernel(const TensorDesc* tensors, const uint64_t* chunk_begin,
                           const uint32_t* chunk_tensor, const ChainSeg* segs, int ntensors,
                           int nversions, uint64_t total_chunks, uint32_t* chain_first,
                           uint32_t* err) {
  const uint64_t x = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (x >= total_chunks * uint64_t(nversions)) return;
  const uint32_t v = uint32_t(x / total_chunks);
  const uint64_t g = x - uint64_t(v) * total_chunks;
  const uint32_t t = chunk_tensor[g];
  const ChainSeg s = segs[size_t(v) * size_t(ntensors) + t];
  uint64_t c = s.count;
  if (c > tensors[t].n) {
    if (g == chunk_begin[t]) record_error(err, kErrIndex);  // once per tensor and version
    c = tensors[t].n;
  }
  const uint64_t start = (g - chunk_begin[t]) * kChunk;
  chain_first[x] = lower_bound_u32(s.idx, uint32_t(c), uint32_t(start));
}

// ------------------------------------------------ chunk-owned apply kernel
// The chained apply (1..kChainMaxVersions versions). Warp roles per CTA:
//  * producer warp: for the CTA's next chunk, reads the entry range of every
//    version (from the partition), asks L2 to prefetch those entries, writes
//    the chunk's description into the buffer's shared slot and, when the
//    chunk goes dense, bulk-copies its w into the buffer; it runs up to
//    BUF chunks ahead of the workers (full / empty mbarriers per buffer),
//    so none of this sits on the workers' path;
//  * 8 worker warps: per chunk, for each version in order, load the entries
//    (kCwPre per thread and version in flight at once, for kCwGroup
//    versions) and store them into the shared copy of the chunk (flagging
//    the changed 32-byte sectors) or, for a sparse chunk, straight to w; a
//    named barrier between versions makes the later patch win; then write
//    the changed sectors back whole.
constexpr int kCwWorkers = 256;                    // 8 worker warps
constexpr int kCwThreads = kCwWorkers + 32;        // + the producer warp
constexpr int kCwBarrier = 1;                      // the workers' named barrier
constexpr uint32_t kModeNone = 0, kModeDirect = 1, kModeDense = 2, kModeEnd = 3;

struct ChunkSlot {
  uint16_t* w;     // the chunk's first element
  uint64_t base;   // tensor-local index of that element
  uint32_t len;    // elements in the chunk
  uint32_t mode;
  uint32_t e0[kChainMaxVersions], e1[kChainMaxVersions];
  const uint32_t* idx[kChainMaxVersions];
  const uint16_t* val[kChainMaxVersions];
};

// Where the segment of version v of tensor t comes from.
struct CwArgs {
  const TensorDesc* tensors;
  const uint64_t* chunk_begin;
  const uint32_t* chunk_tensor;
  const uint32_t* first;   // nversions x total_chunks: first entry of each chunk
  const ChainSeg* segs;    // nversions x ntensors, version-major
  int ntensors;
  int nversions;
  uint64_t total_chunks;
  uint32_t* err;
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ void worker_barrier() {
  asm volatile("bar.sync %0, %1;" ::"n"(kCwBarrier), "n"(kCwWorkers) : "memory");
}

// Named barrier of the workers that also ORs a predicate over them (every
// loop exit goes through it, so the workers always leave together).
__device__ __forceinline__ bool worker_barrier_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(v)), "n"(kCwBarrier), "n"(kCwWorkers)
      : "memory");
  return r != 0;
}

// Bounded wait that gives up at once when another wait of the launch has
// given up (the error word holds kErrTimeout).
__device__ __forceinline__ bool cw_wait(uint64_t* bar, uint32_t parity, const CwArgs& a) {
#pragma unroll 1
  for (int i = 0; i < 4; ++i)
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  if (ld_volatile_u32(a.err) & kErrTimeout) return false;
  if (mbar_wait_bounded(bar, parity, a.wait_limit_ns)) return true;
  record_error(a.err, kErrTimeout);
  return false;
}

// GROUP: versions whose entries are in flight together; PRE: entries per
// thread and version loaded at once; CTAS: resident CTAs per SM; BUF: chunks
// of w staged per CTA (dynamic shared memory, BUF x 16 KB).
template <int GROUP, int PRE, int CTAS, int BUF>
__global__ void __launch_bounds__(kCwThreads, CTAS) chunk_apply_kernel(const CwArgs a) {
  constexpr int kCwGroup = GROUP, kCwPre = PRE, kCwBuf = BUF;
  extern __shared__ __align__(128) uint16_t cw_dyn[];
  uint16_t(*const wsm)[kChunk] = reinterpret_cast<uint16_t(*)[kChunk]>(cw_dyn);
  __shared__ __align__(16) uint8_t dirty[kChunkSectors];  // one flag byte per 32-byte sector
  __shared__ ChunkSlot slot[kCwBuf];
  __shared__ __align__(8) uint64_t full[kCwBuf], empty[kCwBuf];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int b = 0; b < kCwBuf; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], 1);
    }
    fence_mbar_init();
  }
  for (int k = tid; k < kChunkSectors; k += kCwThreads) dirty[k] = 0u;
  __syncthreads();

  if (warp == kCwWorkers / 32) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_policy_evict_first();
    // lane 0: 1 + round of buffer b's latest phase when a bulk copy completes
    // it, else 0 (a parity wait is only meaningful for the latest phase)
    uint32_t armed[kCwBuf] = {};
    for (uint32_t i = 0;; ++i) {
      const int b = int(i % kCwBuf);
      const uint32_t round = i / kCwBuf;
      if (round > 0 && !cw_wait(&empty[b], (round - 1) & 1u, a)) break;
      const uint64_t g = blockIdx.x + uint64_t(i) * gridDim.x;
      ChunkSlot& sl = slot[b];
      // a new phase on buffer b follows the workers' release of its last one,
      // so an earlier bulk copy into b has landed
      armed[b] = 0;
      if (g >= a.total_chunks) {
        if (lane == 0) {
          sl.mode = kModeEnd;
          mbar_arrive(&full[b]);
        }
        break;
      }
      const uint32_t t = a.chunk_tensor[g];
      const TensorDesc& d = a.tensors[t];
      const uint64_t n = d.n;
      const uint64_t base = (g - a.chunk_begin[t]) * kChunk;
      const uint32_t len = uint32_t(n - base < uint64_t(kChunk) ? n - base : uint64_t(kChunk));
      const bool last_of_tensor = g + 1 >= a.chunk_begin[t + 1];
      uint32_t e0 = 0, e1 = 0;
      if (lane < a.nversions) {
        const ChainSeg sg = a.segs[size_t(lane) * size_t(a.ntensors) + t];
        const uint32_t* ip = sg.idx;
        const uint16_t* vp = sg.val;
        uint64_t cnt = sg.count;
        if (cnt > n) cnt = n;
        const uint32_t* f = a.first + uint64_t(lane) * a.total_chunks;
        e0 = f[g];
        e1 = last_of_tensor ? uint32_t(cnt) : f[g + 1];
        if (e1 < e0) e1 = e0;
        if (e1 > e0) {
          l2_prefetch_range(ip + e0, uint64_t(e1 - e0) * 4u);
          l2_prefetch_range(vp + e0, uint64_t(e1 - e0) * 2u);
        }
        sl.e0[lane] = e0;
        sl.e1[lane] = e1;
        sl.idx[lane] = ip;
        sl.val[lane] = vp;
      }
      const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, e1 - e0);
      const bool dense = total >= kDenseMin && (reinterpret_cast<uintptr_t>(d.w) % 16u == 0);
      const uint32_t body = len & ~7u;
      if (dense && lane < int(len - body)) wsm[b][body + lane] = d.w[base + body + lane];
      if (lane == 0) {
        sl.w = d.w + base;
        sl.base = base;
        sl.len = len;
        sl.mode = total == 0 ? kModeNone : (dense ? kModeDense : kModeDirect);
      }
      __syncwarp();  // every lane's slot and tail writes precede the arrival
      if (lane == 0) {
        if (dense && body > 0) {
          mbar_arrive_expect_tx(&full[b], body * 2u);
          bulk_g2s(wsm[b], d.w + base, body * 2u, &full[b], pol);
          armed[b] = round + 1;
        } else {
          mbar_arrive(&full[b]);
        }
      }
    }
    // no bulk copy may still be writing shared memory when the CTA exits
    // (normally the workers have waited for every one; this matters only
    // when a wait gave up)
    if (lane == 0)
      for (int b = 0; b < kCwBuf; ++b)
        if (armed[b] != 0 && !mbar_wait_bounded(&full[b], (armed[b] - 1) & 1u, a.wait_limit_ns))
          record_error(a.err, kErrTimeout);
    return;
  }

  // --------------------------------------------------------------- workers
  for (uint32_t i = 0;; ++i) {
    const int b = int(i % kCwBuf);
    const uint32_t round = i / kCwBuf;
    const bool ok = cw_wait(&full[b], round & 1u, a);
    if (worker_barrier_or(!ok)) break;
    const ChunkSlot& sl = slot[b];
    const uint32_t m = sl.mode;
    if (m == kModeEnd) break;
    if (m != kModeNone) {
      const bool dense = m == kModeDense;
      uint16_t* w = sl.w;
      const uint64_t base = sl.base;
      const uint32_t len = sl.len;
      auto put = [&](uint32_t i, uint16_t v) {
        const uint64_t li = uint64_t(i) - base;  // wraps to a huge value below base
        if (li >= len) {
          record_error(a.err, kErrIndex);
          return;
        }
        if (dense) {
          wsm[b][li] = v;
          dirty[li >> 4] = 1u;
        } else {
          w[li] = v;
        }
      };
      for (int v0 = 0; v0 < a.nversions; v0 += kCwGroup) {
        uint32_t pi[kCwGroup][kCwPre];
        uint16_t pv[kCwGroup][kCwPre];
#pragma unroll
        for (int u = 0; u < kCwGroup; ++u) {
          const int v = v0 + u;
          const int vc = v < a.nversions ? v : 0;  // every shared read stays in bounds
          const uint32_t e0 = sl.e0[vc];
          const uint32_t e1 = v < a.nversions ? sl.e1[vc] : e0;
          const uint32_t* ip = sl.idx[vc];
          const uint16_t* vp = sl.val[vc];
#pragma unroll
          for (int q = 0; q < kCwPre; ++q) {
            const uint32_t j = e0 + uint32_t(q * kCwWorkers + tid);
            pi[u][q] = j < e1 ? ip[j] : 0u;
            pv[u][q] = j < e1 ? vp[j] : uint16_t(0);
          }
        }
#pragma unroll
        for (int u = 0; u < kCwGroup; ++u) {
          const int v = v0 + u;
          if (v >= a.nversions) break;  // uniform
          const uint32_t e0 = sl.e0[v], e1 = sl.e1[v];
#pragma unroll
          for (int q = 0; q < kCwPre; ++q)
            if (e0 + uint32_t(q * kCwWorkers + tid) < e1) put(pi[u][q], pv[u][q]);
          // the rest of a crowded chunk, kCwPre loads in flight per thread
          const uint32_t* ip = sl.idx[v];
          const uint16_t* vp = sl.val[v];
          for (uint32_t j0 = e0 + uint32_t(kCwPre * kCwWorkers); j0 < e1;
               j0 += uint32_t(kCwPre * kCwWorkers)) {
            uint32_t xi[kCwPre];
            uint16_t xv[kCwPre];
#pragma unroll
            for (int q = 0; q < kCwPre; ++q) {
              const uint32_t j = j0 + uint32_t(q * kCwWorkers + tid);
              xi[q] = j < e1 ? ip[j] : 0u;
              xv[q] = j < e1 ? vp[j] : uint16_t(0);
            }
#pragma unroll
            for (int q = 0; q < kCwPre; ++q)
              if (j0 + uint32_t(q * kCwWorkers + tid) < e1) put(xi[q], xv[q]);
          }
          worker_barrier();  // the next version's stores land after these
        }
      }
      if (dense) {
        // changed sectors back whole (two 16-byte stores each), flags cleared
        for (uint32_t sct = tid; sct < uint32_t(kChunkSectors); sct += kCwWorkers) {
          if (!dirty[sct]) continue;
          dirty[sct] = 0u;
          const uint32_t f = sct * 16u;
          if (f + 16u <= len) {
            const uint4* src = reinterpret_cast<const uint4*>(wsm[b] + f);
            uint4* dst = reinterpret_cast<uint4*>(w + f);
            dst[0] = src[0];
            dst[1] = src[1];
          } else {
            for (uint32_t k = f; k < len; ++k) w[k] = wsm[b][k];
          }
        }
        // the buffer is next written by a bulk copy: order this thread's
        // shared-memory accesses before it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
    }
    worker_barrier();  // buffer b, its slot and the flags are free again
    if (tid == 0) mbar_arrive(&empty[b]);
  }
}

// Chained apply: with the entries of four versions loaded per chunk, two
// chunk buffers at four CTAs per SM measured best (a sweep of buffers per CTA
// against CTAs per SM; the depth of w's bulk copies in flight per SM is what
// matters).
#ifndef PULSE_CW_CTAS_CHAIN
#define PULSE_CW_CTAS_CHAIN 4
#endif
#ifndef PULSE_CW_BUF_CHAIN
#define PULSE_CW_BUF_CHAIN 2
#endif
constexpr int kCwBufChain = PULSE_CW_BUF_CHAIN;
constexpr int kCwGroupChain = 2, kCwPreChain = 3, kCwCtasChain = PULSE_CW_CTAS_CHAIN;

// Resident CTAs per SM of a persistent kernel with `dyn` bytes of dynamic
// shared memory, so that every CTA of the grid is resident from the start.
template <class K>
int resident_per_sm(K kernel, int threads, int cap, size_t dyn) {
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(dyn));
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, threads, dyn) != cudaSuccess || b < 1)
    b = 1;
  return b < cap ? b : cap;
}

constexpr size_t cw_smem(int buf) { return size_t(buf) * size_t(kChunk) * sizeof(uint16_t); }

}  // namespace

cudaError_t launch_chain_partition(const TensorDesc* tensors, const uint64_t* chunk_begin,
                                   const uint32_t* chunk_tensor, const ChainSeg* segs,
                                   int ntensors, int nversions, uint64_t total_chunks,
                                   uint32_t* chain_first, uint32_t* error_word,
                                   cudaStream_t stream) {
  const uint64_t parts = total_chunks * uint64_t(nversions);
  if (parts == 0) return cudaSuccess;
  chain_partition_kernel<<<unsigned((parts + 255) / 256), 256, 0, stream>>>(
      tensors, chunk_begin, chunk_tensor, segs, ntensors, nversions, total_chunks, chain_first,
      error_word);
  return cudaGetLastError();
}

cudaError_t launch_apply_chain(const TensorDesc* tensors, const uint64_t* chunk_begin,
                               const uint32_t* chunk_tensor, uint32_t* chain_first,
                               const ChainSeg* segs, int ntensors, int nversions,
                               uint64_t total_chunks, uint32_t* error_word, uint64_t wait_limit_ns,
                               cudaStream_t stream) {
  if (total_chunks == 0 || nversions < 1) return cudaSuccess;
  if (nversions > kChainMaxVersions) return cudaErrorInvalidValue;
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t parts = total_chunks * uint64_t(nversions);
  chain_partition_kernel<<<unsigned((parts + 255) / 256), 256, 0, stream>>>(
      tensors, chunk_begin, chunk_tensor, segs, ntensors, nversions, total_chunks, chain_first,
      error_word);
  auto kernel = chunk_apply_kernel<kCwGroupChain, kCwPreChain, kCwCtasChain, kCwBufChain>;
  static const int per_sm =
      resident_per_sm(kernel, kCwThreads, kCwCtasChain, cw_smem(kCwBufChain));
  const uint64_t cap = uint64_t(sm_count(dev)) * uint64_t(per_sm);
  const unsigned grid = unsigned(total_chunks < cap ? total_chunks : cap);
  const CwArgs args{tensors,   chunk_begin,  chunk_tensor, chain_first,  segs,
                    ntensors,  nversions,    total_chunks, error_word,   wait_limit_ns};
  kernel<<<grid, kCwThreads, cw_smem(kCwBufChain), stream>>>(args);
  return cudaGetLastError();
}

cudaError_t launch_apply(uint16_t* w, uint64_t n, bool checked, const uint32_t* idx,
                         const uint16_t* val, uint64_t count, uint32_t* error_word,
                         cudaStream_t stream) {
  return launch_apply_t(w, n, checked, idx, val, count, error_word, stream);
}

cudaError_t launch_apply_u8(uint8_t* w, uint64_t n, bool checked, const uint32_t* idx,
                            const uint8_t* val, uint64_t count, uint32_t* error_word,
                            cudaStream_t stream) {
  return launch_apply_t(w, n, checked, idx, val, count, error_word, stream);
}

cudaError_t launch_apply_multi(const TensorDesc* tensors, int ntensors, const uint64_t* counts_dev,
                               uint32_t* error_word, int grid, cudaStream_t stream) {
  return launch_apply_multi_t(tensors, ntensors, counts_dev, error_word, grid, stream);
}

cudaError_t launch_apply_u8_multi(const ByteSegment* segs, int nsegs, const uint64_t* counts_dev,
                                  uint32_t* error_word, int grid, cudaStream_t stream) {
  return launch_apply_multi_t(segs, nsegs, counts_dev, error_word, grid, stream);
}

}  // namespace pulse
