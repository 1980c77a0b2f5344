// apply.cu -- sampler-side patch apply: w[idx[j]] = val[j], for 2-byte
// values (the BF16 view) and 1-byte values (the MXFP8 view's codes and
// scales).
//
// "Taking Reinforcement Learning Cross Datacenter", talk 11:08-11:30
// (selective overrides reconstruct the served version bitwise) and the PULSE
// summary, section "Metodologia: PULSE -- 1. PULSESync" (the sampler applies
// the sparse patch of absolute values directly to its BF16 weights).
//
// The patch is read once as a stream (128-bit index loads, 64-bit value
// loads, evict-first) and scattered with 2-byte stores; an encode patch is in
// ascending index order, so one warp's stores land in a narrow window of w
// and L2 merges them into whole sectors before they reach HBM. A 2-byte
// store covers only part of a 32-byte sector, so L2 must fetch the rest of
// the sector from HBM; the kernel first prefetches every target sector of
// its entries into L2 (prefetch.global.L2) and only then stores, so those
// fetches run as many parallel reads instead of write-miss fills (measured
// on the 8B-parameter patch: 9.46 ms -> 6.69 ms).
#include "pulse_device.cuh"
#include "pulse_internal.h"

namespace pulse {
namespace {

constexpr int kGroups = kApplyPerThread / 4;  // 4-entry groups per thread per tile

// Four consecutive patch values in one streaming load.
template <class V>
struct Vals4;
template <>
struct Vals4<uint16_t> {
  static constexpr uintptr_t kAlign = 8;
  static __device__ __forceinline__ void load(const uint16_t* p, uint32_t (&v)[4]) {
    const uint2 x = ld_stream_u2_ro(p);
    v[0] = x.x & 0xFFFFu;
    v[1] = x.x >> 16;
    v[2] = x.y & 0xFFFFu;
    v[3] = x.y >> 16;
  }
};
template <>
struct Vals4<uint8_t> {
  static constexpr uintptr_t kAlign = 4;
  static __device__ __forceinline__ void load(const uint8_t* p, uint32_t (&v)[4]) {
    const uint32_t x = ld_stream_u1_ro(p);
    v[0] = x & 0xFFu;
    v[1] = (x >> 8) & 0xFFu;
    v[2] = (x >> 16) & 0xFFu;
    v[3] = x >> 24;
  }
};

template <class V>
__device__ __forceinline__ bool vec_ok(const uint32_t* idx, const V* val) {
  return (reinterpret_cast<uintptr_t>(idx) % 16u == 0) &&
         (reinterpret_cast<uintptr_t>(val) % Vals4<V>::kAlign == 0);
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

template <bool CHECKED, class V>
__device__ __forceinline__ void prefetch1(const V* w, uint64_t n, uint32_t i) {
  if (!CHECKED || uint64_t(i) < n) prefetch_l2(w + i);
}

template <bool CHECKED, class V>
__device__ __forceinline__ void scatter1(V* w, uint64_t n, uint32_t i, uint32_t v, uint32_t* err) {
  if (CHECKED && uint64_t(i) >= n) {
    record_error(err, kErrIndex);
    return;
  }
  w[i] = V(v);
}

// Apply entries [0, count) of one segment, tile `tile` of kApplyTile entries.
template <bool CHECKED, class V>
__device__ __forceinline__ void apply_tile(V* w, uint64_t n, const uint32_t* idx, const V* val,
                                           uint64_t count, uint64_t tile, bool vec, uint32_t* err) {
  const int tid = threadIdx.x;
  const uint64_t base = tile * kApplyTile;
  if (vec && base + kApplyTile <= count) {
    uint4 iv[kGroups];
    uint32_t vv[kGroups][4];
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      const uint64_t off = base + uint64_t(g * kApplyThreads + tid) * 4u;
      iv[g] = ld_stream_u4_ro(idx + off);
      Vals4<V>::load(val + off, vv[g]);
    }
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      prefetch1<CHECKED>(w, n, iv[g].x);
      prefetch1<CHECKED>(w, n, iv[g].y);
      prefetch1<CHECKED>(w, n, iv[g].z);
      prefetch1<CHECKED>(w, n, iv[g].w);
    }
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      scatter1<CHECKED>(w, n, iv[g].x, vv[g][0], err);
      scatter1<CHECKED>(w, n, iv[g].y, vv[g][1], err);
      scatter1<CHECKED>(w, n, iv[g].z, vv[g][2], err);
      scatter1<CHECKED>(w, n, iv[g].w, vv[g][3], err);
    }
  } else {
    uint32_t ii[kApplyPerThread];
#pragma unroll
    for (int k = 0; k < kApplyPerThread; ++k) {
      const uint64_t j = base + uint64_t(k) * kApplyThreads + tid;
      ii[k] = j < count ? idx[j] : 0u;
      if (j < count) prefetch1<CHECKED>(w, n, ii[k]);
    }
#pragma unroll
    for (int k = 0; k < kApplyPerThread; ++k) {
      const uint64_t j = base + uint64_t(k) * kApplyThreads + tid;
      if (j < count) scatter1<CHECKED>(w, n, ii[k], uint32_t(val[j]), err);
    }
  }
}

template <bool CHECKED, class V>
__global__ void __launch_bounds__(kApplyThreads)
    apply_kernel(V* w, uint64_t n, const uint32_t* idx, const V* val, uint64_t count,
                 uint32_t* err) {
  const uint64_t ntiles = (count + kApplyTile - 1) / kApplyTile;
  const bool vec = vec_ok(idx, val);
  for (uint64_t t = blockIdx.x; t < ntiles; t += gridDim.x)
    apply_tile<CHECKED>(w, n, idx, val, count, t, vec, err);
}

// Whole-model apply over segments (a TensorDesc for the BF16 view, a
// ByteSegment for each MXFP8 code or scale array; both name their target w,
// its length n and the patch idx / val). The segment lengths live in device
// memory, so the tile map (tiles per segment, prefix over the segment list)
// is rebuilt by every CTA in shared memory at the start of the launch.
template <class Seg>
__global__ void __launch_bounds__(kApplyThreads)
    apply_multi_kernel(const Seg* segs, int nsegs, const uint64_t* counts, uint32_t* err,
                       const uint32_t* run_if) {
  extern __shared__ uint64_t tile_begin[];  // nsegs + 1
  __shared__ uint64_t warp_tot[kApplyThreads / 32];
  if (run_if != nullptr && *run_if == 0u) return;  // the other route takes this patch
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
    apply_tile<true>(d.w, d.n, d.idx, d.val, c, g - tile_begin[lo], vec_ok(d.idx, d.val), err);
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
                                 uint32_t* error_word, int grid, cudaStream_t stream,
                                 const uint32_t* run_if) {
  const size_t smem = size_t(nsegs + 1) * sizeof(uint64_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(apply_multi_kernel<Seg>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
  }
  apply_multi_kernel<Seg><<<grid, kApplyThreads, smem, stream>>>(segs, nsegs, counts_dev, error_word,
                                                                 run_if);
  return cudaGetLastError();
}

// ------------------------------------------------------ chunk-owned apply
// Whole-model BF16 apply for ascending patch segments (what encode writes).
// Each tensor is cut into chunks of kChunk elements; a partition kernel finds
// each chunk's first patch entry (lower bound of the chunk's start). One CTA
// owns a chunk at a time: with many entries it bulk-copies the chunk of w
// into shared memory, scatters the entries there, flags the 32-byte sectors
// it changed and writes exactly those sectors back with full 16-byte stores
// (no partial-sector writes reach L2); with few entries it stores them
// directly. Entries outside their chunk (a patch that is not ascending, or
// an index past the tensor) are skipped and reported as PULSE_ERR_INDEX.
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

// One CTA: the route of a whole-model apply (1 = entry scatter for a sparse
// patch, 0 = chunk-owned). Both routes give the same w for an ascending patch.
__global__ void __launch_bounds__(256)
    apply_route_kernel(const TensorDesc* tensors, int ntensors, const uint64_t* counts,
                       uint64_t total_n, uint32_t* route) {
  __shared__ uint64_t part[256 / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t k = 0;
  for (int t = tid; t < ntensors; t += 256) {
    const uint64_t c = counts[t], n = tensors[t].n;
    k += c < n ? c : n;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) k += __shfl_xor_sync(0xFFFFFFFFu, k, o);
  if (lane == 0) part[warp] = k;
  __syncthreads();
  if (tid == 0) {
    uint64_t sum = 0;
    for (int w = 0; w < 256 / 32; ++w) sum += part[w];
    *route = kApplySparseRatio * sum < total_n ? 1u : 0u;
  }
}

__global__ void __launch_bounds__(256)
    apply_partition_kernel(const TensorDesc* tensors, const uint64_t* chunk_begin,
                           const uint32_t* chunk_tensor, const uint64_t* counts,
                           uint64_t total_chunks, uint32_t* chunk_first, uint32_t* err,
                           const uint32_t* skip_if) {
  const uint64_t g = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= total_chunks) return;
  if (skip_if != nullptr && *skip_if != 0u) return;  // the sparse route takes this patch
  const uint32_t t = chunk_tensor[g];
  const TensorDesc& d = tensors[t];
  uint64_t c = counts[t];
  if (c > d.n) {
    if (g == chunk_begin[t]) record_error(err, kErrIndex);  // once per tensor
    c = d.n;
  }
  const uint64_t start = (g - chunk_begin[t]) * kChunk;
  chunk_first[g] = lower_bound_u32(d.idx, uint32_t(c), uint32_t(start));
}

// ------------------------------------------------------------ chained apply
// A receiver that is several versions behind applies the patches of versions
// v0 < v1 < ... in order (talk 16:40-17:04, the sidecar catching up). Each
// patch lists absolute values, so applying them in order equals applying
// their composition once; the chained form gets there without composing:
// one pass over w in which every chunk is loaded once, receives the entries
// of every version in version order (a barrier of the storing warps between
// versions: the later patch wins) and writes its changed sectors back once.
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
// One kernel serves the whole-model apply (one version, counts on the
// device) and the chained apply (1..kChainMaxVersions versions). Warp
// roles per CTA:
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
  const ChainSeg* segs;    // chained: nversions x ntensors; else null
  const uint64_t* counts;  // whole-model apply: device counts; else null
  int ntensors;
  int nversions;
  uint64_t total_chunks;
  uint32_t* err;
  uint64_t wait_limit_ns;
  const uint32_t* skip_if;  // null, or a device word: the launch does nothing when it is non-zero
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
  // the same word for every thread, written by an earlier launch: a uniform exit
  if (a.skip_if != nullptr && *a.skip_if != 0u) return;
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
        const uint32_t* ip;
        const uint16_t* vp;
        uint64_t cnt;
        if (a.segs != nullptr) {
          const ChainSeg sg = a.segs[size_t(lane) * size_t(a.ntensors) + t];
          ip = sg.idx;
          vp = sg.val;
          cnt = sg.count;
        } else {
          ip = d.idx;
          vp = d.val;
          cnt = a.counts[t];
        }
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

// whole-model apply (one version) and chained apply (up to 16 versions).
// One version: three chunk buffers at three CTAs per SM keep more of w's
// bulk copies in flight than two at five (8.03B step: 4.99 against 5.53 ms);
// the chained form, with four versions' entry loads per chunk, measured best
// at two buffers and four CTAs.
#ifndef PULSE_CW_PRE_ONE
#define PULSE_CW_PRE_ONE 4
#endif
#ifndef PULSE_CW_CTAS_ONE
#define PULSE_CW_CTAS_ONE 3
#endif
#ifndef PULSE_CW_CTAS_CHAIN
#define PULSE_CW_CTAS_CHAIN 4
#endif
#ifndef PULSE_CW_BUF_ONE
#define PULSE_CW_BUF_ONE 3
#endif
#ifndef PULSE_CW_BUF_CHAIN
#define PULSE_CW_BUF_CHAIN 2
#endif
constexpr int kCwPreOne = PULSE_CW_PRE_ONE, kCwCtasOne = PULSE_CW_CTAS_ONE;
constexpr int kCwBufOne = PULSE_CW_BUF_ONE, kCwBufChain = PULSE_CW_BUF_CHAIN;
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

cudaError_t launch_apply_chunks(const TensorDesc* tensors, int ntensors, uint64_t total_n,
                                const uint64_t* chunk_begin, const uint32_t* chunk_tensor,
                                uint32_t* chunk_first, const uint64_t* counts_dev,
                                uint64_t total_chunks, uint32_t* route, uint32_t* error_word,
                                uint64_t wait_limit_ns, cudaStream_t stream) {
  if (route != nullptr)
    apply_route_kernel<<<1, 256, 0, stream>>>(tensors, ntensors, counts_dev, total_n, route);
  if (total_chunks == 0) return cudaGetLastError();
  int dev = 0;
  cudaGetDevice(&dev);
  apply_partition_kernel<<<unsigned((total_chunks + 255) / 256), 256, 0, stream>>>(
      tensors, chunk_begin, chunk_tensor, counts_dev, total_chunks, chunk_first, error_word, route);
  auto kernel = chunk_apply_kernel<1, kCwPreOne, kCwCtasOne, kCwBufOne>;
  static const int per_sm = resident_per_sm(kernel, kCwThreads, kCwCtasOne, cw_smem(kCwBufOne));
  const uint64_t cap = uint64_t(sm_count(dev)) * uint64_t(per_sm);
  const unsigned grid = unsigned(total_chunks < cap ? total_chunks : cap);
  const CwArgs args{tensors, chunk_begin, chunk_tensor, chunk_first, nullptr, counts_dev,
                    0,       1,           total_chunks, error_word, wait_limit_ns, route};
  kernel<<<grid, kCwThreads, cw_smem(kCwBufOne), stream>>>(args);
  return cudaGetLastError();
}

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
  const CwArgs args{tensors,  chunk_begin,  chunk_tensor, chain_first, segs, nullptr,
                    ntensors, nversions,    total_chunks, error_word,  wait_limit_ns, nullptr};
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
                               uint32_t* error_word, int grid, cudaStream_t stream,
                               const uint32_t* run_if) {
  return launch_apply_multi_t(tensors, ntensors, counts_dev, error_word, grid, stream, run_if);
}

cudaError_t launch_apply_u8_multi(const ByteSegment* segs, int nsegs, const uint64_t* counts_dev,
                                  uint32_t* error_word, int grid, cudaStream_t stream) {
  return launch_apply_multi_t(segs, nsegs, counts_dev, error_word, grid, stream, nullptr);
}

}  // namespace pulse
