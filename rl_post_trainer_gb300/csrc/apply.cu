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
                                 uint32_t* error_word, int grid, cudaStream_t stream) {
  const size_t smem = size_t(nsegs + 1) * sizeof(uint64_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(apply_multi_kernel<Seg>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
  }
  apply_multi_kernel<Seg><<<grid, kApplyThreads, smem, stream>>>(segs, nsegs, counts_dev, error_word);
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
constexpr int kChunkThreads = 256;
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
    apply_partition_kernel(const TensorDesc* tensors, const uint64_t* chunk_begin,
                           const uint32_t* chunk_tensor, const uint64_t* counts,
                           uint64_t total_chunks, uint32_t* chunk_first, uint32_t* err) {
  const uint64_t g = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (g >= total_chunks) return;
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

// Chunk g's entry range [e0, e1) and whether it goes dense.
struct ChunkWork {
  uint64_t g;
  uint32_t t;
  uint64_t e0, e1, base;
  uint32_t len;
  bool dense;
};

__device__ __forceinline__ ChunkWork chunk_work(const TensorDesc* tensors, const uint64_t* chunk_begin,
                                                const uint32_t* chunk_tensor,
                                                const uint32_t* chunk_first, const uint64_t* counts,
                                                uint64_t g) {
  ChunkWork c;
  c.g = g;
  c.t = chunk_tensor[g];
  const TensorDesc& d = tensors[c.t];
  uint64_t cnt = counts[c.t];
  if (cnt > d.n) cnt = d.n;
  c.e0 = chunk_first[g];
  c.e1 = g + 1 < chunk_begin[c.t + 1] ? chunk_first[g + 1] : cnt;
  if (c.e1 < c.e0) c.e1 = c.e0;
  c.base = (g - chunk_begin[c.t]) * kChunk;
  c.len = uint32_t(d.n - c.base < uint64_t(kChunk) ? d.n - c.base : uint64_t(kChunk));
  c.dense = c.e1 - c.e0 >= kDenseMin && (reinterpret_cast<uintptr_t>(d.w) % 16u == 0);
  return c;
}

constexpr int kPrefetchEntries = 4;  // entries per thread loaded before the chunk lands

__global__ void __launch_bounds__(kChunkThreads, kApplyChunkCtas)
    apply_chunk_kernel(const TensorDesc* tensors, const uint64_t* chunk_begin,
                       const uint32_t* chunk_tensor, const uint32_t* chunk_first,
                       const uint64_t* counts, uint64_t total_chunks, uint32_t* err,
                       uint64_t wait_limit_ns) {
  __shared__ __align__(128) uint16_t wsm[2][kChunk];  // double buffer
  __shared__ __align__(16) uint8_t dirty[kChunkSectors];  // one flag byte per 32-byte sector
  __shared__ __align__(8) uint64_t bar[2];
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t pol = l2_policy_evict_first();
  uint32_t phases = 0;  // bit b: parity of buffer b's next phase
  // issue the bulk copy of a dense chunk's body into buffer b (thread 0)
  auto stage = [&](const ChunkWork& c, int b) {
    if (tid == 0 && c.dense) {
      const TensorDesc& d = tensors[c.t];
      const uint32_t body = c.len & ~7u;
      mbar_arrive_expect_tx(&bar[b], body * 2u);
      if (body) bulk_g2s(wsm[b], d.w + c.base, body * 2u, &bar[b], pol);
    }
  };
  uint64_t g = blockIdx.x;
  ChunkWork cur{};
  if (g < total_chunks) {
    cur = chunk_work(tensors, chunk_begin, chunk_tensor, chunk_first, counts, g);
    stage(cur, 0);
  }
  for (int b = 0; g < total_chunks; g += gridDim.x, b ^= 1) {
    // the next chunk of this CTA starts loading into the other buffer now
    const uint64_t gn = g + gridDim.x;
    ChunkWork nxt{};
    if (gn < total_chunks) {
      nxt = chunk_work(tensors, chunk_begin, chunk_tensor, chunk_first, counts, gn);
      stage(nxt, b ^ 1);
    }
    const TensorDesc& d = tensors[cur.t];
    if (cur.e1 > cur.e0 && !cur.dense) {
      for (uint64_t j = cur.e0 + tid; j < cur.e1; j += kChunkThreads) {
        const uint32_t i = d.idx[j];
        if (uint64_t(i) < cur.base || uint64_t(i) >= cur.base + cur.len) {
          record_error(err, kErrIndex);
          continue;
        }
        d.w[i] = d.val[j];
      }
    } else if (cur.dense) {
      // entries of this chunk, loaded while its copy is in flight
      uint32_t pi[kPrefetchEntries];
      uint16_t pv[kPrefetchEntries];
#pragma unroll
      for (int q = 0; q < kPrefetchEntries; ++q) {
        const uint64_t j = cur.e0 + uint64_t(q) * kChunkThreads + tid;
        pi[q] = j < cur.e1 ? d.idx[j] : 0u;
        pv[q] = j < cur.e1 ? d.val[j] : uint16_t(0);
      }
      for (uint32_t k = tid; k < uint32_t(kChunkSectors) / 4u; k += kChunkThreads)
        reinterpret_cast<uint32_t*>(dirty)[k] = 0u;
      const uint32_t body = cur.len & ~7u;
      for (uint32_t k = body + tid; k < cur.len; k += kChunkThreads) wsm[b][k] = d.w[cur.base + k];
      const uint32_t par = (phases >> b) & 1u;
      const bool ok = mbar_wait_bounded(&bar[b], par, wait_limit_ns);
      phases ^= 1u << b;
      if (!__syncthreads_and(ok)) {
        // a copy did not land in time: report, give both buffers one more
        // bounded wait (no copy may still write shared memory at exit), stop
        if (tid == 0) record_error(err, kErrTimeout);
        mbar_wait_bounded(&bar[b], par, wait_limit_ns);
        if (nxt.dense) mbar_wait_bounded(&bar[b ^ 1], (phases >> (b ^ 1)) & 1u, wait_limit_ns);
        break;
      }
      auto put = [&](uint32_t i, uint16_t v) {
        if (uint64_t(i) < cur.base || uint64_t(i) >= cur.base + cur.len) {
          record_error(err, kErrIndex);
          return;
        }
        const uint32_t li = uint32_t(i - cur.base);
        wsm[b][li] = v;
        dirty[li >> 4] = 1u;  // plain store: every writer stores the same value
      };
#pragma unroll
      for (int q = 0; q < kPrefetchEntries; ++q) {
        const uint64_t j = cur.e0 + uint64_t(q) * kChunkThreads + tid;
        if (j < cur.e1) put(pi[q], pv[q]);
      }
      for (uint64_t j = cur.e0 + uint64_t(kPrefetchEntries) * kChunkThreads + tid; j < cur.e1;
           j += kChunkThreads)
        put(d.idx[j], d.val[j]);
      __syncthreads();
      // write back the changed sectors: 16 elements = two 16-byte stores each
      for (uint32_t sct = tid; sct < uint32_t(kChunkSectors); sct += kChunkThreads) {
        if (!dirty[sct]) continue;
        const uint32_t first = sct * 16u;
        if (first + 16u <= cur.len) {
          const uint4* src = reinterpret_cast<const uint4*>(wsm[b] + first);
          uint4* dst = reinterpret_cast<uint4*>(d.w + cur.base + first);
          dst[0] = src[0];
          dst[1] = src[1];
        } else {
          for (uint32_t k = first; k < cur.len; ++k) d.w[cur.base + k] = wsm[b][k];
        }
      }
      __syncthreads();  // buffer b and the dirty bits are reused
    }
    cur = nxt;
  }
}

}  // namespace

cudaError_t launch_apply_chunks(const TensorDesc* tensors, const uint64_t* chunk_begin,
                                const uint32_t* chunk_tensor, uint32_t* chunk_first,
                                const uint64_t* counts_dev, uint64_t total_chunks,
                                uint32_t* error_word, uint64_t wait_limit_ns, cudaStream_t stream) {
  if (total_chunks == 0) return cudaSuccess;
  int dev = 0;
  cudaGetDevice(&dev);
  apply_partition_kernel<<<unsigned((total_chunks + 255) / 256), 256, 0, stream>>>(
      tensors, chunk_begin, chunk_tensor, counts_dev, total_chunks, chunk_first, error_word);
  const uint64_t cap = uint64_t(sm_count(dev)) * uint64_t(kApplyChunkCtas);
  const unsigned grid = unsigned(total_chunks < cap ? total_chunks : cap);
  apply_chunk_kernel<<<grid, kChunkThreads, 0, stream>>>(tensors, chunk_begin, chunk_tensor,
                                                         chunk_first, counts_dev, total_chunks,
                                                         error_word, wait_limit_ns);
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
