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

}  // namespace

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
