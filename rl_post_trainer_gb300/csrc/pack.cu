// pack.cu -- codec-friendly packing of patch indices and its inverse.
//
// The pages compress patches with byte-oriented general codecs (PULSE
// summary, "1. PULSESync -- Compressione": zstd; humansand.ai summary,
// "Pipeline'i GPU'lara tasimak": LZ4 on nvCOMP, no entropy stage) and note
// that trainer-side compression latency can eat the gain. This step turns
// the ascending indices into small bit-packed gaps on the GPU, before such a
// codec:
//  * blocks of 128 entries: firsts[i] = first index, widths[i] = bit length
//    of the largest gap (gap = next - previous - 1), payload = 16 * width
//    bytes holding the 127 gaps as one little-endian bit string;
//  * chunks of 32 blocks (4096 entries): chunk_off[c] = byte offset of the
//    chunk's first payload, so every chunk decodes on its own.
//
// Pack: persistent CTAs (8 per SM) take chunks in ticket order, a ticket
// when its chunk starts; each warp measures and packs 4 blocks (bits OR-ed
// into shared-memory words); the chunk's payload offset is the exclusive
// prefix of the chunk sizes, found with the decoupled look-back shared with
// the encode kernels (warp 0), counted in 16-byte units.
// The pack CTAs keep the segments' chunk ranges in shared memory (loaded
// once per CTA when there are fewer than kSegCache segments), so finding a
// chunk's segment costs no dependent global loads.
// Unpack: one CTA per chunk; each warp extracts a block's gaps and rebuilds
// its indices with a warp scan.
#include "encode_common.cuh"

namespace pulse {
namespace {

constexpr int kPackBlock = 128;
constexpr int kPackChunkBlocks = 32;
constexpr int kPackChunk = kPackBlock * kPackChunkBlocks;  // 4096 entries
constexpr int kPackThreads = 256;
constexpr int kPackWarps = kPackThreads / 32;
constexpr int kBlocksPerWarp = kPackChunkBlocks / kPackWarps;  // 4

struct PackLaunch {
  PackSegment one;             // single-segment mode (chunk_begin 0)
  const PackSegment* segs;     // multi-segment mode: device table
  const uint64_t* chunk_begin; // multi-segment mode: nsegs + 1 entries (device)
  int nsegs;
  uint64_t total_chunks;
  uint64_t* status;
  uint32_t* counters;
  uint32_t epoch;
  uint64_t wait_limit_ns;
};

constexpr int kSegCache = 1024;  // segments whose chunk ranges a CTA keeps in shared memory
#ifndef PULSE_PACK_LOOKBACK
#define PULSE_PACK_LOOKBACK 1
#endif
// Status words per lane and look-back round trip. The whole CTA waits for
// its chunk's prefix, so the look-back's own latency is what counts: one word
// per lane (32 predecessors per round trip) measured faster than 2, 4 or 8.
constexpr int kPackLookback = PULSE_PACK_LOOKBACK;
constexpr int kPackCtasPerSm = 8;

// Copy the chunk ranges into shared memory when they fit (multi-segment).
template <bool MULTI>
__device__ __forceinline__ void load_seg_begin(const PackLaunch& a, uint64_t* sbeg) {
  if (MULTI && a.nsegs < kSegCache)
    for (int k = threadIdx.x; k <= a.nsegs; k += kPackThreads) sbeg[k] = a.chunk_begin[k];
}

// The segment that global chunk c belongs to: the largest s with
// chunk_begin[s] <= c (chunk_begin[nsegs] = total > c); sbeg: the shared
// copy of chunk_begin, or null to search the global one.
template <bool MULTI>
__device__ __forceinline__ PackSegment segment_of(const PackLaunch& a, const uint64_t* sbeg,
                                                  uint64_t c) {
  if (!MULTI) return a.one;
  if (sbeg == nullptr || a.nsegs >= kSegCache)
    return a.segs[enc::find_tensor(a.chunk_begin, a.nsegs, c)];
  int lo = 0, hi = a.nsegs;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sbeg[mid] <= c) lo = mid; else hi = mid - 1;
  }
  return a.segs[lo];
}

__device__ __forceinline__ uint32_t bit_width(uint32_t v) { return v ? 32u - __clz(v) : 0u; }

struct PackSmem {
  uint32_t words[kPackWarps][kBlocksPerWarp][kPackBlock];  // every block's packed words
  uint32_t width_of[kPackChunkBlocks];
  uint32_t prefix16;
};

// Pack chunk c (of segment sg): firsts, widths, the chunk's payload offset
// (look-back) and its payload. Ends with every thread done with `sm`.
template <bool MULTI>
__device__ __forceinline__ void pack_chunk(const PackLaunch& a, PackSmem& sm, uint64_t c,
                                           const PackSegment& sg) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint64_t lc = c - sg.chunk_begin;  // chunk within the segment
  const uint64_t chunk_first = lc * kPackChunk;

  // ---- widths and firsts; the gaps stay in registers
  uint32_t gap[kBlocksPerWarp][4];
  uint32_t cnt_blk[kBlocksPerWarp];
#pragma unroll
  for (int q = 0; q < kBlocksPerWarp; ++q) {
    const int lb = warp * kBlocksPerWarp + q;
    const uint64_t start = chunk_first + uint64_t(lb) * kPackBlock;
    const uint32_t cnt = start < sg.count ? uint32_t(sg.count - start < kPackBlock ? sg.count - start : kPackBlock) : 0u;
    cnt_blk[q] = cnt;
    uint32_t v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t j = uint32_t(lane) * 4u + uint32_t(e);
      v[e] = j < cnt ? sg.idx[start + j] : 0u;
    }
    const uint32_t before = __shfl_up_sync(0xFFFFFFFFu, v[3], 1);  // lane - 1's last entry
    uint32_t mx = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t j = uint32_t(lane) * 4u + uint32_t(e);
      const uint32_t prev = e == 0 ? before : v[e - 1];
      gap[q][e] = (j >= 1 && j < cnt) ? v[e] - prev - 1u : 0u;
      mx = max(mx, gap[q][e]);
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) {
      sm.width_of[lb] = cnt ? bit_width(mx) : 0u;
      if (cnt) {
        sg.firsts[start / kPackBlock] = v[0];
        sg.widths[start / kPackBlock] = uint8_t(bit_width(mx));
      }
    }
  }
  __syncthreads();

  // ---- every block's gaps into shared words; warp 0 first finds the chunk's
  // payload offset (16-byte units) with the look-back, so the other warps
  // pack while it waits
  auto pack_words = [&](int q) {
    const int lb = warp * kBlocksPerWarp + q;
    const uint32_t b = sm.width_of[lb];
    if (b == 0u) return;  // warp-uniform
    uint32_t* words = sm.words[warp][q];
    for (uint32_t w = lane; w < 4u * b; w += 32) words[w] = 0u;
    __syncwarp();
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t j = uint32_t(lane) * 4u + uint32_t(e);
      if (j >= 1 && j < cnt_blk[q] && gap[q][e] != 0u) {
        const uint32_t bit = (j - 1u) * b;
        const uint32_t w0 = bit >> 5, sh = bit & 31u;
        atomicOr(&words[w0], gap[q][e] << sh);
        if (sh + b > 32u) atomicOr(&words[w0 + 1], gap[q][e] >> (32u - sh));
      }
    }
  };
  if (warp == 0) {
    const uint32_t wl = sm.width_of[lane];
    const uint32_t agg = __reduce_add_sync(0xFFFFFFFFu, wl);
    // the look-back restarts at each segment's first chunk
    const uint64_t first = sg.chunk_begin;
    if (lane == 0)
      st_relaxed_u64(a.status + c, make_status(c == first ? kFlagPrefix : kFlagAggregate, a.epoch, agg));
    uint32_t p = 0;
    if (c != first) {
      uint64_t win[kPackLookback];
      enc::load_window<enc::StatusEpoch, PackLaunch, kPackLookback>(a, int64_t(c) - 1, first, lane,
                                                                   win);
      p = enc::resolve_prefix<enc::StatusEpoch, PackLaunch, 32, kPackLookback>(a, c, first, agg,
                                                                              lane, win);
    }
    if (lane == 0) {
      sm.prefix16 = p;
      sg.chunk_off[lc] = uint64_t(p) * 16u;
      if ((lc + 1) * kPackChunk >= sg.count) *sg.payload_bytes = (uint64_t(p) + agg) * 16u;
    }
  }
#pragma unroll
  for (int q = 0; q < kBlocksPerWarp; ++q) pack_words(q);
  __syncthreads();  // the offset and every block's words are in shared memory

  // ---- write the words out
  uint32_t off16 = sm.prefix16;
  for (int q = 0; q < warp * kBlocksPerWarp; ++q) off16 += sm.width_of[q];
#pragma unroll
  for (int q = 0; q < kBlocksPerWarp; ++q) {
    const uint32_t b = sm.width_of[warp * kBlocksPerWarp + q];
    uint32_t* dst = reinterpret_cast<uint32_t*>(sg.payload + uint64_t(off16) * 16u);
    for (uint32_t w = lane; w < 4u * b; w += 32) dst[w] = sm.words[warp][q][w];
    off16 += b;
  }
  __syncthreads();  // the shared words and widths are free again
}

template <bool MULTI>
__global__ void __launch_bounds__(kPackThreads, kPackCtasPerSm)
    pack_kernel(const __grid_constant__ PackLaunch a) {
  __shared__ PackSmem sm;
  __shared__ uint32_t ticket;
  __shared__ uint64_t sbeg[MULTI ? kSegCache : 1];
  const int tid = threadIdx.x;
  load_seg_begin<MULTI>(a, sbeg);
  // Chunks are taken in ticket order, so every smaller ticket is held by a
  // running CTA. A ticket is taken only when its chunk starts: a ticket held
  // ahead would keep its aggregate from the look-backs behind it meanwhile.
  for (;;) {
    if (tid == 0) ticket = atomicAdd(a.counters + 0, 1u);
    __syncthreads();
    const uint64_t c = ticket;
    if (c >= a.total_chunks) break;  // the same shared word for every thread
    pack_chunk<MULTI>(a, sm, c, segment_of<MULTI>(a, sbeg, c));  // ends in a CTA barrier
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

struct UnpackSmem {
  uint32_t words[kPackWarps][kPackBlock + 1];
};

// Rebuild the indices of chunk c (of segment sg).
template <bool MULTI>
__device__ __forceinline__ void unpack_chunk(UnpackSmem& sm, uint64_t c, const PackSegment& sg) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t lc = c - sg.chunk_begin;  // chunk within the segment
  const uint64_t chunk_first = lc * kPackChunk;
  const uint64_t count = sg.count;
  const uint32_t* __restrict__ firsts = sg.firsts;
  const uint8_t* __restrict__ widths = sg.widths;
  const uint8_t* __restrict__ payload = sg.payload;
  uint32_t* __restrict__ idx_out = sg.idx;
  const uint64_t nblocks = (count + kPackBlock - 1) / kPackBlock;
  // widths of the chunk's blocks and their exclusive prefix (16-byte units)
  const uint64_t gb_lane = lc * kPackChunkBlocks + uint64_t(lane);
  const uint32_t wl = gb_lane < nblocks ? widths[gb_lane] : 0u;
  uint32_t incl = wl;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  const uint64_t base_off = sg.chunk_off[lc];
#pragma unroll
  for (int q = 0; q < kBlocksPerWarp; ++q) {
    const int lb = warp * kBlocksPerWarp + q;
    const uint32_t b = __shfl_sync(0xFFFFFFFFu, wl, lb);
    const uint32_t pre = __shfl_sync(0xFFFFFFFFu, incl - wl, lb);
    const uint64_t start = chunk_first + uint64_t(lb) * kPackBlock;
    if (start >= count) break;  // warp-uniform
    const uint32_t cnt = uint32_t(count - start < kPackBlock ? count - start : kPackBlock);
    const uint32_t* src = reinterpret_cast<const uint32_t*>(payload + base_off + uint64_t(pre) * 16u);
    for (uint32_t w = lane; w < 4u * b; w += 32) sm.words[warp][w] = src[w];
    if (lane == 0) sm.words[warp][4u * b] = 0u;  // a zero word past the end for two-word reads
    __syncwarp();
    // x_j = gap_j + 1 for j >= 1, x_0 = 0; idx_j = first + inclusive sum of x
    uint32_t x[4];
    uint32_t sum = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t j = uint32_t(lane) * 4u + uint32_t(e);
      uint32_t g = 0;
      if (j >= 1 && j < cnt && b != 0u) {
        const uint32_t bit = (j - 1u) * b;
        const uint32_t w0 = bit >> 5, sh = bit & 31u;
        const uint64_t two = uint64_t(sm.words[warp][w0]) | (uint64_t(sm.words[warp][w0 + 1]) << 32);
        g = uint32_t((two >> sh) & ((b == 32u) ? 0xFFFFFFFFull : ((1ull << b) - 1ull)));
      }
      x[e] = (j >= 1 && j < cnt) ? g + 1u : 0u;
      sum += x[e];
    }
    uint32_t run = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, run, o);
      if (lane >= o) run += v;
    }
    uint32_t cur = firsts[start / kPackBlock] + (run - sum);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t j = uint32_t(lane) * 4u + uint32_t(e);
      cur += x[e];
      if (j < cnt) idx_out[start + j] = cur;
    }
    __syncwarp();
  }
}

// One CTA per chunk (no ordering between chunks; as short-lived CTAs the
// chunks overlap better than in a persistent loop).
template <bool MULTI>
__global__ void __launch_bounds__(kPackThreads) unpack_kernel(const __grid_constant__ PackLaunch a) {
  __shared__ UnpackSmem sm;
  const uint64_t c = blockIdx.x;
  unpack_chunk<MULTI>(sm, c, segment_of<MULTI>(a, nullptr, c));
}

// Persistent pack grid: kPackCtasPerSm CTAs per SM, or fewer chunks.
unsigned pack_grid(uint64_t chunks) {
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t cap = uint64_t(sm_count(dev)) * uint64_t(kPackCtasPerSm);
  return unsigned(chunks < cap ? chunks : cap);
}

}  // namespace

uint64_t pack_chunks(uint64_t count) { return (count + kPackChunk - 1) / kPackChunk; }

cudaError_t launch_pack(const uint32_t* idx, uint64_t count, uint32_t* firsts, uint8_t* widths,
                        uint64_t* chunk_off, uint8_t* payload, uint64_t* payload_bytes,
                        uint64_t* status, uint32_t* counters, uint32_t epoch,
                        uint64_t wait_limit_ns, cudaStream_t stream) {
  PackLaunch a{};
  a.one = PackSegment{const_cast<uint32_t*>(idx), count, firsts, widths, chunk_off, payload,
                      payload_bytes, 0};
  a.nsegs = 1;
  a.total_chunks = pack_chunks(count);
  a.status = status;
  a.counters = counters;
  a.epoch = epoch;
  a.wait_limit_ns = wait_limit_ns;
  if (a.total_chunks == 0) return cudaSuccess;
  pack_kernel<false><<<pack_grid(a.total_chunks), kPackThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_pack_multi(const PackSegment* segs, const uint64_t* chunk_begin, int nsegs,
                              uint64_t total_chunks, uint64_t* status, uint32_t* counters,
                              uint32_t epoch, uint64_t wait_limit_ns, cudaStream_t stream) {
  if (total_chunks == 0) return cudaSuccess;
  PackLaunch a{};
  a.segs = segs;
  a.chunk_begin = chunk_begin;
  a.nsegs = nsegs;
  a.total_chunks = total_chunks;
  a.status = status;
  a.counters = counters;
  a.epoch = epoch;
  a.wait_limit_ns = wait_limit_ns;
  pack_kernel<true><<<pack_grid(total_chunks), kPackThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t* firsts, const uint8_t* widths, const uint64_t* chunk_off,
                          const uint8_t* payload, uint64_t count, uint32_t* idx_out,
                          cudaStream_t stream) {
  const uint64_t chunks = pack_chunks(count);
  if (chunks == 0) return cudaSuccess;
  PackLaunch a{};
  a.one = PackSegment{idx_out, count, const_cast<uint32_t*>(firsts), const_cast<uint8_t*>(widths),
                      const_cast<uint64_t*>(chunk_off), const_cast<uint8_t*>(payload), nullptr, 0};
  a.nsegs = 1;
  a.total_chunks = chunks;
  unpack_kernel<false><<<unsigned(chunks), kPackThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_unpack_multi(const PackSegment* segs, const uint64_t* chunk_begin, int nsegs,
                                uint64_t total_chunks, cudaStream_t stream) {
  if (total_chunks == 0) return cudaSuccess;
  PackLaunch a{};
  a.segs = segs;
  a.chunk_begin = chunk_begin;
  a.nsegs = nsegs;
  a.total_chunks = total_chunks;
  unpack_kernel<true><<<unsigned(total_chunks), kPackThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pulse
