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
// Pack: persistent warp-specialized CTAs (3 per SM). A producer warp stages
// each chunk's indices with a bulk copy; 8 compute warps measure and pack 4
// blocks each and park the chunk's words in a shared-memory ring; a look-back
// warp finds the chunk's payload offset (the exclusive prefix of the chunk
// sizes, in 16-byte units, with the decoupled look-back shared with the
// encode kernels) and copies the words out, so no compute warp waits on
// another CTA. The CTAs keep the segments' chunk ranges in shared memory
// (loaded once per CTA when there are fewer than kSegCache segments), so
// finding a chunk's segment costs no dependent global loads.
// Unpack: one CTA per chunk; each warp extracts a block's gaps and rebuilds
// its indices with a warp scan.
#include <type_traits>

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
// Status words per lane and look-back round trip (32 predecessors per round
// trip with one word per lane).
constexpr int kPackLookback = PULSE_PACK_LOOKBACK;
#ifndef PULSE_PK_LB_SLEEP
#define PULSE_PK_LB_SLEEP 32
#endif
constexpr unsigned kPkLookbackSleepNs = PULSE_PK_LB_SLEEP;  // look-back poll pause

// Copy the chunk ranges into shared memory when they fit (multi-segment).
template <bool MULTI>
__device__ __forceinline__ void load_seg_begin(const PackLaunch& a, uint32_t* sbeg, int nthreads) {
  // fewer than kSegCache segments of fewer than 2^20 chunks each: the chunk
  // numbers fit 32 bits
  if (MULTI && a.nsegs < kSegCache)
    for (int k = threadIdx.x; k <= a.nsegs; k += nthreads) sbeg[k] = uint32_t(a.chunk_begin[k]);
}

// The segment that global chunk c belongs to: the largest s with
// chunk_begin[s] <= c (chunk_begin[nsegs] = total > c); sbeg: the shared
// copy of chunk_begin, or null to search the global one.
template <bool MULTI>
__device__ __forceinline__ PackSegment segment_of(const PackLaunch& a, const uint32_t* sbeg,
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

// ----------------------------------------------------------------- pack
// Persistent, warp-specialized CTA (the shape of the BF16 encode kernel):
//  * producer warp (one thread): takes a chunk ticket whenever a stage is
//    free and stages the chunk's 4096 indices (16 KB) in a kPkStages-deep
//    ring with a bulk copy (plain loads by the compute threads for a
//    segment's last, partial chunk or an index array that is not 16-byte
//    aligned);
//  * 8 compute warps (4 blocks each): form the gaps, take each block's width,
//    write firsts and widths, publish the chunk's size (16-byte units) in its
//    status word, and park the chunk's packed words in a shared-memory word
//    ring (each lane ORs its four gaps, as one bit string, into the block's
//    zeroed words);
//  * one look-back warp: resolves each parked chunk's payload offset with the
//    decoupled look-back, writes chunk_off (and the segment's payload size
//    after its last chunk), copies the words to the payload with 16-byte
//    stores and frees the ring.
// The compute warps never wait on another CTA: while a chunk's offset is
// resolved they pack the next ones (up to kPkSlots parked chunks).
constexpr int kPkCompute = 256;                     // compute threads (8 warps)
constexpr int kPkWarps = kPkCompute / 32;
constexpr int kPkProducerWarp = kPkWarps;
constexpr int kPkLookbackWarp = kPkWarps + 1;
constexpr int kPkThreads = kPkCompute + 64;
#ifndef PULSE_PK_STAGES
#define PULSE_PK_STAGES 2
#endif
#ifndef PULSE_PK_CTAS
#define PULSE_PK_CTAS 3
#endif
constexpr int kPkStages = PULSE_PK_STAGES;
#ifndef PULSE_PK_PARKED
#define PULSE_PK_PARKED 16  // 0.962 against 0.966 ms with 8 on the 8.03B patch
#endif
constexpr int kPkSlots = PULSE_PK_PARKED;           // parked chunks per CTA
#ifndef PULSE_PK_RING
#define PULSE_PK_RING 4096
#endif
constexpr uint32_t kPkRing = PULSE_PK_RING;         // parked payload words per CTA
constexpr uint32_t kPkRingMask = kPkRing - 1u;
static_assert((kPkRing & (kPkRing - 1u)) == 0u, "the word ring is a power of two");
constexpr uint32_t kPkStageBytes = kPackChunk * 4;  // 16 KB of indices
constexpr int kPkCtasPerSm = PULSE_PK_CTAS;
static_assert(kPkCompute == kEncThreads, "the compute warps use the encode's named barrier");
static_assert(kBlocksPerWarp * kPkWarps == kPackChunkBlocks, "8 warps x 4 blocks per chunk");
static_assert(kPkRing >= uint32_t(kPackChunkBlocks) * 4u * 32u, "a chunk of 32-bit gaps fits the ring");
constexpr size_t kPkDynSmem = size_t(kPkStages) * kPkStageBytes + size_t(kPkRing) * 4 + 128;

enum : uint32_t { kPkEnd = 0, kPkBulk = 1, kPkGeneric = 2 };

struct PkStageMeta {
  uint64_t c;        // global chunk
  uint64_t lc;       // chunk within its segment
  uint32_t mode;
  uint32_t cnt;      // indices in the chunk
  PackSegment sg;
};

struct PkParked {
  uint64_t c, first, lc;
  uint32_t agg;      // payload size in 16-byte units
  uint32_t ring_start;
  uint32_t last;     // 1: the segment's last chunk; 2: no more chunks
  uint64_t* chunk_off;
  uint8_t* payload;
  uint64_t* payload_bytes;
};

struct __align__(16) PkShared {
  uint64_t full[kPkStages];
  uint64_t empty[kPkStages];
  uint64_t agg_ready[kPkSlots];
  uint64_t slot_free[kPkSlots];
  PkStageMeta meta[kPkStages];
  PkParked parked[kPkSlots];
  uint32_t wid[2][kPackChunkBlocks];  // block widths, by iteration parity
  uint32_t ring_tail;
};

template <bool MULTI>
__device__ __forceinline__ void pk_producer(const PackLaunch& a, PkShared& sh, uint8_t* stages,
                                            const uint32_t* sbeg) {
  const uint64_t pol_stream = l2_policy_evict_first();
  uint32_t fills_done = 0;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kPkStages);
    if (it >= uint32_t(kPkStages) &&
        !enc::helper_wait(&sh.empty[s], ((it / kPkStages) - 1) & 1u, a))
      break;
    // the ticket only once its stage is free: a chunk's count is published
    // soon after its ticket, so look-backs behind it wait less
    const uint64_t ticket = atomicAdd(a.counters + 0, 1u);
    const bool end = ticket >= a.total_chunks;
    fills_done = it + 1;
    PkStageMeta m{};
    m.c = ticket;
    if (end) {
      m.mode = kPkEnd;
      sh.meta[s] = m;
      mbar_arrive(&sh.full[s]);
      break;
    }
    m.sg = segment_of<MULTI>(a, sbeg, ticket);
    m.lc = ticket - m.sg.chunk_begin;
    const uint64_t start = m.lc * kPackChunk;
    m.cnt = uint32_t(m.sg.count - start < uint64_t(kPackChunk) ? m.sg.count - start : kPackChunk);
    const uint32_t* src = m.sg.idx + start;
    if (m.cnt == uint32_t(kPackChunk) && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
      m.mode = kPkBulk;
      sh.meta[s] = m;
      mbar_arrive_expect_tx(&sh.full[s], kPkStageBytes);
      bulk_g2s(stages + size_t(s) * kPkStageBytes, src, kPkStageBytes, &sh.full[s], pol_stream);
    } else {
      m.mode = kPkGeneric;
      sh.meta[s] = m;
      mbar_arrive(&sh.full[s]);
    }
  }
  // no bulk copy may still be in flight when the CTA exits
  for (uint32_t f = fills_done > uint32_t(kPkStages) ? fills_done - kPkStages : 0u; f < fills_done; ++f)
    mbar_wait_bounded(&sh.full[f % kPkStages], (f / kPkStages) & 1u, a.wait_limit_ns);
  // the last CTA to stop taking tickets rewinds the counters for the next launch
  __threadfence();
  const uint32_t finished = atomicAdd(a.counters + 1, 1u);
  if (finished == gridDim.x - 1) {
    atomicExch(a.counters + 0, 0u);
    atomicExch(a.counters + 1, 0u);
  }
}

// Copy a parked chunk's words to payload + 16 * prefix (16-byte units; the
// payload is 16-byte aligned and the chunk's words start at a ring position
// that is a multiple of 4, so no unit straddles the ring's end).
__device__ __forceinline__ void pk_copy_out(const PkParked& pm, uint32_t prefix, const uint32_t* ring,
                                            int lane) {
  uint4* dst = reinterpret_cast<uint4*>(pm.payload) + prefix;
  for (uint32_t k = uint32_t(lane); k < pm.agg; k += 32)
    dst[k] = *reinterpret_cast<const uint4*>(ring + ((pm.ring_start + 4u * k) & kPkRingMask));
}

__device__ __forceinline__ void pk_lookback(const PackLaunch& a, PkShared& sh, const uint32_t* ring,
                                            int lane) {
  for (uint32_t i = 0;;) {
    const bool ok = enc::helper_wait(&sh.agg_ready[i % kPkSlots], (i / kPkSlots) & 1u, a);
    if (!__all_sync(0xFFFFFFFFu, ok)) break;
    int more = 0;
    if (lane == 0) {
      for (int b = 1; b < enc::kLookbackBatch; ++b) {
        const uint32_t ii = i + uint32_t(b);
        if (!mbar_test_wait(&sh.agg_ready[ii % kPkSlots], (ii / kPkSlots) & 1u)) break;
        more = b;
      }
    }
    more = __shfl_sync(0xFFFFFFFFu, more, 0);
    int nb = 0;
    bool end = false;
    uint64_t win[enc::kLookbackBatch][kPackLookback];
#pragma unroll
    for (int b = 0; b < enc::kLookbackBatch; ++b) {
      if (b > more || end) continue;
      const uint32_t ii = i + uint32_t(b);
      const int q = int(ii % kPkSlots);
      if (b > 0) mbar_test_wait(&sh.agg_ready[q], (ii / kPkSlots) & 1u);  // acquire for every lane
      const PkParked& pm = sh.parked[q];
      if (pm.last == 2u) {
        end = true;
        continue;
      }
      if (pm.c != pm.first)
        enc::load_window<enc::StatusEpoch, PackLaunch, kPackLookback>(a, int64_t(pm.c) - 1, pm.first,
                                                                      lane, win[b]);
      nb = b + 1;
    }
#pragma unroll
    for (int b = 0; b < enc::kLookbackBatch; ++b) {
      if (b >= nb) continue;
      const uint32_t ii = i + uint32_t(b);
      const int q = int(ii % kPkSlots);
      const PkParked pm = sh.parked[q];
      const uint32_t prefix = enc::resolve_prefix<enc::StatusEpoch, PackLaunch, kPkLookbackSleepNs, kPackLookback>(
          a, pm.c, pm.first, pm.agg, lane, win[b]);
      if (lane == 0) {
        pm.chunk_off[pm.lc] = uint64_t(prefix) * 16u;
        if (pm.last == 1u) *pm.payload_bytes = (uint64_t(prefix) + pm.agg) * 16u;
      }
      pk_copy_out(pm, prefix, ring, lane);
      __syncwarp();
      if (lane == 0) {
        // chunks are copied out in order: every word before this chunk's end is free
        __threadfence_block();
        *reinterpret_cast<volatile uint32_t*>(&sh.ring_tail) = pm.ring_start + 4u * pm.agg;
        mbar_arrive(&sh.slot_free[q]);
      }
    }
    if (end) break;
    i += uint32_t(nb);
  }
}

// A block's payload words from its gaps. Lane l holds the gaps of entries
// 4l .. 4l+3, i.e. bit slots 4l-1 .. 4l+2 of the block's bit string (slot t
// at bits t*b; lane 0's first gap is the block's first entry, always 0), so
// its 4b-bit string S_l lies at bit 4lb - b (lane 0: its last 3b bits at bit
// 0). The block's 4b words (ring positions base + w, masked) are zeroed,
// then each lane ORs S_l in: at most 2 words for b <= 8, 5 for wider gaps;
// only non-zero parts are written, and every written word lies inside the
// block's 4b (its string ends at bit 127b). Whole warp; b warp-uniform.
__device__ __forceinline__ void pk_block_words(const uint32_t (&g)[4], uint32_t b, uint32_t* ring,
                                               uint32_t base, int lane) {
  if (b == 0u) return;
  const uint32_t L = 4u * b;
  for (uint32_t w = uint32_t(lane); w < L; w += 32) ring[(base + w) & kPkRingMask] = 0u;
  __syncwarp();
  const uint32_t P = lane == 0 ? 0u : uint32_t(lane) * L - b;  // first bit of this lane's string
  const uint32_t w0 = base + (P >> 5), sh = P & 31u;
  if (b <= 8u) {
    uint32_t S = g[0] | (g[1] << b) | (g[2] << (2u * b)) | (g[3] << (3u * b));
    if (lane == 0) S >>= b;
    const uint32_t x0 = S << sh, x1 = sh ? S >> (32u - sh) : 0u;
    if (x0) atomicOr(&ring[w0 & kPkRingMask], x0);
    if (x1) atomicOr(&ring[(w0 + 1u) & kPkRingMask], x1);
  } else {
    // the 128-bit string in four words, then shifted by sh into five
    uint64_t lo = uint64_t(g[0]) | (uint64_t(g[1]) << b);
    const uint64_t hi = uint64_t(g[2]) | (uint64_t(g[3]) << b);
    uint64_t top;
    if (b == 32u) {
      top = hi;
    } else {
      lo |= hi << (2u * b);
      top = hi >> (64u - 2u * b);
    }
    uint32_t s0 = uint32_t(lo), s1 = uint32_t(lo >> 32), s2 = uint32_t(top), s3 = uint32_t(top >> 32);
    if (lane == 0) {  // drop the leading b zero bits (9 <= b <= 32)
      const uint32_t q = b >> 5, r = b & 31u;  // q is 1 only for b == 32
      if (q) { s0 = s1; s1 = s2; s2 = s3; s3 = 0u; }
      if (r) {
        s0 = __funnelshift_r(s0, s1, r);
        s1 = __funnelshift_r(s1, s2, r);
        s2 = __funnelshift_r(s2, s3, r);
        s3 >>= r;
      }
    }
    uint32_t x[5];
    x[0] = s0 << sh;
    x[1] = __funnelshift_l(s0, s1, sh);
    x[2] = __funnelshift_l(s1, s2, sh);
    x[3] = __funnelshift_l(s2, s3, sh);
    x[4] = sh ? s3 >> (32u - sh) : 0u;
#pragma unroll
    for (int k = 0; k < 5; ++k)
      if (x[k]) atomicOr(&ring[(w0 + uint32_t(k)) & kPkRingMask], x[k]);
  }
}

template <bool MULTI>
__device__ __forceinline__ void pk_compute(const PackLaunch& a, PkShared& sh, const uint8_t* stages,
                                           uint32_t* ring, int tid, int lane, int warp) {
  uint32_t posted = 0, ring_head = 0;
  bool failed = false;
  for (uint32_t it = 0;; ++it) {
    const int s = int(it % kPkStages);
    failed |= !enc::wait_or_flag(&sh.full[s], (it / kPkStages) & 1u, a);
    const PkStageMeta m = sh.meta[s];
    const bool live = m.mode != kPkEnd;
    const bool bulk = m.mode == kPkBulk;
    const uint32_t* sidx = reinterpret_cast<const uint32_t*>(stages + size_t(s) * kPkStageBytes);
    const uint64_t chunk_first = m.lc * kPackChunk;
    const int pc = int(it & 1u);

    // ---- gaps and widths of this warp's 4 blocks (gaps stay in registers);
    // compiled apart for a full staged chunk, where every block has 128 entries
    uint32_t gap[kBlocksPerWarp][4];
    uint32_t wb[kBlocksPerWarp];  // block widths (every lane)
    auto widths = [&](auto full_tag) {
      constexpr bool kFull = decltype(full_tag)::value;
#pragma unroll
      for (int q = 0; q < kBlocksPerWarp; ++q) {
        const int lb = warp * kBlocksPerWarp + q;
        const uint32_t b0 = uint32_t(lb) * kPackBlock;  // block start within the chunk
        const uint32_t cnt = kFull ? uint32_t(kPackBlock)
                                   : (live && m.cnt > b0 ? (m.cnt - b0 < uint32_t(kPackBlock) ? m.cnt - b0 : kPackBlock) : 0u);
        uint32_t v[4];
        if constexpr (kFull) {
          const uint4 x = reinterpret_cast<const uint4*>(sidx + b0)[lane];
          v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t j = uint32_t(lane) * 4u + uint32_t(e);
            v[e] = j < cnt ? m.sg.idx[chunk_first + b0 + j] : 0u;
          }
        }
        const uint32_t before = __shfl_up_sync(0xFFFFFFFFu, v[3], 1);  // lane - 1's last index
        uint32_t mx = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t j = uint32_t(lane) * 4u + uint32_t(e);
          const uint32_t prev = e == 0 ? before : v[e - 1];
          gap[q][e] = (j >= 1 && j < cnt) ? v[e] - prev - 1u : 0u;
          mx = max(mx, gap[q][e]);
        }
        mx = __reduce_max_sync(0xFFFFFFFFu, mx);
        wb[q] = cnt ? bit_width(mx) : 0u;
        if (lane == 0) {
          sh.wid[pc][lb] = wb[q];
          if (cnt) {
            const uint64_t gb = (chunk_first + b0) / kPackBlock;
            m.sg.firsts[gb] = v[0];
            m.sg.widths[gb] = uint8_t(wb[q]);
          }
        }
      }
    };
    if (bulk) widths(std::true_type{}); else widths(std::false_type{});
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[s]);  // this warp is done with stage s
    if (enc::compute_barrier_or(failed || !live)) break;

    // ---- block offsets within the chunk (16-byte units) and the chunk's size
    const uint32_t wl = sh.wid[pc][lane];
    uint32_t incl = wl;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    const uint32_t agg = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint32_t my_off = __shfl_sync(0xFFFFFFFFu, incl - wl, warp * kBlocksPerWarp);
    const uint64_t first = m.sg.chunk_begin;  // the look-back restarts at each segment
    if (tid == 0)
      st_relaxed_u64(a.status + m.c, make_status(m.c == first ? kFlagPrefix : kFlagAggregate, a.epoch, agg));

    // ---- room: the parked slot must be free and the ring must hold the words
    const int q = int(posted % kPkSlots);
    if (posted >= uint32_t(kPkSlots))
      failed |= !enc::wait_or_flag(&sh.slot_free[q], ((posted - kPkSlots) / kPkSlots) & 1u, a);
    failed |= !enc::wait_ring_room<64>(&sh.ring_tail, ring_head, 4u * agg, kPkRing, a);

    // ---- park: each block's 4 * width words
    uint32_t off = my_off;
#pragma unroll
    for (int k = 0; k < kBlocksPerWarp; ++k) {
      pk_block_words(gap[k], wb[k], ring, ring_head + 4u * off, lane);
      off += wb[k];
    }
    if (tid == 0) {
      PkParked pm;
      pm.c = m.c;
      pm.first = first;
      pm.lc = m.lc;
      pm.agg = agg;
      pm.ring_start = ring_head;
      pm.last = (chunk_first + m.cnt >= m.sg.count) ? 1u : 0u;
      pm.chunk_off = m.sg.chunk_off;
      pm.payload = m.sg.payload;
      pm.payload_bytes = m.sg.payload_bytes;
      sh.parked[q] = pm;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.agg_ready[q]);  // 8 arrivals: every warp's words are in
    ++posted;
    ring_head += 4u * agg;
  }
  // no more chunks: wait until every parked chunk is copied out, then send
  // the look-back warp its end marker
  for (uint32_t e = posted > uint32_t(kPkSlots) ? posted - kPkSlots : 0u; e < posted; ++e)
    enc::wait_or_flag(&sh.slot_free[e % kPkSlots], (e / kPkSlots) & 1u, a);
  enc::compute_barrier();
  const int q = int(posted % kPkSlots);
  if (tid == 0) {
    PkParked pm{};
    pm.last = 2u;
    sh.parked[q] = pm;
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&sh.agg_ready[q]);
}

template <bool MULTI>
__global__ void __launch_bounds__(kPkThreads, kPkCtasPerSm)
    pack_kernel(const __grid_constant__ PackLaunch a) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ PkShared sh;
  __shared__ uint32_t sbeg[MULTI ? kSegCache : 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 127) & ~uintptr_t(127));
  uint32_t* ring = reinterpret_cast<uint32_t*>(stages + size_t(kPkStages) * kPkStageBytes);
  load_seg_begin<MULTI>(a, sbeg, kPkThreads);
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < kPkStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kPkWarps);
      sh.meta[s] = PkStageMeta{};
    }
#pragma unroll
    for (int q = 0; q < kPkSlots; ++q) {
      mbar_init(&sh.agg_ready[q], kPkWarps);
      mbar_init(&sh.slot_free[q], 1);
      sh.parked[q] = PkParked{};
      sh.parked[q].last = 2u;
    }
    sh.ring_tail = 0;
    fence_mbar_init();
  }
  __syncthreads();  // the last CTA-wide barrier: roles split below
  if (warp < kPkWarps) {
    pk_compute<MULTI>(a, sh, stages, ring, tid, lane, warp);
  } else if (warp == kPkProducerWarp) {
    if (lane == 0) pk_producer<MULTI>(a, sh, stages, sbeg);
  } else if (warp == kPkLookbackWarp) {
    pk_lookback(a, sh, ring, lane);
  }
}

struct __align__(16) UnpackSmem {
  // every block's words, then 4 zero words (two-word reads past the end)
  uint32_t words[kPackWarps][kBlocksPerWarp][kPackBlock + 4];
};

// Rebuild the indices of chunk c (of segment sg). Each warp first copies its
// 4 blocks' words to shared memory (16-byte loads when the payload is 16-byte
// aligned), then per block: lane l takes the gaps of entries 4l .. 4l+3 (bit
// slots 4l-1 .. 4l+2; for widths up to 8 all four come from one 64-bit window
// of two words), and a warp scan of gap + 1 from the block's first index
// gives the indices (one 16-byte store per lane for a full, aligned block).
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
  const bool vec_in = (reinterpret_cast<uintptr_t>(payload) & 15u) == 0;
  uint32_t bw[kBlocksPerWarp], first_idx[kBlocksPerWarp];
  // ---- every block's words into shared memory
#pragma unroll
  for (int q = 0; q < kBlocksPerWarp; ++q) {
    const int lb = warp * kBlocksPerWarp + q;
    const uint32_t b = __shfl_sync(0xFFFFFFFFu, wl, lb);
    const uint32_t pre = __shfl_sync(0xFFFFFFFFu, incl - wl, lb);
    const uint64_t start = chunk_first + uint64_t(lb) * kPackBlock;
    bw[q] = b;
    first_idx[q] = start < count ? firsts[start / kPackBlock] : 0u;
    uint32_t* dst = sm.words[warp][q];
    const uint8_t* src = payload + base_off + uint64_t(pre) * 16u;
    if (start < count) {
      if (vec_in) {
        if (uint32_t(lane) < b)
          reinterpret_cast<uint4*>(dst)[lane] = reinterpret_cast<const uint4*>(src)[lane];
      } else {
        for (uint32_t w = lane; w < 4u * b; w += 32)
          dst[w] = reinterpret_cast<const uint32_t*>(src)[w];
      }
    }
    if (lane < 4) dst[4u * b + uint32_t(lane)] = 0u;
  }
  __syncwarp();
  // ---- gaps and indices, block by block
  const bool vec_out = (reinterpret_cast<uintptr_t>(idx_out) & 15u) == 0;
#pragma unroll
  for (int q = 0; q < kBlocksPerWarp; ++q) {
    const int lb = warp * kBlocksPerWarp + q;
    const uint64_t start = chunk_first + uint64_t(lb) * kPackBlock;
    if (start >= count) break;  // warp-uniform
    const uint32_t cnt = uint32_t(count - start < kPackBlock ? count - start : kPackBlock);
    const uint32_t b = bw[q];
    const uint32_t* words = sm.words[warp][q];
    const uint32_t mask = b == 32u ? 0xFFFFFFFFu : (1u << b) - 1u;
    // x_j = gap_j + 1 for j >= 1, x_0 = 0; idx_j = first + inclusive sum of x
    uint32_t x[4];
    uint32_t sum = 0;
    if (b <= 8u) {
      // the lane's four slots: bits (4l-1)b .. (4l+3)b (lane 0: its three from bit 0)
      const uint32_t P = lane ? (4u * uint32_t(lane) - 1u) * b : 0u;
      const uint64_t two = uint64_t(words[P >> 5]) | (uint64_t(words[(P >> 5) + 1]) << 32);
      const uint32_t window = uint32_t(two >> (P & 31u));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t j = uint32_t(lane) * 4u + uint32_t(e);
        const int k = lane ? e : e - 1;  // slot within the lane's window
        const uint32_t g = k < 0 ? 0u : (window >> (uint32_t(k) * b)) & mask;
        x[e] = (j >= 1 && j < cnt) ? g + 1u : 0u;
        sum += x[e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t j = uint32_t(lane) * 4u + uint32_t(e);
        uint32_t g = 0;
        if (j >= 1 && j < cnt) {
          const uint32_t bit = (j - 1u) * b;
          const uint32_t w0 = bit >> 5, sh = bit & 31u;
          const uint64_t two = uint64_t(words[w0]) | (uint64_t(words[w0 + 1]) << 32);
          g = uint32_t(two >> sh) & mask;
        }
        x[e] = (j >= 1 && j < cnt) ? g + 1u : 0u;
        sum += x[e];
      }
    }
    uint32_t run = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, run, o);
      if (lane >= o) run += v;
    }
    uint32_t cur = first_idx[q] + (run - sum);
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      cur += x[e];
      out[e] = cur;
    }
    if (vec_out && cnt == uint32_t(kPackBlock)) {
      reinterpret_cast<uint4*>(idx_out + start)[lane] = make_uint4(out[0], out[1], out[2], out[3]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t j = uint32_t(lane) * 4u + uint32_t(e);
        if (j < cnt) idx_out[start + j] = out[e];
      }
    }
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

// Persistent pack grid: as many CTAs as fit on the GPU, or fewer chunks.
template <bool MULTI>
unsigned pack_grid(uint64_t chunks) {
  static int per_sm = [] {
    cudaFuncSetAttribute(pack_kernel<MULTI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         int(kPkDynSmem));
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, pack_kernel<MULTI>, kPkThreads,
                                                      kPkDynSmem) != cudaSuccess || b < 1)
      b = 1;
    return b;
  }();
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t cap = uint64_t(sm_count(dev)) * uint64_t(per_sm);
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
  pack_kernel<false><<<pack_grid<false>(a.total_chunks), kPkThreads, kPkDynSmem, stream>>>(a);
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
  pack_kernel<true><<<pack_grid<true>(total_chunks), kPkThreads, kPkDynSmem, stream>>>(a);
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
