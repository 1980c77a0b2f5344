// api.cu -- the C ABI declared in include/pulse.h: argument checks, the
// per-(device, stream) workspace of the single-tensor calls, and multi-tensor
// plans (tile tables built once on the host and replayed every step, as in
// the static schedule of "Weight transfer for RL post-training in under 2
// seconds", section "Statyczny harmonogram", and the CPU-prepared tiling and
// address map of the humansand.ai summary, section "Pipeline'i GPU'lara
// tasimak").
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "pulse.h"
#include "pulse_device.cuh"
#include "pulse_internal.h"

namespace pulse {

int sm_count(int device) {
  static std::mutex mu;
  static std::map<int, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(device);
  if (it != cache.end()) return it->second;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms < 1)
    sms = 1;
  cache[device] = sms;
  return sms;
}

namespace {

constexpr uint64_t kMaxElems = 0xFFFFFFFFull;      // n < 2^32 (uint32 indices)
constexpr uint64_t kMaxTiles = 0x7FFFFFFFull;      // tile tickets are uint32
constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // 1 s per bounded wait
constexpr size_t kCounterBytes = 256;               // ticket, finished, error (+ padding)
constexpr int kAmaxWord = 8;  // counters word holding a single-tensor NVFP4 maximum
constexpr int kMaxTensorsPerApplyLaunch = 16384;     // bound on the apply kernel's smem table

uint64_t div_up(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PULSE_OK : PULSE_ERR_CUDA; }

// Allocate (or grow) a workspace to hold `tiles` look-back words. Growing
// synchronises `stream` so no running launch still uses the old arrays.
int workspace_reserve(Workspace& ws, uint64_t tiles, cudaStream_t stream) {
  if (ws.counters == nullptr) {
    if (cudaMalloc(&ws.counters, kCounterBytes) != cudaSuccess) return PULSE_ERR_NOMEM;
    if (cudaMemsetAsync(ws.counters, 0, kCounterBytes, stream) != cudaSuccess) return PULSE_ERR_CUDA;
  }
  if (tiles > ws.capacity_tiles) {
    uint64_t cap = ws.capacity_tiles ? ws.capacity_tiles : 4096;
    while (cap < tiles) cap *= 2;
    if (ws.status != nullptr) {
      if (cudaStreamSynchronize(stream) != cudaSuccess) return PULSE_ERR_CUDA;
      cudaFree(ws.status);
      ws.status = nullptr;
      ws.capacity_tiles = 0;
    }
    if (cudaMalloc(&ws.status, cap * sizeof(uint64_t)) != cudaSuccess) return PULSE_ERR_NOMEM;
    if (cudaMemsetAsync(ws.status, 0, cap * sizeof(uint64_t), stream) != cudaSuccess)
      return PULSE_ERR_CUDA;
    ws.capacity_tiles = cap;
  }
  return PULSE_OK;
}

// Next launch epoch; when the 30-bit epoch wraps, clear the status words so
// no stale word can match a reused epoch.
int workspace_next_epoch(Workspace& ws, cudaStream_t stream, uint32_t* epoch) {
  ws.epoch += 1;
  if (ws.epoch > kEpochMask) {
    if (cudaMemsetAsync(ws.status, 0, ws.capacity_tiles * sizeof(uint64_t), stream) != cudaSuccess)
      return PULSE_ERR_CUDA;
    ws.epoch = 1;
  }
  *epoch = ws.epoch;
  return PULSE_OK;
}

void workspace_free(Workspace& ws) {
  if (ws.status) cudaFree(ws.status);
  if (ws.counters) cudaFree(ws.counters);
  ws = Workspace{};
}

// Reads and clears the error word (caller has synchronised the stream).
int workspace_take_error(Workspace& ws, cudaStream_t stream) {
  if (ws.counters == nullptr) return PULSE_OK;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, ws.counters + 2, sizeof word, cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaMemsetAsync(ws.counters + 2, 0, sizeof(uint32_t), stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  if (word & kErrTimeout) return PULSE_ERR_TIMEOUT;
  if (word & kErrIndex) return PULSE_ERR_INDEX;
  return PULSE_OK;
}

// ---- per-(device, stream) workspaces of the single-tensor entry points
std::mutex g_ws_mu;
std::map<std::pair<int, uintptr_t>, Workspace*> g_ws;

Workspace* stream_workspace(int device, cudaStream_t stream) {
  auto key = std::make_pair(device, reinterpret_cast<uintptr_t>(stream));
  auto it = g_ws.find(key);
  if (it != g_ws.end()) return it->second;
  Workspace* ws = new (std::nothrow) Workspace();
  if (ws == nullptr) return nullptr;
  ws->device = device;
  g_ws[key] = ws;
  return ws;
}

TensorDesc make_desc(const pulse_tensor& t, uint64_t tile_begin) {
  TensorDesc d{};
  d.master = t.master;
  d.prev = t.prev;
  d.w = t.w;
  d.idx = t.idx;
  d.val = t.val;
  d.mask = t.mask;
  d.n = t.n;
  d.tile_begin = tile_begin;
  d.bulk_ok = (t.master && t.prev && aligned(t.master, 16) && aligned(t.prev, 16)) ? 1u : 0u;
  d.vec_ok = 0;
  if (t.master && t.prev && t.mask && aligned(t.master, 16) && aligned(t.prev, 8) &&
      aligned(t.mask, 8))
    d.vec_ok |= kVecMask;
  if (t.w && t.mask && aligned(t.w, 8) && aligned(t.mask, 8)) d.vec_ok |= kVecApply;
  return d;
}

int xor_grid(int device, uint64_t tiles) {
  const uint64_t cap = uint64_t(sm_count(device)) * uint64_t(2048 / kXorThreads);  // 2048 threads per SM
  return int(tiles < cap ? tiles : cap);
}

int encode_impl(const float* master, uint16_t* prev, uint64_t n, uint32_t* idx, uint16_t* val,
                uint64_t* count_out, uint32_t first_ticket, uint64_t wait_ns,
                cudaStream_t stream) {
  if (n >= kMaxElems + 1) return PULSE_ERR_RANGE;
  if (count_out == nullptr) return PULSE_ERR_INVALID;
  if (n > 0 && (master == nullptr || prev == nullptr || idx == nullptr || val == nullptr))
    return PULSE_ERR_INVALID;
  if (n == 0) return cuda_status(cudaMemsetAsync(count_out, 0, sizeof(uint64_t), stream));
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  const uint64_t tiles = div_up(n, kEncTile);
  std::lock_guard<std::mutex> lock(g_ws_mu);
  Workspace* ws = stream_workspace(device, stream);
  if (ws == nullptr) return PULSE_ERR_NOMEM;
  int st = workspace_reserve(*ws, tiles, stream);
  if (st != PULSE_OK) return st;
  EncodeLaunch a{};
  pulse_tensor t{};
  t.master = master;
  t.prev = prev;
  t.n = n;
  t.idx = idx;
  t.val = val;
  a.one = make_desc(t, 0);
  a.tensors = nullptr;
  a.tile_begin = nullptr;
  a.ntensors = 1;
  a.total_tiles = tiles;
  a.status = ws->status;
  a.counters = ws->counters;
  a.counts_out = count_out;
  a.first_ticket = first_ticket;
  a.wait_limit_ns = wait_ns;
  st = workspace_next_epoch(*ws, stream, &a.epoch);
  if (st != PULSE_OK) return st;
  const uint64_t cap = uint64_t(encode_grid_size(device));
  const int grid = int(tiles < cap ? tiles : cap);
  return cuda_status(launch_encode(a, false, grid, stream));
}

// ---- MXFP8 view: workspaces of the single-tensor calls. Their status words
// use the packed layout without an epoch and are cleared before every
// launch, so they are never shared with the BF16 calls' workspaces.
std::map<std::pair<int, uintptr_t>, Workspace*> g_mx_ws;

Workspace* stream_mx_workspace(int device, cudaStream_t stream) {
  auto key = std::make_pair(device, reinterpret_cast<uintptr_t>(stream));
  auto it = g_mx_ws.find(key);
  if (it != g_mx_ws.end()) return it->second;
  Workspace* ws = new (std::nothrow) Workspace();
  if (ws == nullptr) return nullptr;
  ws->device = device;
  g_mx_ws[key] = ws;
  return ws;
}

MxTensorDesc make_mx_desc(const pulse_mx_tensor& t, uint64_t tile_begin) {
  MxTensorDesc d{};
  d.master = t.master;
  d.prev_codes = t.prev_codes;
  d.prev_scales = t.prev_scales;
  d.idx = t.idx;
  d.val = t.val;
  d.sidx = t.sidx;
  d.sval = t.sval;
  d.n = t.n;
  d.tile_begin = tile_begin;
  d.bulk_ok = (t.master && t.prev_codes && t.prev_scales && aligned(t.master, 16) &&
               aligned(t.prev_codes, 16) && aligned(t.prev_scales, 16))
                  ? 1u
                  : 0u;
  return d;
}

// Clear the status words of `tiles` tiles, then launch the MX encode.
// NVFP4 (amax_scratch: ntensors words): the tensor maxima first, into the
// scratch the encode reads.
int launch_encode_mx_ws(MxLaunch& a, int format, Workspace& ws, bool multi, int device,
                        cudaStream_t stream, uint32_t* amax_scratch = nullptr) {
  int st = workspace_reserve(ws, a.total_tiles, stream);
  if (st != PULSE_OK) return st;
  if (format == PULSE_MX_NVFP4) {
    if (amax_scratch == nullptr) amax_scratch = ws.counters + kAmaxWord;
    if (cudaMemsetAsync(amax_scratch, 0, sizeof(uint32_t) * size_t(a.ntensors), stream) !=
            cudaSuccess ||
        launch_mx_amax(a, multi, amax_scratch, stream) != cudaSuccess)
      return PULSE_ERR_CUDA;
    a.amax_bits = amax_scratch;
  }
  if (cudaMemsetAsync(ws.status, 0, a.total_tiles * sizeof(uint64_t), stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  a.status = ws.status;
  a.counters = ws.counters;
  a.epoch = 0;
  const uint64_t cap = uint64_t(encode_mx_grid_size(device, format));
  const int grid = int(a.total_tiles < cap ? a.total_tiles : cap);
  return cuda_status(launch_encode_mx(a, format, multi, grid, stream));
}

// ---- compose: per-(device, stream) workspace with the merge-path splits and
// the segment table of multi-segment calls.
struct CmpWorkspace {
  Workspace ws;
  uint32_t* splits = nullptr;
  uint64_t split_cap = 0;
  CmpSegment* segs = nullptr;
  uint64_t* tile_begin = nullptr;
  int table_cap = 0;
};
std::map<std::pair<int, uintptr_t>, CmpWorkspace*> g_cmp_ws;

CmpWorkspace* stream_cmp_workspace(int device, cudaStream_t stream) {
  auto key = std::make_pair(device, reinterpret_cast<uintptr_t>(stream));
  auto it = g_cmp_ws.find(key);
  if (it != g_cmp_ws.end()) return it->second;
  CmpWorkspace* ws = new (std::nothrow) CmpWorkspace();
  if (ws == nullptr) return nullptr;
  ws->ws.device = device;
  g_cmp_ws[key] = ws;
  return ws;
}

// Grow the split array / segment table (growth synchronises `stream`).
int cmp_reserve(CmpWorkspace& w, uint64_t tiles, int nsegs, cudaStream_t stream) {
  int st = workspace_reserve(w.ws, tiles, stream);
  if (st != PULSE_OK) return st;
  if (tiles > w.split_cap) {
    uint64_t cap = w.split_cap ? w.split_cap : 4096;
    while (cap < tiles) cap *= 2;
    if (w.splits != nullptr) {
      if (cudaStreamSynchronize(stream) != cudaSuccess) return PULSE_ERR_CUDA;
      cudaFree(w.splits);
      w.splits = nullptr;
      w.split_cap = 0;
    }
    // two words per tile: the merge-path split, and the tile's segment
    if (cudaMalloc(&w.splits, 2 * cap * sizeof(uint32_t)) != cudaSuccess) return PULSE_ERR_NOMEM;
    w.split_cap = cap;
  }
  if (nsegs > w.table_cap) {
    int cap = w.table_cap ? w.table_cap : 64;
    while (cap < nsegs) cap *= 2;
    if (w.segs != nullptr || w.tile_begin != nullptr) {
      if (cudaStreamSynchronize(stream) != cudaSuccess) return PULSE_ERR_CUDA;
      if (w.segs) cudaFree(w.segs);
      if (w.tile_begin) cudaFree(w.tile_begin);
      w.segs = nullptr;
      w.tile_begin = nullptr;
      w.table_cap = 0;
    }
    if (cudaMalloc(&w.segs, sizeof(CmpSegment) * size_t(cap)) != cudaSuccess ||
        cudaMalloc(&w.tile_begin, sizeof(uint64_t) * (size_t(cap) + 1)) != cudaSuccess)
      return PULSE_ERR_NOMEM;
    w.table_cap = cap;
  }
  return PULSE_OK;
}

int compose_one(const uint32_t* idx_a, const void* val_a, uint64_t count_a, const uint32_t* idx_b,
                const void* val_b, uint64_t count_b, uint32_t* idx_out, void* val_out,
                uint64_t* count_out, int value_bytes, cudaStream_t stream) {
  if (count_out == nullptr) return PULSE_ERR_INVALID;
  if (count_a >= kMaxElems + 1 || count_b >= kMaxElems + 1) return PULSE_ERR_RANGE;
  if ((count_a > 0 && (idx_a == nullptr || val_a == nullptr)) ||
      (count_b > 0 && (idx_b == nullptr || val_b == nullptr)) ||
      (count_a + count_b > 0 && (idx_out == nullptr || val_out == nullptr)))
    return PULSE_ERR_INVALID;
  if (count_a + count_b == 0) return cuda_status(cudaMemsetAsync(count_out, 0, sizeof(uint64_t), stream));
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  const uint64_t tiles = compose_tiles(count_a + count_b);
  if (tiles > kMaxTiles) return PULSE_ERR_RANGE;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  CmpWorkspace* w = stream_cmp_workspace(device, stream);
  if (w == nullptr) return PULSE_ERR_NOMEM;
  int st = cmp_reserve(*w, tiles, 0, stream);
  if (st != PULSE_OK) return st;
  uint32_t epoch = 0;
  st = workspace_next_epoch(w->ws, stream, &epoch);
  if (st != PULSE_OK) return st;
  CmpSegment one{idx_a, val_a, count_a, idx_b, val_b, count_b, idx_out, val_out, 0};
  return cuda_status(launch_compose(nullptr, one, nullptr, 1, tiles, w->splits,
                                    w->splits + w->split_cap, w->ws.status, w->ws.counters,
                                    count_out, epoch, kDefaultWaitNs, value_bytes, stream));
}

int take_error_pair(Workspace* a, Workspace* b, cudaStream_t stream) {
  const int ea = a ? workspace_take_error(*a, stream) : PULSE_OK;
  const int eb = b ? workspace_take_error(*b, stream) : PULSE_OK;
  if (ea == PULSE_ERR_CUDA || eb == PULSE_ERR_CUDA) return PULSE_ERR_CUDA;
  if (ea == PULSE_ERR_TIMEOUT || eb == PULSE_ERR_TIMEOUT) return PULSE_ERR_TIMEOUT;
  return ea != PULSE_OK ? ea : eb;
}

}  // namespace
}  // namespace pulse

using namespace pulse;

// ------------------------------------------------------------------ plans

struct pulse_plan {
  int device = 0;
  int ntensors = 0;
  uint64_t total_tiles = 0;
  uint64_t total_n = 0;             // elements over every tensor
  bool can_encode = false, can_apply = false, can_xor_mask = false, can_xor_apply = false;
  bool can_chain = false;  // every tensor with n > 0 has w: chained applies are possible
  std::vector<TensorDesc> host_desc;
  TensorDesc* desc = nullptr;       // device copy
  uint64_t* tile_begin = nullptr;   // device, ntensors + 1
  uint64_t* counts = nullptr;       // device, ntensors (host-count apply staging)
  // chunk-owned apply: chunk tables (built once) and the per-call partition
  uint64_t total_chunks = 0;
  uint64_t* chunk_begin = nullptr;  // device, ntensors + 1
  uint32_t* chunk_tensor = nullptr; // device, total_chunks
  // chained apply: per-call patch table and partition scratch (grown on demand)
  ChainSeg* chain_segs = nullptr;   // device, chain_seg_cap entries
  uint64_t chain_seg_cap = 0;
  uint32_t* chain_first = nullptr;  // device, kChainMaxVersions x total_chunks (first use)
  CcOut* cc_outs = nullptr;         // device, ntensors (first k-way compose)
  Workspace ws;
};

struct pulse_loco_plan {
  int device = 0;
  int ntensors = 0;
  uint64_t total_tiles = 0;
  bool can_gate = false, can_accumulate = false;
  LocoTensorDesc* desc = nullptr;   // device
  uint64_t* tile_begin = nullptr;   // device, ntensors + 1
  Workspace ws;
};

struct pulse_mx_plan {
  int device = 0;
  int format = PULSE_MX_E4M3;
  uint32_t* amax = nullptr;         // NVFP4: device, ntensors (tensor maxima)
  int ntensors = 0;
  uint64_t total_tiles = 0;
  bool can_encode = false, can_apply = false;
  std::vector<MxTensorDesc> host_desc;
  MxTensorDesc* desc = nullptr;     // device copy
  uint64_t* tile_begin = nullptr;   // device, ntensors + 1
  ByteSegment* segs = nullptr;      // device, 2 x ntensors: codes then scales of each tensor
  uint64_t* counts = nullptr;       // device, 2 x ntensors (host-count apply staging)
  Workspace ws;
};

extern "C" {

const char* pulse_error_string(int status) {
  switch (status) {
    case PULSE_OK: return "PULSE_OK";
    case PULSE_ERR_INVALID: return "PULSE_ERR_INVALID: invalid argument";
    case PULSE_ERR_RANGE:
      return "PULSE_ERR_RANGE: element count past the entry point's limit (2^32 - 1, or "
             "PULSE_NOALLOC_MAX_ELEMS for pulse_encode_noalloc)";
    case PULSE_ERR_CUDA: return "PULSE_ERR_CUDA: CUDA runtime call or launch failed";
    case PULSE_ERR_TIMEOUT: return "PULSE_ERR_TIMEOUT: a bounded device wait gave up";
    case PULSE_ERR_INDEX: return "PULSE_ERR_INDEX: patch index out of range (entry skipped)";
    case PULSE_ERR_NOMEM: return "PULSE_ERR_NOMEM: workspace allocation failed";
    default: return "PULSE_ERR_UNKNOWN";
  }
}

uint32_t pulse_encode_tile_elems(void) { return uint32_t(kEncTile); }

int pulse_encode(const float* master_f32, uint16_t* prev_bf16, uint64_t n, uint32_t* idx_out,
                 uint16_t* val_out, uint64_t* count_out, cudaStream_t stream) {
  return encode_impl(master_f32, prev_bf16, n, idx_out, val_out, count_out, 0u, kDefaultWaitNs,
                     stream);
}

int pulse_debug_encode_orphan_tile(const float* master_f32, uint16_t* prev_bf16, uint64_t n,
                                   uint32_t* idx_out, uint16_t* val_out, uint64_t* count_out,
                                   uint64_t wait_limit_ns, cudaStream_t stream) {
  if (n <= uint64_t(kEncTile)) return PULSE_ERR_INVALID;
  return encode_impl(master_f32, prev_bf16, n, idx_out, val_out, count_out, 1u, wait_limit_ns,
                     stream);
}

int pulse_apply(uint16_t* w_bf16, const uint32_t* idx, const uint16_t* val, uint64_t count,
                cudaStream_t stream) {
  if (count == 0) return PULSE_OK;
  if (w_bf16 == nullptr || idx == nullptr || val == nullptr) return PULSE_ERR_INVALID;
  return cuda_status(launch_apply(w_bf16, 0, false, idx, val, count, nullptr, stream));
}

int pulse_apply_checked(uint16_t* w_bf16, uint64_t n, const uint32_t* idx, const uint16_t* val,
                        uint64_t count, cudaStream_t stream) {
  if (count == 0) return PULSE_OK;
  if (w_bf16 == nullptr || idx == nullptr || val == nullptr) return PULSE_ERR_INVALID;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  uint32_t* err = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    Workspace* ws = stream_workspace(device, stream);
    if (ws == nullptr) return PULSE_ERR_NOMEM;
    const int st = workspace_reserve(*ws, 0, stream);
    if (st != PULSE_OK) return st;
    err = ws->counters + 2;
  }
  return cuda_status(launch_apply(w_bf16, n, true, idx, val, count, err, stream));
}

int pulse_xor_mask(const float* master_f32, uint16_t* prev_bf16, uint64_t n, uint16_t* mask_out,
                   cudaStream_t stream) {
  if (n >= kMaxElems + 1) return PULSE_ERR_RANGE;
  if (n == 0) return PULSE_OK;
  if (master_f32 == nullptr || prev_bf16 == nullptr || mask_out == nullptr) return PULSE_ERR_INVALID;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  pulse_tensor t{};
  t.master = master_f32;
  t.prev = prev_bf16;
  t.mask = mask_out;
  t.n = n;
  const TensorDesc d = make_desc(t, 0);
  const uint64_t tiles = div_up(n, kXorTile);
  return cuda_status(launch_xor_mask(d, nullptr, nullptr, 1, tiles, false, xor_grid(device, tiles), stream));
}

int pulse_xor_apply(uint16_t* w_bf16, const uint16_t* mask, uint64_t n, cudaStream_t stream) {
  if (n >= kMaxElems + 1) return PULSE_ERR_RANGE;
  if (n == 0) return PULSE_OK;
  if (w_bf16 == nullptr || mask == nullptr) return PULSE_ERR_INVALID;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  pulse_tensor t{};
  t.w = w_bf16;
  t.mask = const_cast<uint16_t*>(mask);
  t.n = n;
  const TensorDesc d = make_desc(t, 0);
  const uint64_t tiles = div_up(n, kXorTile);
  return cuda_status(launch_xor_apply(d, nullptr, nullptr, 1, tiles, false, xor_grid(device, tiles), stream));
}

int pulse_get_error(cudaStream_t stream) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PULSE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  const auto key = std::make_pair(device, reinterpret_cast<uintptr_t>(stream));
  auto it = g_ws.find(key);
  auto mt = g_mx_ws.find(key);
  auto ct = g_cmp_ws.find(key);
  const int e1 = take_error_pair(it == g_ws.end() ? nullptr : it->second,
                                 mt == g_mx_ws.end() ? nullptr : mt->second, stream);
  const int e2 = take_error_pair(ct == g_cmp_ws.end() ? nullptr : &ct->second->ws, nullptr, stream);
  if (e1 == PULSE_ERR_CUDA || e2 == PULSE_ERR_CUDA) return PULSE_ERR_CUDA;
  if (e1 == PULSE_ERR_TIMEOUT || e2 == PULSE_ERR_TIMEOUT) return PULSE_ERR_TIMEOUT;
  return e1 != PULSE_OK ? e1 : e2;
}

int pulse_plan_create(const pulse_tensor* tensors, int ntensors, pulse_plan** plan_out) {
  if (plan_out == nullptr) return PULSE_ERR_INVALID;
  *plan_out = nullptr;
  if (tensors == nullptr || ntensors < 1) return PULSE_ERR_INVALID;
  pulse_plan* p = new (std::nothrow) pulse_plan();
  if (p == nullptr) return PULSE_ERR_NOMEM;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return PULSE_ERR_CUDA;
  }
  p->ntensors = ntensors;
  p->can_encode = p->can_apply = p->can_xor_mask = p->can_xor_apply = p->can_chain = true;
  std::vector<uint64_t> tb(size_t(ntensors) + 1, 0);
  p->host_desc.reserve(size_t(ntensors));
  uint64_t tiles = 0;
  for (int i = 0; i < ntensors; ++i) {
    const pulse_tensor& t = tensors[i];
    if (t.n >= kMaxElems + 1) {
      delete p;
      return PULSE_ERR_RANGE;
    }
    tb[size_t(i)] = tiles;
    p->host_desc.push_back(make_desc(t, tiles));
    tiles += div_up(t.n, kEncTile);
    p->total_n += t.n;
    if (t.n > 0) {
      p->can_encode = p->can_encode && t.master && t.prev && t.idx && t.val;
      p->can_apply = p->can_apply && t.w && t.idx && t.val;
      p->can_chain = p->can_chain && t.w;
      p->can_xor_mask = p->can_xor_mask && t.master && t.prev && t.mask;
      p->can_xor_apply = p->can_xor_apply && t.w && t.mask;
    }
  }
  tb[size_t(ntensors)] = tiles;
  if (tiles > kMaxTiles) {
    delete p;
    return PULSE_ERR_RANGE;
  }
  p->total_tiles = tiles;
  const size_t desc_bytes = sizeof(TensorDesc) * size_t(ntensors);
  const size_t tb_bytes = sizeof(uint64_t) * (size_t(ntensors) + 1);
  int st = PULSE_OK;
  if (cudaMalloc(&p->desc, desc_bytes) != cudaSuccess ||
      cudaMalloc(&p->tile_begin, tb_bytes) != cudaSuccess ||
      cudaMalloc(&p->counts, sizeof(uint64_t) * size_t(ntensors)) != cudaSuccess) {
    st = PULSE_ERR_NOMEM;
  } else if (cudaMemcpy(p->desc, p->host_desc.data(), desc_bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(p->tile_begin, tb.data(), tb_bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemset(p->counts, 0, sizeof(uint64_t) * size_t(ntensors)) != cudaSuccess) {
    st = PULSE_ERR_CUDA;
  } else {
    st = workspace_reserve(p->ws, tiles, nullptr);
  }
  if (st == PULSE_OK) {
    // chunk tables of the chained apply and the k-way compose
    std::vector<uint64_t> cb(size_t(ntensors) + 1, 0);
    uint64_t chunks = 0;
    for (int i = 0; i < ntensors; ++i) {
      cb[size_t(i)] = chunks;
      chunks += div_up(tensors[i].n, uint64_t(kApplyChunk));
    }
    cb[size_t(ntensors)] = chunks;
    std::vector<uint32_t> ct(size_t(chunks > 0 ? chunks : 1), 0);
    for (int i = 0; i < ntensors; ++i)
      for (uint64_t g = cb[size_t(i)]; g < cb[size_t(i) + 1]; ++g) ct[size_t(g)] = uint32_t(i);
    p->total_chunks = chunks;
    if (cudaMalloc(&p->chunk_begin, sizeof(uint64_t) * cb.size()) != cudaSuccess ||
        cudaMalloc(&p->chunk_tensor, sizeof(uint32_t) * ct.size()) != cudaSuccess) {
      st = PULSE_ERR_NOMEM;
    } else if (cudaMemcpy(p->chunk_begin, cb.data(), sizeof(uint64_t) * cb.size(),
                          cudaMemcpyHostToDevice) != cudaSuccess ||
               cudaMemcpy(p->chunk_tensor, ct.data(), sizeof(uint32_t) * ct.size(),
                          cudaMemcpyHostToDevice) != cudaSuccess) {
      st = PULSE_ERR_CUDA;
    }
  }
  if (st == PULSE_OK && cudaDeviceSynchronize() != cudaSuccess) st = PULSE_ERR_CUDA;
  if (st != PULSE_OK) {
    pulse_plan_destroy(p);
    return st;
  }
  *plan_out = p;
  return PULSE_OK;
}

int pulse_plan_destroy(pulse_plan* plan) {
  if (plan == nullptr) return PULSE_OK;
  const cudaError_t e = cudaDeviceSynchronize();
  if (plan->desc) cudaFree(plan->desc);
  if (plan->tile_begin) cudaFree(plan->tile_begin);
  if (plan->counts) cudaFree(plan->counts);
  if (plan->chunk_begin) cudaFree(plan->chunk_begin);
  if (plan->chunk_tensor) cudaFree(plan->chunk_tensor);
  if (plan->chain_segs) cudaFree(plan->chain_segs);
  if (plan->chain_first) cudaFree(plan->chain_first);
  if (plan->cc_outs) cudaFree(plan->cc_outs);
  workspace_free(plan->ws);
  delete plan;
  return cuda_status(e);
}

int pulse_plan_num_tensors(const pulse_plan* plan) { return plan ? plan->ntensors : 0; }

uint64_t pulse_plan_num_tiles(const pulse_plan* plan) { return plan ? plan->total_tiles : 0; }

int pulse_encode_multi(pulse_plan* plan, uint64_t* counts_out, cudaStream_t stream) {
  if (plan == nullptr || counts_out == nullptr || !plan->can_encode) return PULSE_ERR_INVALID;
  if (plan->total_tiles == 0)
    return cuda_status(cudaMemsetAsync(counts_out, 0, sizeof(uint64_t) * size_t(plan->ntensors), stream));
  EncodeLaunch a{};
  a.tensors = plan->desc;
  a.tile_begin = plan->tile_begin;
  a.ntensors = plan->ntensors;
  a.total_tiles = plan->total_tiles;
  a.status = plan->ws.status;
  a.counters = plan->ws.counters;
  a.counts_out = counts_out;
  a.first_ticket = 0;
  a.wait_limit_ns = kDefaultWaitNs;
  const int st = workspace_next_epoch(plan->ws, stream, &a.epoch);
  if (st != PULSE_OK) return st;
  const uint64_t cap = uint64_t(encode_grid_size(plan->device));
  const int grid = int(plan->total_tiles < cap ? plan->total_tiles : cap);
  return cuda_status(launch_encode(a, true, grid, stream));
}

namespace {
// Whole-model apply: the entry scatter over every segment, in groups of at
// most kMaxTensorsPerApplyLaunch tensors per launch.
int apply_multi_launch(pulse_plan* plan, const uint64_t* counts_dev, cudaStream_t stream) {
  const int grid = sm_count(plan->device) * 8;
  for (int t0 = 0; t0 < plan->ntensors; t0 += kMaxTensorsPerApplyLaunch) {
    const int nt = plan->ntensors - t0 < kMaxTensorsPerApplyLaunch ? plan->ntensors - t0
                                                                   : kMaxTensorsPerApplyLaunch;
    const cudaError_t e = launch_apply_multi(plan->desc + t0, nt, counts_dev + t0,
                                             plan->ws.counters + 2, grid, stream);
    if (e != cudaSuccess) return PULSE_ERR_CUDA;
  }
  return PULSE_OK;
}
}  // namespace

int pulse_apply_multi_device(pulse_plan* plan, const uint64_t* counts_dev, cudaStream_t stream) {
  if (plan == nullptr || counts_dev == nullptr || !plan->can_apply) return PULSE_ERR_INVALID;
  return apply_multi_launch(plan, counts_dev, stream);
}

int pulse_apply_multi(pulse_plan* plan, const uint64_t* counts_host, cudaStream_t stream) {
  if (plan == nullptr || counts_host == nullptr || !plan->can_apply) return PULSE_ERR_INVALID;
  // From pageable memory the copy is staged before this call returns, so the
  // caller may reuse counts_host at once.
  if (cudaMemcpyAsync(plan->counts, counts_host, sizeof(uint64_t) * size_t(plan->ntensors),
                      cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  return apply_multi_launch(plan, plan->counts, stream);
}

namespace {
// Check a chain's host references and upload them into the plan's table
// (growth synchronises `stream`); allocates the partition scratch on first use.
int upload_chain(pulse_plan* plan, const pulse_patch_ref* patches, int nversions,
                 cudaStream_t stream) {
  const uint64_t nseg = uint64_t(nversions) * uint64_t(plan->ntensors);
  std::vector<ChainSeg> segs(static_cast<size_t>(nseg));
  for (uint64_t i = 0; i < nseg; ++i) {
    const pulse_patch_ref& r = patches[i];
    if (r.count >= kMaxElems + 1) return PULSE_ERR_RANGE;
    if (r.count > 0 && (r.idx == nullptr || r.val == nullptr)) return PULSE_ERR_INVALID;
    segs[size_t(i)] = ChainSeg{r.idx, r.val, r.count};
  }
  if (plan->total_chunks == 0) return PULSE_OK;
  // grow the patch table; replacing a buffer waits for the work that reads it
  if (nseg > plan->chain_seg_cap) {
    uint64_t cap = plan->chain_seg_cap ? plan->chain_seg_cap : 256;
    while (cap < nseg) cap *= 2;
    if (plan->chain_segs != nullptr) {
      if (cudaStreamSynchronize(stream) != cudaSuccess) return PULSE_ERR_CUDA;
      cudaFree(plan->chain_segs);
      plan->chain_segs = nullptr;
      plan->chain_seg_cap = 0;
    }
    if (cudaMalloc(&plan->chain_segs, sizeof(ChainSeg) * size_t(cap)) != cudaSuccess)
      return PULSE_ERR_NOMEM;
    plan->chain_seg_cap = cap;
  }
  if (plan->chain_first == nullptr &&
      cudaMalloc(&plan->chain_first, sizeof(uint32_t) * size_t(plan->total_chunks) *
                                         size_t(kChainMaxVersions)) != cudaSuccess)
    return PULSE_ERR_NOMEM;
  // from pageable memory the copy is staged before this call returns
  if (cudaMemcpyAsync(plan->chain_segs, segs.data(), sizeof(ChainSeg) * size_t(nseg),
                      cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  return PULSE_OK;
}
}  // namespace

int pulse_apply_chain_multi(pulse_plan* plan, const pulse_patch_ref* patches, int nversions,
                            cudaStream_t stream) {
  if (plan == nullptr || patches == nullptr || nversions < 1 || !plan->can_chain)
    return PULSE_ERR_INVALID;
  const int st = upload_chain(plan, patches, nversions, stream);
  if (st != PULSE_OK || plan->total_chunks == 0) return st;
  for (int v0 = 0; v0 < nversions; v0 += kChainMaxVersions) {
    const int nv = nversions - v0 < kChainMaxVersions ? nversions - v0 : kChainMaxVersions;
    const cudaError_t e = launch_apply_chain(
        plan->desc, plan->chunk_begin, plan->chunk_tensor, plan->chain_first,
        plan->chain_segs + size_t(v0) * size_t(plan->ntensors), plan->ntensors, nv,
        plan->total_chunks, plan->ws.counters + 2, kDefaultWaitNs, stream);
    if (e != cudaSuccess) return PULSE_ERR_CUDA;
  }
  return PULSE_OK;
}

int pulse_compose_chain_multi(pulse_plan* plan, const pulse_patch_ref* patches, int nversions,
                              const pulse_patch_out* outs, uint64_t* counts_out,
                              cudaStream_t stream) {
  if (plan == nullptr || patches == nullptr || outs == nullptr || counts_out == nullptr ||
      nversions < 1 || nversions > kChainMaxVersions)
    return PULSE_ERR_INVALID;
  const int nt = plan->ntensors;
  std::vector<CcOut> table(static_cast<size_t>(nt));
  for (int t = 0; t < nt; ++t) {
    // the composed segment holds at most min(n, sum of the versions' counts)
    const uint64_t n = plan->host_desc[size_t(t)].n;
    uint64_t need = 0;
    for (int v = 0; v < nversions; ++v) {
      const uint64_t c = patches[size_t(v) * size_t(nt) + size_t(t)].count;
      need += c < n ? c : n;
    }
    if (need > n) need = n;
    const pulse_patch_out& o = outs[t];
    if (o.room < need || (need > 0 && (o.idx == nullptr || o.val == nullptr)))
      return PULSE_ERR_INVALID;
    table[size_t(t)] = CcOut{o.idx, o.val, o.room};
  }
  int st = upload_chain(plan, patches, nversions, stream);
  if (st != PULSE_OK) return st;
  // tensors without chunks (n == 0) keep a count of 0; the others are
  // written by their last chunk
  if (cudaMemsetAsync(counts_out, 0, sizeof(uint64_t) * size_t(nt), stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  if (plan->total_chunks == 0) return PULSE_OK;
  if (plan->cc_outs == nullptr &&
      cudaMalloc(&plan->cc_outs, sizeof(CcOut) * size_t(nt)) != cudaSuccess)
    return PULSE_ERR_NOMEM;
  if (cudaMemcpyAsync(plan->cc_outs, table.data(), sizeof(CcOut) * size_t(nt),
                      cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  if (launch_chain_partition(plan->desc, plan->chunk_begin, plan->chunk_tensor, plan->chain_segs,
                             nt, nversions, plan->total_chunks, plan->chain_first,
                             plan->ws.counters + 2, stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  CcArgs a{};
  a.tensors = plan->desc;
  a.chunk_begin = plan->chunk_begin;
  a.chunk_tensor = plan->chunk_tensor;
  a.first = plan->chain_first;
  a.segs = plan->chain_segs;
  a.outs = plan->cc_outs;
  a.counts_out = counts_out;
  a.ntensors = nt;
  a.nversions = nversions;
  a.total_chunks = plan->total_chunks;
  a.status = plan->ws.status;
  a.counters = plan->ws.counters;
  a.wait_limit_ns = kDefaultWaitNs;
  st = workspace_next_epoch(plan->ws, stream, &a.epoch);
  if (st != PULSE_OK) return st;
  return cuda_status(launch_compose_chunks(a, stream));
}

int pulse_xor_mask_multi(pulse_plan* plan, cudaStream_t stream) {
  if (plan == nullptr || !plan->can_xor_mask) return PULSE_ERR_INVALID;
  if (plan->total_tiles == 0) return PULSE_OK;
  return cuda_status(launch_xor_mask(plan->host_desc[0], plan->desc, plan->tile_begin,
                                     plan->ntensors, plan->total_tiles, true,
                                     xor_grid(plan->device, plan->total_tiles), stream));
}

int pulse_xor_apply_multi(pulse_plan* plan, cudaStream_t stream) {
  if (plan == nullptr || !plan->can_xor_apply) return PULSE_ERR_INVALID;
  if (plan->total_tiles == 0) return PULSE_OK;
  return cuda_status(launch_xor_apply(plan->host_desc[0], plan->desc, plan->tile_begin,
                                      plan->ntensors, plan->total_tiles, true,
                                      xor_grid(plan->device, plan->total_tiles), stream));
}

int pulse_plan_get_error(pulse_plan* plan) {
  if (plan == nullptr) return PULSE_ERR_INVALID;
  if (cudaDeviceSynchronize() != cudaSuccess) return PULSE_ERR_CUDA;
  return workspace_take_error(plan->ws, nullptr);
}

// ------------------------------------------------------------ PULSELoCo

namespace {
LocoTensorDesc make_loco_desc(const pulse_loco_tensor& t, uint64_t tile_begin) {
  LocoTensorDesc d{};
  d.global = t.global_w;
  d.local = t.local_w;
  d.err = t.err;
  d.idx = t.idx;
  d.val = t.val;
  d.acc = t.acc;
  d.n = t.n;
  d.tile_begin = tile_begin;
  d.bulk_ok = (t.global_w && t.local_w && t.err && aligned(t.global_w, 16) &&
               aligned(t.local_w, 16) && aligned(t.err, 16))
                  ? 1u
                  : 0u;
  return d;
}
}  // namespace

int pulse_loco_gate(const float* global_w, const float* local_w, float* err, uint64_t n,
                    uint32_t* idx_out, float* val_out, uint64_t* count_out, cudaStream_t stream) {
  if (n >= kMaxElems + 1) return PULSE_ERR_RANGE;
  if (count_out == nullptr) return PULSE_ERR_INVALID;
  if (n > 0 && (global_w == nullptr || local_w == nullptr || err == nullptr || idx_out == nullptr ||
                val_out == nullptr))
    return PULSE_ERR_INVALID;
  if (n == 0) return cuda_status(cudaMemsetAsync(count_out, 0, sizeof(uint64_t), stream));
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  const uint64_t tiles = loco_tiles(n);
  std::lock_guard<std::mutex> lock(g_ws_mu);
  Workspace* ws = stream_workspace(device, stream);
  if (ws == nullptr) return PULSE_ERR_NOMEM;
  int st = workspace_reserve(*ws, tiles, stream);
  if (st != PULSE_OK) return st;
  pulse_loco_tensor t{};
  t.global_w = global_w;
  t.local_w = local_w;
  t.err = err;
  t.n = n;
  t.idx = idx_out;
  t.val = val_out;
  LocoLaunch a{};
  a.one = make_loco_desc(t, 0);
  a.ntensors = 1;
  a.total_tiles = tiles;
  a.status = ws->status;
  a.counters = ws->counters;
  a.counts_out = count_out;
  a.wait_limit_ns = kDefaultWaitNs;
  st = workspace_next_epoch(*ws, stream, &a.epoch);
  if (st != PULSE_OK) return st;
  const uint64_t cap = uint64_t(loco_grid_size(device));
  return cuda_status(launch_loco_gate(a, false, int(tiles < cap ? tiles : cap), stream));
}

int pulse_loco_accumulate(float* acc, uint64_t n, const uint32_t* idx, const float* val,
                          uint64_t count, cudaStream_t stream) {
  if (n >= kMaxElems + 1) return PULSE_ERR_RANGE;
  if (count == 0) return PULSE_OK;
  if (acc == nullptr || idx == nullptr || val == nullptr) return PULSE_ERR_INVALID;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  uint32_t* err = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    Workspace* ws = stream_workspace(device, stream);
    if (ws == nullptr) return PULSE_ERR_NOMEM;
    const int st = workspace_reserve(*ws, 0, stream);
    if (st != PULSE_OK) return st;
    err = ws->counters + 2;
  }
  return cuda_status(launch_loco_accumulate(acc, n, idx, val, count, err, stream));
}

int pulse_loco_plan_create(const pulse_loco_tensor* tensors, int ntensors, pulse_loco_plan** plan_out) {
  if (plan_out == nullptr) return PULSE_ERR_INVALID;
  *plan_out = nullptr;
  if (tensors == nullptr || ntensors < 1 || ntensors > kMaxTensorsPerApplyLaunch) return PULSE_ERR_INVALID;
  pulse_loco_plan* p = new (std::nothrow) pulse_loco_plan();
  if (p == nullptr) return PULSE_ERR_NOMEM;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return PULSE_ERR_CUDA;
  }
  p->ntensors = ntensors;
  p->can_gate = p->can_accumulate = true;
  std::vector<LocoTensorDesc> desc;
  std::vector<uint64_t> tb(size_t(ntensors) + 1, 0);
  uint64_t tiles = 0;
  for (int i = 0; i < ntensors; ++i) {
    const pulse_loco_tensor& t = tensors[i];
    if (t.n >= kMaxElems + 1) {
      delete p;
      return PULSE_ERR_RANGE;
    }
    tb[size_t(i)] = tiles;
    desc.push_back(make_loco_desc(t, tiles));
    tiles += loco_tiles(t.n);
    if (t.n > 0) {
      p->can_gate = p->can_gate && t.global_w && t.local_w && t.err && t.idx && t.val;
      p->can_accumulate = p->can_accumulate && t.acc && t.idx && t.val;
    }
  }
  tb[size_t(ntensors)] = tiles;
  if (tiles > kMaxTiles) {
    delete p;
    return PULSE_ERR_RANGE;
  }
  p->total_tiles = tiles;
  int st = PULSE_OK;
  if (cudaMalloc(&p->desc, sizeof(LocoTensorDesc) * desc.size()) != cudaSuccess ||
      cudaMalloc(&p->tile_begin, sizeof(uint64_t) * tb.size()) != cudaSuccess) {
    st = PULSE_ERR_NOMEM;
  } else if (cudaMemcpy(p->desc, desc.data(), sizeof(LocoTensorDesc) * desc.size(),
                        cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(p->tile_begin, tb.data(), sizeof(uint64_t) * tb.size(),
                        cudaMemcpyHostToDevice) != cudaSuccess) {
    st = PULSE_ERR_CUDA;
  } else {
    st = workspace_reserve(p->ws, tiles, nullptr);
    if (st == PULSE_OK && cudaDeviceSynchronize() != cudaSuccess) st = PULSE_ERR_CUDA;
  }
  if (st != PULSE_OK) {
    pulse_loco_plan_destroy(p);
    return st;
  }
  *plan_out = p;
  return PULSE_OK;
}

int pulse_loco_plan_destroy(pulse_loco_plan* plan) {
  if (plan == nullptr) return PULSE_OK;
  const cudaError_t e = cudaDeviceSynchronize();
  if (plan->desc) cudaFree(plan->desc);
  if (plan->tile_begin) cudaFree(plan->tile_begin);
  workspace_free(plan->ws);
  delete plan;
  return cuda_status(e);
}

int pulse_loco_gate_multi(pulse_loco_plan* plan, uint64_t* counts_out, cudaStream_t stream) {
  if (plan == nullptr || counts_out == nullptr || !plan->can_gate) return PULSE_ERR_INVALID;
  if (plan->total_tiles == 0)
    return cuda_status(cudaMemsetAsync(counts_out, 0, sizeof(uint64_t) * size_t(plan->ntensors), stream));
  LocoLaunch a{};
  a.tensors = plan->desc;
  a.tile_begin = plan->tile_begin;
  a.ntensors = plan->ntensors;
  a.total_tiles = plan->total_tiles;
  a.status = plan->ws.status;
  a.counters = plan->ws.counters;
  a.counts_out = counts_out;
  a.wait_limit_ns = kDefaultWaitNs;
  const int st = workspace_next_epoch(plan->ws, stream, &a.epoch);
  if (st != PULSE_OK) return st;
  const uint64_t cap = uint64_t(loco_grid_size(plan->device));
  return cuda_status(launch_loco_gate(a, true, int(plan->total_tiles < cap ? plan->total_tiles : cap), stream));
}

int pulse_loco_accumulate_multi(pulse_loco_plan* plan, const uint64_t* counts_dev, cudaStream_t stream) {
  if (plan == nullptr || counts_dev == nullptr || !plan->can_accumulate) return PULSE_ERR_INVALID;
  return cuda_status(launch_loco_accumulate_multi(plan->desc, plan->ntensors, counts_dev,
                                                  plan->ws.counters + 2, sm_count(plan->device) * 8,
                                                  stream));
}

int pulse_loco_plan_get_error(pulse_loco_plan* plan) {
  if (plan == nullptr) return PULSE_ERR_INVALID;
  if (cudaDeviceSynchronize() != cudaSuccess) return PULSE_ERR_CUDA;
  return workspace_take_error(plan->ws, nullptr);
}

// ------------------------------------------------------------ index packing

int pulse_pack_indices(const uint32_t* idx, uint64_t count, uint32_t* firsts, uint8_t* widths,
                       uint64_t* chunk_off, uint8_t* payload, uint64_t* payload_bytes,
                       cudaStream_t stream) {
  if (count >= kMaxElems + 1) return PULSE_ERR_RANGE;
  if (payload_bytes == nullptr) return PULSE_ERR_INVALID;
  if (count > 0 && (idx == nullptr || firsts == nullptr || widths == nullptr ||
                    chunk_off == nullptr || payload == nullptr))
    return PULSE_ERR_INVALID;
  if (count > 0 && !aligned(payload, 16)) return PULSE_ERR_INVALID;
  if (count == 0) return cuda_status(cudaMemsetAsync(payload_bytes, 0, sizeof(uint64_t), stream));
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  const uint64_t chunks = pack_chunks(count);
  std::lock_guard<std::mutex> lock(g_ws_mu);
  Workspace* ws = stream_workspace(device, stream);
  if (ws == nullptr) return PULSE_ERR_NOMEM;
  int st = workspace_reserve(*ws, chunks, stream);
  if (st != PULSE_OK) return st;
  uint32_t epoch = 0;
  st = workspace_next_epoch(*ws, stream, &epoch);
  if (st != PULSE_OK) return st;
  return cuda_status(launch_pack(idx, count, firsts, widths, chunk_off, payload, payload_bytes,
                                 ws->status, ws->counters, epoch, kDefaultWaitNs, stream));
}

int pulse_unpack_indices(const uint32_t* firsts, const uint8_t* widths, const uint64_t* chunk_off,
                         const uint8_t* payload, uint64_t count, uint32_t* idx_out,
                         cudaStream_t stream) {
  if (count >= kMaxElems + 1) return PULSE_ERR_RANGE;
  if (count == 0) return PULSE_OK;
  if (firsts == nullptr || widths == nullptr || chunk_off == nullptr || payload == nullptr ||
      idx_out == nullptr)
    return PULSE_ERR_INVALID;
  if (!aligned(payload, 4)) return PULSE_ERR_INVALID;
  return cuda_status(launch_unpack(firsts, widths, chunk_off, payload, count, idx_out, stream));
}

namespace {
// Segment tables of the multi-segment pack calls, per (device, stream); the
// look-back scratch is the stream's encode workspace.
struct PackTables {
  PackSegment* segs = nullptr;
  uint64_t* begin = nullptr;
  int cap = 0;
};
std::map<std::pair<int, uintptr_t>, PackTables*> g_pack_tables;

// Check a host segment table, build the device-side one and the chunk
// offsets; `unpack` selects the unpack alignment rule.
int pack_table(const pulse_pack_segment* segs, int nsegs, uint64_t* payload_bytes, bool unpack,
               std::vector<PackSegment>& table, std::vector<uint64_t>& begin) {
  if (segs == nullptr || nsegs < 1) return PULSE_ERR_INVALID;
  table.resize(static_cast<size_t>(nsegs));
  begin.resize(static_cast<size_t>(nsegs) + 1);
  uint64_t chunks = 0;
  for (int i = 0; i < nsegs; ++i) {
    const pulse_pack_segment& g = segs[i];
    if (g.count >= kMaxElems + 1) return PULSE_ERR_RANGE;
    if (g.count > 0 && (g.idx == nullptr || g.firsts == nullptr || g.widths == nullptr ||
                        g.chunk_off == nullptr || g.payload == nullptr))
      return PULSE_ERR_INVALID;
    if (g.count > 0 && !aligned(g.payload, unpack ? 4 : 16)) return PULSE_ERR_INVALID;
    begin[size_t(i)] = chunks;
    table[size_t(i)] = PackSegment{g.idx,     g.count,   g.firsts,
                                   g.widths,  g.chunk_off, g.payload,
                                   payload_bytes == nullptr ? nullptr : payload_bytes + i, chunks};
    chunks += pack_chunks(g.count);
  }
  begin[size_t(nsegs)] = chunks;
  return chunks > kMaxTiles ? PULSE_ERR_RANGE : PULSE_OK;
}

// Upload the tables (growth synchronises `stream`).
int pack_upload(int device, cudaStream_t stream, const std::vector<PackSegment>& table,
                const std::vector<uint64_t>& begin, PackTables** out) {
  auto key = std::make_pair(device, reinterpret_cast<uintptr_t>(stream));
  PackTables*& t = g_pack_tables[key];
  if (t == nullptr) t = new (std::nothrow) PackTables();
  if (t == nullptr) return PULSE_ERR_NOMEM;
  const int nsegs = int(table.size());
  if (nsegs > t->cap) {
    int cap = t->cap ? t->cap : 64;
    while (cap < nsegs) cap *= 2;
    if (t->segs != nullptr || t->begin != nullptr) {
      if (cudaStreamSynchronize(stream) != cudaSuccess) return PULSE_ERR_CUDA;
      if (t->segs) cudaFree(t->segs);
      if (t->begin) cudaFree(t->begin);
      t->segs = nullptr;
      t->begin = nullptr;
      t->cap = 0;
    }
    if (cudaMalloc(&t->segs, sizeof(PackSegment) * size_t(cap)) != cudaSuccess ||
        cudaMalloc(&t->begin, sizeof(uint64_t) * (size_t(cap) + 1)) != cudaSuccess)
      return PULSE_ERR_NOMEM;
    t->cap = cap;
  }
  // (copies from pageable memory are staged before cudaMemcpyAsync returns)
  if (cudaMemcpyAsync(t->segs, table.data(), sizeof(PackSegment) * table.size(),
                      cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(t->begin, begin.data(), sizeof(uint64_t) * begin.size(),
                      cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  *out = t;
  return PULSE_OK;
}
}  // namespace

int pulse_pack_indices_multi(const pulse_pack_segment* segs, int nsegs, uint64_t* payload_bytes,
                             cudaStream_t stream) {
  if (payload_bytes == nullptr) return PULSE_ERR_INVALID;
  std::vector<PackSegment> table;
  std::vector<uint64_t> begin;
  int st = pack_table(segs, nsegs, payload_bytes, false, table, begin);
  if (st != PULSE_OK) return st;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  // empty segments have no chunk: their size is 0; the others are written
  // by their last chunk
  if (cudaMemsetAsync(payload_bytes, 0, sizeof(uint64_t) * size_t(nsegs), stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  const uint64_t chunks = begin.back();
  if (chunks == 0) return PULSE_OK;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  Workspace* ws = stream_workspace(device, stream);
  if (ws == nullptr) return PULSE_ERR_NOMEM;
  st = workspace_reserve(*ws, chunks, stream);
  if (st != PULSE_OK) return st;
  PackTables* t = nullptr;
  st = pack_upload(device, stream, table, begin, &t);
  if (st != PULSE_OK) return st;
  uint32_t epoch = 0;
  st = workspace_next_epoch(*ws, stream, &epoch);
  if (st != PULSE_OK) return st;
  return cuda_status(launch_pack_multi(t->segs, t->begin, nsegs, chunks, ws->status, ws->counters,
                                       epoch, kDefaultWaitNs, stream));
}

int pulse_unpack_indices_multi(const pulse_pack_segment* segs, int nsegs, cudaStream_t stream) {
  std::vector<PackSegment> table;
  std::vector<uint64_t> begin;
  int st = pack_table(segs, nsegs, nullptr, true, table, begin);
  if (st != PULSE_OK) return st;
  const uint64_t chunks = begin.back();
  if (chunks == 0) return PULSE_OK;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  PackTables* t = nullptr;
  st = pack_upload(device, stream, table, begin, &t);
  if (st != PULSE_OK) return st;
  return cuda_status(launch_unpack_multi(t->segs, t->begin, nsegs, chunks, stream));
}

// ------------------------------------------------------------ compose

int pulse_compose(const uint32_t* idx_a, const uint16_t* val_a, uint64_t count_a,
                  const uint32_t* idx_b, const uint16_t* val_b, uint64_t count_b,
                  uint32_t* idx_out, uint16_t* val_out, uint64_t* count_out, cudaStream_t stream) {
  return compose_one(idx_a, val_a, count_a, idx_b, val_b, count_b, idx_out, val_out, count_out, 2,
                     stream);
}

int pulse_compose_u8(const uint32_t* idx_a, const uint8_t* val_a, uint64_t count_a,
                     const uint32_t* idx_b, const uint8_t* val_b, uint64_t count_b,
                     uint32_t* idx_out, uint8_t* val_out, uint64_t* count_out, cudaStream_t stream) {
  return compose_one(idx_a, val_a, count_a, idx_b, val_b, count_b, idx_out, val_out, count_out, 1,
                     stream);
}

int pulse_compose_multi(const pulse_compose_segment* segs, int nsegs, int value_bytes,
                        uint64_t* counts_out, cudaStream_t stream) {
  if (segs == nullptr || nsegs < 1 || counts_out == nullptr) return PULSE_ERR_INVALID;
  if (value_bytes != 1 && value_bytes != 2) return PULSE_ERR_INVALID;
  std::vector<CmpSegment> table(static_cast<size_t>(nsegs));
  std::vector<uint64_t> tb(static_cast<size_t>(nsegs) + 1);
  uint64_t tiles = 0;
  for (int i = 0; i < nsegs; ++i) {
    const pulse_compose_segment& g = segs[i];
    if (g.count_a >= kMaxElems + 1 || g.count_b >= kMaxElems + 1) return PULSE_ERR_RANGE;
    if ((g.count_a > 0 && (g.idx_a == nullptr || g.val_a == nullptr)) ||
        (g.count_b > 0 && (g.idx_b == nullptr || g.val_b == nullptr)) ||
        (g.count_a + g.count_b > 0 && (g.idx_out == nullptr || g.val_out == nullptr)))
      return PULSE_ERR_INVALID;
    tb[size_t(i)] = tiles;
    table[size_t(i)] = CmpSegment{g.idx_a, g.val_a, g.count_a, g.idx_b, g.val_b, g.count_b,
                                  g.idx_out, g.val_out, tiles};
    tiles += compose_tiles(g.count_a + g.count_b);
  }
  tb[size_t(nsegs)] = tiles;
  if (tiles > kMaxTiles) return PULSE_ERR_RANGE;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  CmpWorkspace* w = stream_cmp_workspace(device, stream);
  if (w == nullptr) return PULSE_ERR_NOMEM;
  int st = cmp_reserve(*w, tiles, nsegs, stream);
  if (st != PULSE_OK) return st;
  // empty segments have no tile: their count is 0; the others are written
  // by their last tile
  if (cudaMemsetAsync(counts_out, 0, sizeof(uint64_t) * size_t(nsegs), stream) != cudaSuccess ||
      cudaMemcpyAsync(w->segs, table.data(), sizeof(CmpSegment) * size_t(nsegs),
                      cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(w->tile_begin, tb.data(), sizeof(uint64_t) * (size_t(nsegs) + 1),
                      cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  // (copies from pageable memory are staged before cudaMemcpyAsync returns,
  // so the host tables may go out of scope now)
  if (tiles == 0) return PULSE_OK;
  uint32_t epoch = 0;
  st = workspace_next_epoch(w->ws, stream, &epoch);
  if (st != PULSE_OK) return st;
  return cuda_status(launch_compose(w->segs, table[0], w->tile_begin, nsegs, tiles, w->splits,
                                    w->splits + w->split_cap, w->ws.status, w->ws.counters,
                                    counts_out, epoch, kDefaultWaitNs, value_bytes, stream));
}

// ------------------------------------------------------------ MXFP8 view

namespace {
bool mx_format_ok(int format) {
  return format == PULSE_MX_E4M3 || format == PULSE_MX_E2M1 || format == PULSE_MX_NVFP4;
}
// code bytes and block scales of an n-element view
uint64_t mx_code_bytes(int format, uint64_t n) { return format == PULSE_MX_E4M3 ? n : div_up(n, 2); }
uint64_t mx_scale_count(int format, uint64_t n) {
  return div_up(n, format == PULSE_MX_NVFP4 ? 16 : kMxBlock);
}
}  // namespace

int pulse_mx_quantize_fmt(int format, const float* master_f32, uint64_t n, uint8_t* codes_out,
                          uint8_t* scales_out, cudaStream_t stream) {
  if (!mx_format_ok(format) || format == PULSE_MX_NVFP4) return PULSE_ERR_INVALID;
  if (n >= kMaxElems + 1) return PULSE_ERR_RANGE;
  if (n == 0) return PULSE_OK;
  if (master_f32 == nullptr || codes_out == nullptr || scales_out == nullptr) return PULSE_ERR_INVALID;
  return cuda_status(
      launch_mx_quantize(format, master_f32, n, codes_out, scales_out, nullptr, nullptr, stream));
}

int pulse_nvfp4_quantize(const float* master_f32, uint64_t n, uint8_t* codes_out,
                         uint8_t* scales_out, float* tscale_out, cudaStream_t stream) {
  if (n >= kMaxElems + 1) return PULSE_ERR_RANGE;
  if (tscale_out == nullptr) return PULSE_ERR_INVALID;
  if (n == 0) return cuda_status(cudaMemsetAsync(tscale_out, 0, sizeof(float), stream));
  if (master_f32 == nullptr || codes_out == nullptr || scales_out == nullptr) return PULSE_ERR_INVALID;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  uint32_t* amax = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    Workspace* ws = stream_mx_workspace(device, stream);
    if (ws == nullptr) return PULSE_ERR_NOMEM;
    const int st = workspace_reserve(*ws, 0, stream);
    if (st != PULSE_OK) return st;
    amax = ws->counters + kAmaxWord;
  }
  pulse_mx_tensor t{};
  t.master = master_f32;
  t.n = n;
  MxLaunch a{};
  a.one = make_mx_desc(t, 0);
  a.ntensors = 1;
  a.total_tiles = div_up(n, kEncTile);
  if (cudaMemsetAsync(amax, 0, sizeof(uint32_t), stream) != cudaSuccess ||
      launch_mx_amax(a, false, amax, stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  return cuda_status(launch_mx_quantize(PULSE_MX_NVFP4, master_f32, n, codes_out, scales_out, amax,
                                        tscale_out, stream));
}

int pulse_mx_quantize(const float* master_f32, uint64_t n, uint8_t* codes_out, uint8_t* scales_out,
                      cudaStream_t stream) {
  return pulse_mx_quantize_fmt(PULSE_MX_E4M3, master_f32, n, codes_out, scales_out, stream);
}

namespace {
int mx_encode_one(int format, const float* master_f32, uint8_t* prev_codes, uint8_t* prev_scales,
                  uint64_t n, uint32_t* idx_out, uint8_t* val_out, uint32_t* sidx_out,
                  uint8_t* sval_out, uint64_t* counts_out, float* tscale_out, cudaStream_t stream) {
  if (n >= kMaxElems + 1) return PULSE_ERR_RANGE;
  if (counts_out == nullptr) return PULSE_ERR_INVALID;
  if (n > 0 && (master_f32 == nullptr || prev_codes == nullptr || prev_scales == nullptr ||
                idx_out == nullptr || val_out == nullptr || sidx_out == nullptr || sval_out == nullptr))
    return PULSE_ERR_INVALID;
  if (n == 0) {
    if (tscale_out != nullptr &&
        cudaMemsetAsync(tscale_out, 0, sizeof(float), stream) != cudaSuccess)
      return PULSE_ERR_CUDA;
    return cuda_status(cudaMemsetAsync(counts_out, 0, 2 * sizeof(uint64_t), stream));
  }
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  pulse_mx_tensor t{};
  t.master = master_f32;
  t.prev_codes = prev_codes;
  t.prev_scales = prev_scales;
  t.n = n;
  t.idx = idx_out;
  t.val = val_out;
  t.sidx = sidx_out;
  t.sval = sval_out;
  MxLaunch a{};
  a.one = make_mx_desc(t, 0);
  a.ntensors = 1;
  a.total_tiles = div_up(n, kEncTile);
  a.counts_out = counts_out;
  a.first_ticket = 0;
  a.wait_limit_ns = kDefaultWaitNs;
  a.tscale_out = tscale_out;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  Workspace* ws = stream_mx_workspace(device, stream);
  if (ws == nullptr) return PULSE_ERR_NOMEM;
  return launch_encode_mx_ws(a, format, *ws, false, device, stream);
}
}  // namespace

int pulse_mx_encode_fmt(int format, const float* master_f32, uint8_t* prev_codes,
                        uint8_t* prev_scales, uint64_t n, uint32_t* idx_out, uint8_t* val_out,
                        uint32_t* sidx_out, uint8_t* sval_out, uint64_t* counts_out,
                        cudaStream_t stream) {
  if (!mx_format_ok(format) || format == PULSE_MX_NVFP4) return PULSE_ERR_INVALID;
  return mx_encode_one(format, master_f32, prev_codes, prev_scales, n, idx_out, val_out, sidx_out,
                       sval_out, counts_out, nullptr, stream);
}

int pulse_nvfp4_encode(const float* master_f32, uint8_t* prev_codes, uint8_t* prev_scales,
                       uint64_t n, uint32_t* idx_out, uint8_t* val_out, uint32_t* sidx_out,
                       uint8_t* sval_out, uint64_t* counts_out, float* tscale_out,
                       cudaStream_t stream) {
  if (tscale_out == nullptr) return PULSE_ERR_INVALID;
  return mx_encode_one(PULSE_MX_NVFP4, master_f32, prev_codes, prev_scales, n, idx_out, val_out,
                       sidx_out, sval_out, counts_out, tscale_out, stream);
}

int pulse_mx_encode(const float* master_f32, uint8_t* prev_codes, uint8_t* prev_scales, uint64_t n,
                    uint32_t* idx_out, uint8_t* val_out, uint32_t* sidx_out, uint8_t* sval_out,
                    uint64_t* counts_out, cudaStream_t stream) {
  return pulse_mx_encode_fmt(PULSE_MX_E4M3, master_f32, prev_codes, prev_scales, n, idx_out, val_out,
                             sidx_out, sval_out, counts_out, stream);
}

int pulse_mx_apply_fmt(int format, uint8_t* codes, uint8_t* scales, uint64_t n,
                       const uint32_t* idx, const uint8_t* val, uint64_t count,
                       const uint32_t* sidx, const uint8_t* sval, uint64_t scount,
                       cudaStream_t stream) {
  if (!mx_format_ok(format)) return PULSE_ERR_INVALID;
  if (n >= kMaxElems + 1) return PULSE_ERR_RANGE;
  if (count == 0 && scount == 0) return PULSE_OK;
  if (count > 0 && (codes == nullptr || idx == nullptr || val == nullptr)) return PULSE_ERR_INVALID;
  if (scount > 0 && (scales == nullptr || sidx == nullptr || sval == nullptr)) return PULSE_ERR_INVALID;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  uint32_t* err = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    Workspace* ws = stream_mx_workspace(device, stream);
    if (ws == nullptr) return PULSE_ERR_NOMEM;
    const int st = workspace_reserve(*ws, 0, stream);
    if (st != PULSE_OK) return st;
    err = ws->counters + 2;
  }
  if (launch_apply_u8(codes, mx_code_bytes(format, n), true, idx, val, count, err, stream) !=
      cudaSuccess)
    return PULSE_ERR_CUDA;
  return cuda_status(
      launch_apply_u8(scales, mx_scale_count(format, n), true, sidx, sval, scount, err, stream));
}

int pulse_mx_apply(uint8_t* codes, uint8_t* scales, uint64_t n, const uint32_t* idx,
                   const uint8_t* val, uint64_t count, const uint32_t* sidx, const uint8_t* sval,
                   uint64_t scount, cudaStream_t stream) {
  return pulse_mx_apply_fmt(PULSE_MX_E4M3, codes, scales, n, idx, val, count, sidx, sval, scount,
                            stream);
}

int pulse_mx_plan_create_fmt(const pulse_mx_tensor* tensors, int ntensors, int format,
                             pulse_mx_plan** plan_out) {
  if (plan_out == nullptr) return PULSE_ERR_INVALID;
  *plan_out = nullptr;
  if (!mx_format_ok(format)) return PULSE_ERR_INVALID;
  if (tensors == nullptr || ntensors < 1 || ntensors > kMaxTensorsPerApplyLaunch / 2)
    return PULSE_ERR_INVALID;
  pulse_mx_plan* p = new (std::nothrow) pulse_mx_plan();
  if (p == nullptr) return PULSE_ERR_NOMEM;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return PULSE_ERR_CUDA;
  }
  p->ntensors = ntensors;
  p->format = format;
  p->can_encode = p->can_apply = true;
  std::vector<uint64_t> tb(size_t(ntensors) + 1, 0);
  std::vector<ByteSegment> segs(2 * size_t(ntensors));
  p->host_desc.reserve(size_t(ntensors));
  uint64_t tiles = 0;
  for (int i = 0; i < ntensors; ++i) {
    const pulse_mx_tensor& t = tensors[i];
    if (t.n >= kMaxElems + 1) {
      delete p;
      return PULSE_ERR_RANGE;
    }
    tb[size_t(i)] = tiles;
    p->host_desc.push_back(make_mx_desc(t, tiles));
    tiles += div_up(t.n, kEncTile);
    segs[2 * size_t(i)] = ByteSegment{t.codes, t.idx, t.val, mx_code_bytes(format, t.n)};
    segs[2 * size_t(i) + 1] = ByteSegment{t.scales, t.sidx, t.sval, mx_scale_count(format, t.n)};
    if (t.n > 0) {
      p->can_encode = p->can_encode && t.master && t.prev_codes && t.prev_scales && t.idx &&
                      t.val && t.sidx && t.sval;
      p->can_apply = p->can_apply && t.codes && t.scales && t.idx && t.val && t.sidx && t.sval;
    }
  }
  tb[size_t(ntensors)] = tiles;
  if (tiles > kMaxTiles) {
    delete p;
    return PULSE_ERR_RANGE;
  }
  p->total_tiles = tiles;
  const size_t desc_bytes = sizeof(MxTensorDesc) * size_t(ntensors);
  const size_t tb_bytes = sizeof(uint64_t) * (size_t(ntensors) + 1);
  const size_t seg_bytes = sizeof(ByteSegment) * segs.size();
  const size_t cnt_bytes = sizeof(uint64_t) * segs.size();
  int st = PULSE_OK;
  if (cudaMalloc(&p->desc, desc_bytes) != cudaSuccess ||
      cudaMalloc(&p->tile_begin, tb_bytes) != cudaSuccess ||
      cudaMalloc(&p->segs, seg_bytes) != cudaSuccess ||
      cudaMalloc(&p->counts, cnt_bytes) != cudaSuccess ||
      (format == PULSE_MX_NVFP4 &&
       cudaMalloc(&p->amax, sizeof(uint32_t) * size_t(ntensors)) != cudaSuccess)) {
    st = PULSE_ERR_NOMEM;
  } else if (cudaMemcpy(p->desc, p->host_desc.data(), desc_bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(p->tile_begin, tb.data(), tb_bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemcpy(p->segs, segs.data(), seg_bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
             cudaMemset(p->counts, 0, cnt_bytes) != cudaSuccess) {
    st = PULSE_ERR_CUDA;
  } else {
    st = workspace_reserve(p->ws, tiles, nullptr);
    if (st == PULSE_OK && cudaDeviceSynchronize() != cudaSuccess) st = PULSE_ERR_CUDA;
  }
  if (st != PULSE_OK) {
    pulse_mx_plan_destroy(p);
    return st;
  }
  *plan_out = p;
  return PULSE_OK;
}

int pulse_mx_plan_create(const pulse_mx_tensor* tensors, int ntensors, pulse_mx_plan** plan_out) {
  return pulse_mx_plan_create_fmt(tensors, ntensors, PULSE_MX_E4M3, plan_out);
}

int pulse_mx_plan_destroy(pulse_mx_plan* plan) {
  if (plan == nullptr) return PULSE_OK;
  const cudaError_t e = cudaDeviceSynchronize();
  if (plan->desc) cudaFree(plan->desc);
  if (plan->tile_begin) cudaFree(plan->tile_begin);
  if (plan->segs) cudaFree(plan->segs);
  if (plan->counts) cudaFree(plan->counts);
  if (plan->amax) cudaFree(plan->amax);
  workspace_free(plan->ws);
  delete plan;
  return cuda_status(e);
}

int pulse_mx_plan_num_tensors(const pulse_mx_plan* plan) { return plan ? plan->ntensors : 0; }

namespace {
int mx_encode_plan(pulse_mx_plan* plan, uint64_t* counts_out, float* tscales_out,
                   cudaStream_t stream) {
  if (tscales_out != nullptr &&
      cudaMemsetAsync(tscales_out, 0, sizeof(float) * size_t(plan->ntensors), stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  if (plan->total_tiles == 0)
    return cuda_status(
        cudaMemsetAsync(counts_out, 0, 2 * sizeof(uint64_t) * size_t(plan->ntensors), stream));
  MxLaunch a{};
  a.tensors = plan->desc;
  a.tile_begin = plan->tile_begin;
  a.ntensors = plan->ntensors;
  a.total_tiles = plan->total_tiles;
  a.counts_out = counts_out;
  a.first_ticket = 0;
  a.wait_limit_ns = kDefaultWaitNs;
  a.tscale_out = tscales_out;
  return launch_encode_mx_ws(a, plan->format, plan->ws, true, plan->device, stream, plan->amax);
}
}  // namespace

int pulse_mx_encode_multi(pulse_mx_plan* plan, uint64_t* counts_out, cudaStream_t stream) {
  if (plan == nullptr || counts_out == nullptr || !plan->can_encode ||
      plan->format == PULSE_MX_NVFP4)
    return PULSE_ERR_INVALID;
  return mx_encode_plan(plan, counts_out, nullptr, stream);
}

int pulse_nvfp4_encode_multi(pulse_mx_plan* plan, uint64_t* counts_out, float* tscales_out,
                             cudaStream_t stream) {
  if (plan == nullptr || counts_out == nullptr || tscales_out == nullptr || !plan->can_encode ||
      plan->format != PULSE_MX_NVFP4)
    return PULSE_ERR_INVALID;
  return mx_encode_plan(plan, counts_out, tscales_out, stream);
}

int pulse_mx_apply_multi_device(pulse_mx_plan* plan, const uint64_t* counts_dev, cudaStream_t stream) {
  if (plan == nullptr || counts_dev == nullptr || !plan->can_apply) return PULSE_ERR_INVALID;
  const int grid = sm_count(plan->device) * 8;
  return cuda_status(launch_apply_u8_multi(plan->segs, 2 * plan->ntensors, counts_dev,
                                           plan->ws.counters + 2, grid, stream));
}

int pulse_mx_apply_multi(pulse_mx_plan* plan, const uint64_t* counts_host, cudaStream_t stream) {
  if (plan == nullptr || counts_host == nullptr || !plan->can_apply) return PULSE_ERR_INVALID;
  if (cudaMemcpyAsync(plan->counts, counts_host, 2 * sizeof(uint64_t) * size_t(plan->ntensors),
                      cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return PULSE_ERR_CUDA;
  return pulse_mx_apply_multi_device(plan, plan->counts, stream);
}

int pulse_mx_plan_get_error(pulse_mx_plan* plan) {
  if (plan == nullptr) return PULSE_ERR_INVALID;
  if (cudaDeviceSynchronize() != cudaSuccess) return PULSE_ERR_CUDA;
  return workspace_take_error(plan->ws, nullptr);
}

}  // extern "C"
