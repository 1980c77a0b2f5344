// encode_noalloc.cu -- pulse_encode for callers that cannot allocate device
// memory.
//
// pulse_encode keeps its look-back scratch (one status word per 4096-element
// tile, plus a ticket counter, a finish counter and an error word) in a
// workspace it allocates with cudaMalloc the first time a (device, stream)
// pair is seen, and grows later if a larger tensor arrives. Some callers may
// not allocate at that point: engines that hand all device memory to their
// own pool at start-up, runtimes that forbid allocation once serving has
// begun, or code that must not synchronise the device (cudaMalloc and
// cudaFree can). For them, pulse_encode_noalloc keeps the same scratch in
// one fixed file-scope device array instead, sized for tensors of up to
// PULSE_NOALLOC_MAX_ELEMS elements. Every GPU that loads this library holds
// that array (512 KB of status words + 256 bytes) until the process exits.
//
// The array is shared by every call on a device and keeps the previous
// call's contents, so each call clears, on its stream and before its kernel,
// the status words of its own tiles and the counters (8 bytes per 4096
// elements plus 256 bytes; cudaMemsetAsync allocates nothing). Each call's
// device work then depends only on its arguments, never on how many calls
// came before it. Two calls whose kernels overlap on the GPU (different
// streams, no ordering between them) race on the array and give wrong
// results; callers must order them.
#include <mutex>

#include "pulse.h"
#include "pulse_device.cuh"
#include "pulse_internal.h"

namespace pulse {
namespace {

constexpr uint64_t kNoallocMaxTiles = PULSE_NOALLOC_MAX_ELEMS / kEncTile;
static_assert(PULSE_NOALLOC_MAX_ELEMS % kEncTile == 0, "whole tiles");
constexpr int kNoallocCounterWords = 64;  // ticket, finished, error word, padding (256 bytes)
constexpr int kNoallocMaxDevices = 64;
constexpr uint64_t kNoallocWaitNs = 1000000000ull;

struct NoallocScratch {
  uint64_t status[kNoallocMaxTiles];
  uint32_t counters[kNoallocCounterWords];
};

// Zero when the module is loaded. In host code this name is only a stand-in
// for the device symbol: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) NoallocScratch g_noalloc_scratch;

// Every call clears the status words it reads, so one fixed epoch serves.
constexpr uint32_t kNoallocEpoch = 1u;

struct DeviceState {
  NoallocScratch* scratch;  // device address of g_noalloc_scratch on this device
};

std::mutex g_noalloc_mu;
DeviceState g_noalloc_state[kNoallocMaxDevices];  // static storage: no host allocation either

// After the encode kernel: turn a recorded device error into a count of
// UINT64_MAX and clear the error word for the next call.
__global__ void noalloc_report_kernel(uint32_t* error_word, uint64_t* count_out) {
  if (*error_word != 0u) *count_out = ~0ull;
  *error_word = 0u;
}

}  // namespace
}  // namespace pulse

using namespace pulse;

extern "C" int pulse_encode_noalloc(const float* master_f32, uint16_t* prev_bf16, uint64_t n,
                                    uint32_t* idx_out, uint16_t* val_out, uint64_t* count_out,
                                    cudaStream_t stream) {
  if (count_out == nullptr) return PULSE_ERR_INVALID;
  if (n > PULSE_NOALLOC_MAX_ELEMS) return PULSE_ERR_RANGE;
  if (n > 0 && (master_f32 == nullptr || prev_bf16 == nullptr || idx_out == nullptr ||
                val_out == nullptr))
    return PULSE_ERR_INVALID;
  if (n == 0)
    return cudaMemsetAsync(count_out, 0, sizeof(uint64_t), stream) == cudaSuccess ? PULSE_OK
                                                                                 : PULSE_ERR_CUDA;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PULSE_ERR_CUDA;
  if (device < 0 || device >= kNoallocMaxDevices) return PULSE_ERR_INVALID;

  EncodeLaunch a{};
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    DeviceState& st = g_noalloc_state[device];
    if (st.scratch == nullptr) {
      // set-up, once per device, with that device current
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
        return PULSE_ERR_CUDA;
      st.scratch = static_cast<NoallocScratch*>(ptr);
    }
    a.status = st.scratch->status;
    a.counters = st.scratch->counters;
  }
  a.epoch = kNoallocEpoch;
  a.total_tiles = (n + kEncTile - 1) / kEncTile;
  // this call's status words read "not yet published"; ticket, finish
  // counter and error word start at zero
  if (cudaMemsetAsync(a.status, 0, sizeof(uint64_t) * size_t(a.total_tiles), stream) != cudaSuccess ||
      cudaMemsetAsync(a.counters, 0, sizeof(uint32_t) * kNoallocCounterWords, stream) != cudaSuccess)
    return PULSE_ERR_CUDA;

  a.one.master = master_f32;
  a.one.prev = prev_bf16;
  a.one.idx = idx_out;
  a.one.val = val_out;
  a.one.n = n;
  a.one.tile_begin = 0;
  a.one.bulk_ok = (reinterpret_cast<uintptr_t>(master_f32) % 16u == 0 &&
                   reinterpret_cast<uintptr_t>(prev_bf16) % 16u == 0)
                      ? 1u
                      : 0u;
  a.one.vec_ok = 0u;
  a.tensors = nullptr;
  a.tile_begin = nullptr;
  a.ntensors = 1;
  a.counts_out = count_out;
  a.first_ticket = 0;
  a.wait_limit_ns = kNoallocWaitNs;
  const uint64_t cap = uint64_t(encode_grid_size(device));
  const int grid = int(a.total_tiles < cap ? a.total_tiles : cap);
  if (launch_encode(a, false, grid, stream) != cudaSuccess) return PULSE_ERR_CUDA;
  noalloc_report_kernel<<<1, 1, 0, stream>>>(a.counters + 2, count_out);
  return cudaGetLastError() == cudaSuccess ? PULSE_OK : PULSE_ERR_CUDA;
}
