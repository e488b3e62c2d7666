// moe_route_noalloc: the router entry point for callers that cannot allocate
// device memory -- for example a plugin that is handed only its input and
// output buffers by a host framework that owns every byte of device memory
// through its own pool, or a latency-critical caller that must not enter the
// CUDA allocator (cudaMalloc / cudaFree can synchronise the device). Its
// scratch memory (an error word and the router's fixed-point statistic
// accumulators) lives in a file-scope device array of fixed size, so the call
// allocates nothing.
//
// The array is shared by every call in the process on a given device and keeps
// the last call's contents; calls that overlap on the GPU (different streams,
// or different host threads) race on it and must be serialised by the caller.
// The first call on each device looks up the array's device address with
// cudaGetSymbolAddress (with that device current); make that first call before
// any stream capture. Everything else it does is the same launch sequence as
// moe_route, reusing the same kernels.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "stats.cuh"

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = 4096;  // per device, held until process exit: E <= 318
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_route_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch array (looked up once per device).
moe_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" MOE_API moe_status moe_route_noalloc(const moe_config* cfg, const void* x, const moe_weights* w,
                                                int32_t* idx, float* gate, float* logits, float* probs, void* stats,
                                                void* stream) {
  Plan p;
  moe_status s = make_plan(cfg, &p);
  if (s != MOE_OK) return s;
  if (!w || !x || !idx || !gate || !stats) return MOE_ERR_INVALID_ARG;
  p.rsplit = 1;  // no workspace for partial logits
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(idx) | reinterpret_cast<uintptr_t>(gate) |
       reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(probs) |
       reinterpret_cast<uintptr_t>(stats) | reinterpret_cast<uintptr_t>(w->w_router) |
       reinterpret_cast<uintptr_t>(w->logit_bias)) & 15u)
    return MOE_ERR_INVALID_ARG;
  if (!w->w_router) return MOE_ERR_INVALID_ARG;
  // Buffers the workspace would otherwise hold must come from the caller.
  if (router_uses_tc(p) && !logits) return MOE_ERR_INVALID_ARG;  // tensor-core router writes logits first
  if (p.ec && !probs) return MOE_ERR_INVALID_ARG;                 // expert choice selects on the probabilities
  if (p.N == 0) return MOE_OK;
  // Scratch layout inside the static array: error word, then the statistic accumulators.
  size_t o = 0;
  const size_t status_off = o;
  o += align256(32);
  p.stat_acc = o;
  o += align256(stats_acc_bytes(p.E));
  if (o > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;  // layer too large for the fixed scratch
  p.L.status = status_off;
  void* scratch = nullptr;
  if ((s = scratch_address(&scratch)) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  // The error word and the statistic accumulators must start at zero.
  if (cudaMemsetAsync(static_cast<uint8_t*>(scratch) + status_off, 0, p.stat_acc + stats_acc_bytes(p.E) - status_off,
                      st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_router(p, x, w, idx, gate, logits, probs, stats, scratch, st, nullptr, true) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (p.ec && launch_ec_select(p, probs, idx, gate, nullptr, st) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

// The error word sits at the start of the scratch array (offset 0 in the layout above).
extern "C" MOE_API moe_status moe_get_noalloc_status(void* stream, int32_t* device_error) {
  void* scratch = nullptr;
  moe_status s = scratch_address(&scratch);
  if (s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t word[4] = {0, 0, 0, 0};
  cudaGetLastError();
  if (cudaMemcpyAsync(word, scratch, sizeof word, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(scratch, 0, sizeof word, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (device_error) *device_error = word[0];
  if (word[0] & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (word[0] & kErrIndex) return MOE_ERR_DEVICE_CHECK;
  return MOE_OK;
}
