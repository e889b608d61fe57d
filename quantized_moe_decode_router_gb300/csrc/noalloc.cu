// moe_decode_forward_noalloc: the decode forward for callers that cannot
// allocate device memory.  Its workspace is a file-scope device array of a
// fixed size that every GPU loading the library holds until the process
// exits; nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "kernels.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)32 << 20;  // 32 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

std::mutex g_mu;
// Device address of g_scratch at which the first call on each device cleared
// the control block (error word included); 0 before that call.
uintptr_t g_ready[kMaxDevices];

// Device address of g_scratch on the current device.  In host code
// g_scratch names only a host-side stand-in, so kernels must be given this
// address, never the symbol.  The lookup runs on every call (it is cheap), so
// a module reloaded at another address after a device reset is noticed.
int32_t scratch_address(int* dev, void** out) {
  if (cudaGetDevice(dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (*dev < 0 || *dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
  *out = p;
  return MOE_OK;
}

}  // namespace

int32_t qmoe::noalloc_array_if_used(void** out) {
  *out = nullptr;
  int dev = 0;
  void* p = nullptr;
  const int32_t st = scratch_address(&dev, &p);
  if (st != MOE_OK) return st;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_ready[dev] == reinterpret_cast<uintptr_t>(p)) *out = p;
  return MOE_OK;
}

extern "C" int32_t moe_decode_forward_noalloc(const moe_layer* layer, const void* x, int32_t T, void* y,
                                              const moe_options* opts, moe_stream_t stream) {
  // every host check first: a rejected call touches neither the array nor the device
  int32_t st = qmoe::check_decode_args(layer, x, T, y, opts);
  if (st != MOE_OK) return st;
  const size_t need = moe_workspace_size(layer, T, opts);
  if (need == 0) return MOE_ERR_INVALID_ARG;
  if (need > kScratchBytes) return MOE_ERR_WORKSPACE;  // this layer and T need more than the fixed array
  int dev = 0;
  void* ws = nullptr;
  if ((st = scratch_address(&dev, &ws)) != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bool first;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    first = g_ready[dev] != reinterpret_cast<uintptr_t>(ws);
    g_ready[dev] = reinterpret_cast<uintptr_t>(ws);
  }
  // The array keeps the previous call's contents: clear, on the caller's
  // stream, every counter that must start at zero.  The device-side error
  // word is cleared only by the first call on a device; after that it keeps
  // the first error any call reported until moe_check(NULL, 0, stream) reads it.
  if ((st = qmoe::clear_workspace_counters(layer, ws, need, !first, s)) != MOE_OK) return st;
  return moe_decode_forward(layer, x, T, y, opts, ws, need, stream);
}
