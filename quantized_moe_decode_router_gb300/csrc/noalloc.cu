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
void* g_scratch_ptr[kMaxDevices];

// Device address of g_scratch on the current device, looked up once per
// device (with that device current) and cached; the first lookup also zeroes
// the array (synchronously).  In host code g_scratch names only a host-side
// stand-in, so kernels must be given this address, never the symbol.
int32_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    if (cudaMemset(p, 0, kScratchBytes) != cudaSuccess) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" int32_t moe_decode_forward_noalloc(const moe_layer* layer, const void* x, int32_t T, void* y,
                                              const moe_options* opts, moe_stream_t stream) {
  const size_t need = moe_workspace_size(layer, T < 1 ? 1 : T, opts);
  if (need == 0) return MOE_ERR_INVALID_ARG;
  if (need > kScratchBytes) return MOE_ERR_WORKSPACE;  // this layer and T need more than the fixed array
  void* ws = nullptr;
  int32_t st = scratch_for_current_device(&ws);
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: clear what must start at zero
  if ((st = qmoe::clear_workspace_counters(layer, ws, need, s)) != MOE_OK) return st;
  return moe_decode_forward(layer, x, T, y, opts, ws, need, stream);
}
