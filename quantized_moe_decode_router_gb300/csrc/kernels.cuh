// Kernel argument blocks and launch entry points shared by the host ABI and
// the kernel translation units.
#pragma once

#include "common.cuh"

namespace qmoe {

struct QW {
  const uint8_t* data;
  const uint8_t* scales;
  const float* ts;  // NVFP4 tensor scales [count], else nullptr
};

// Routing results and scratch buffers inside the caller's workspace.
struct RouteBufs {
  Ctrl* ctrl;
  float* logits;      // [T, E]
  int32_t* topk_idx;  // [T, k]
  float* topk_w;      // [T, k]
  int32_t* cnt;       // [E]
  int32_t* off;       // [E + 1]
  int32_t* pair;      // [T * k]
  int32_t* act;       // [E] active experts, ascending
};

// Optional copies of the routing results into caller buffers (moe_route).
struct RouteOut {
  int32_t* topk_idx;
  float* topk_w;
  int32_t* cnt;
  int32_t* off;
  int32_t* pair;
};

struct RouterArgs {
  int H, E, k, T;
  const uint16_t* x;  // bf16 [T, H]
  const float* w;     // [E, H]
  const float* bias;  // [E] or nullptr
  RouteBufs rb;
  RouteOut out;
};

// Decode-path expert kernels.
struct ExpertArgs {
  int H, I, E, k, T;
  int fmt, sfmt, Is;  // routed format; shared format (0 = none) and size
  const uint16_t* x;  // bf16 [T, H]
  QW gate, up, down, sgate, sup, sdown;
  RouteBufs rb;
  uint16_t* h;        // bf16 [T*k, I]
  uint16_t* hs;       // bf16 [T, Is]
  float* P;           // f32 [T*k, H] per-pair down partials
  float* S;           // f32 [T, H] shared expert output
  uint32_t* rb_cnt;   // [H / (16 * wr_dn)] arrival counters of the combine
  uint16_t* y;        // bf16 [T, H]
  // warp split of a CTA's 8 warps: wk ways along K, wr ways along rows
  int wk_gu, wr_gu, wk_dn, wr_dn;
  // shared-memory layout of the staged activations (in halfs)
  int xs_q_stride, xs_tok_stride;  // gate/up: x
  int hs_q_stride, hs_tok_stride;  // down: h
};

constexpr int kExpertThreads = 256;  // 8 warps
constexpr int kRouterThreads = 256;

cudaError_t launch_router_decode(const RouterArgs& a, cudaStream_t s);
cudaError_t launch_gateup_decode(const ExpertArgs& a, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_down_decode(const ExpertArgs& a, int grid, size_t smem, cudaStream_t s);

// moe_dequantize / moe_quantize_act_nvfp4
cudaError_t launch_dequantize(int fmt, QW w, int N, int K, int expert, int row0, int nrows, float* out,
                              cudaStream_t s);
cudaError_t launch_quantize_act_nvfp4(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales,
                                      cudaStream_t s);

// Bytes of one matrix's codes / scales in a format.
__host__ __device__ inline size_t data_bytes(int fmt, int N, int K) {
  switch (fmt) {
    case MOE_FMT_NVFP4: case MOE_FMT_MXFP4: case MOE_FMT_INT4_G64: return (size_t)N * K / 2;
    case MOE_FMT_INT8_G64: case MOE_FMT_FP8_B128: return (size_t)N * K;
    default: return 0;
  }
}

__host__ __device__ inline size_t scale_bytes(int fmt, int N, int K) {
  switch (fmt) {
    case MOE_FMT_NVFP4: return (size_t)N * (K / 16);
    case MOE_FMT_MXFP4: return (size_t)N * (K / 32);
    case MOE_FMT_INT4_G64: case MOE_FMT_INT8_G64: return (size_t)N * (K / 64) * 2;
    case MOE_FMT_FP8_B128: return (size_t)(N / 128) * (K / 128) * 4;
    default: return 0;
  }
}

// Columns of one decode work unit (four lanes' chunks) in a format; a warp's
// share of K must be a multiple of it.
__host__ __device__ inline int decode_unit_k(int fmt) {
  switch (fmt) {
    case MOE_FMT_NVFP4: return 128;
    case MOE_FMT_MXFP4: return 32;
    case MOE_FMT_INT4_G64: return 64;
    case MOE_FMT_INT8_G64: return 64;
    case MOE_FMT_FP8_B128: return 64;
    default: return 0;
  }
}

}  // namespace qmoe
