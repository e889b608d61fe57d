// Router and dispatch for decode-sized batches (T <= 8).
//
// Logits: each expert row is split over `wpr` warps; every lane accumulates
// the exact products x[t, h] * Wr[e, h] of its columns into a float-float
// pair (Dot2), the pairs are merged across lanes and then across the row's
// warps in a fixed order, and one final rounding gives the FP32 logit: the
// correctly rounded value unless the exact dot product lies within ~2^-44
// (relative) of an FP32 rounding midpoint.  The last CTA to finish (arrival
// counter, no spinning) computes softmax + top-k per token with the token's
// logits held in registers, then the dispatch index: per-expert counts,
// offsets, the pair list as a stable counting sort, and the active experts.
//
// DGPP README "Execution and performance": engine.expert_tile_list (routed
// segments per expert); the top-k tie rule (logit descending, lower expert
// id first) keeps routing deterministic (DGPP README intro bullet "Exact").
#include "kernels.cuh"

namespace qmoe {

namespace {

constexpr int kMaxT = MOE_DECODE_MAX_TOKENS;
constexpr int kWarpsR = kRouterThreads / 32;

// Larger logit first; equal logits -> smaller expert id first.  A NaN logit
// ranks like -inf, so every untaken expert beats the empty state.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  if (v != v) v = -__int_as_float(0x7F800000);
  return (v > bv) || (v == bv && i < bi);
}

// One warp: top-k of one token.  E <= 1024: lane holds experts lane + 32 q.
__device__ void topk_warp(const float* __restrict__ logits_row, int E, int k, int32_t* idx_out, float* w_out,
                          int32_t* idx_out2, float* w_out2) {
  const int lane = threadIdx.x & 31;
  const float kNegInf = -__int_as_float(0x7F800000);
  float v[32];
#pragma unroll
  for (int q = 0; q < 32; ++q) {
    const int e = q * 32 + lane;
    v[q] = (e < E) ? __ldcg(logits_row + e) : kNegInf;
    if (v[q] != v[q]) v[q] = kNegInf;
  }
  uint32_t taken = 0;
  float sel_v0 = 0.f, sum = 0.f, my_ex = 0.f;
  int my_i = 0;
  for (int j = 0; j < k; ++j) {
    float bv = kNegInf;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int q = 0; q < 32; ++q) {
      const int e = q * 32 + lane;
      if (e < E && !((taken >> q) & 1u) && better(v[q], e, bv, bi)) { bv = v[q]; bi = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (bi < E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (j == 0) sel_v0 = bv;
    // w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0); the sum runs in j order
    const float ex = expf(bv - sel_v0);
    sum += ex;
    if (lane == j) { my_ex = ex; my_i = bi; }
  }
  if (lane < k) {
    const float w = my_ex / sum;
    idx_out[lane] = my_i;
    w_out[lane] = w;
    if (idx_out2) idx_out2[lane] = my_i;
    if (w_out2) w_out2[lane] = w;
  }
}

// Logits of this CTA's expert rows; returns after writing them to global memory.
__device__ void router_logits_cta(const RouterArgs& a, const uint16_t* xs, float (*s_hi)[kMaxT],
                                  float (*s_lo)[kMaxT]) {
  const int H = a.H, E = a.E, T = a.T, wpr = a.wpr;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows_per_cta = kWarpsR / wpr;
  const int e = blockIdx.x * rows_per_cta + warp / wpr;
  const int part = warp % wpr;
  const int Hw = H / wpr;
  float hi[kMaxT], lo[kMaxT];
#pragma unroll
  for (int t = 0; t < kMaxT; ++t) { hi[t] = 0.f; lo[t] = 0.f; }
  if (e < E) {
    const float4* wrow = reinterpret_cast<const float4*>(a.w + (size_t)e * H + (size_t)part * Hw);
    const uint16_t* xp = xs + (size_t)part * Hw;
#pragma unroll 2
    for (int h4 = lane; h4 < Hw / 4; h4 += 32) {
      const float4 wv = __ldg(wrow + h4);
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) {
        if (t < T) {
          const uint2 xv = *reinterpret_cast<const uint2*>(xp + (size_t)t * H + h4 * 4);
          dot2_step(bf16_bits_to_float(xv.x & 0xFFFF), wv.x, hi[t], lo[t]);
          dot2_step(bf16_bits_to_float(xv.x >> 16), wv.y, hi[t], lo[t]);
          dot2_step(bf16_bits_to_float(xv.y & 0xFFFF), wv.z, hi[t], lo[t]);
          dot2_step(bf16_bits_to_float(xv.y >> 16), wv.w, hi[t], lo[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
      if (t < T) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float h2 = __shfl_xor_sync(0xFFFFFFFFu, hi[t], o);
          const float l2 = __shfl_xor_sync(0xFFFFFFFFu, lo[t], o);
          dot2_merge(hi[t], lo[t], h2, l2);
        }
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) { s_hi[warp][t] = hi[t]; s_lo[warp][t] = lo[t]; }
    }
  }
  __syncthreads();
  // the first warp of each row merges the row's parts in order and rounds once
  if (e < E && part == 0 && lane < T) {
    float h = s_hi[warp][lane], l = s_lo[warp][lane];
    for (int p = 1; p < wpr; ++p) dot2_merge(h, l, s_hi[warp + p][lane], s_lo[warp + p][lane]);
    float lg = __fadd_rn(h, l);
    if (a.bias) lg = __fadd_rn(lg, __ldg(a.bias + e));
    a.rb.logits[(size_t)lane * E + e] = lg;
  }
}

__global__ void __launch_bounds__(kRouterThreads) router_decode_kernel(RouterArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);  // bf16 [T][H]
  __shared__ float s_hi[kWarpsR][kMaxT], s_lo[kWarpsR][kMaxT];
  __shared__ int is_last;
  const int H = a.H, E = a.E, T = a.T, k = a.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the expert kernel that follows may be scheduled now: it stages the
  // activations and then waits for this grid's results (griddepcontrol.wait)
  asm volatile("griddepcontrol.launch_dependents;");
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    const int n16 = T * H / 8;
    for (int i = tid; i < n16; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  router_logits_cta(a, xs, s_hi, s_lo);

  // ---- last CTA: top-k and dispatch ----
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t prev = atomicAdd(&a.rb.ctrl->router_arrive, 1u);
    is_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  for (int t = warp; t < T; t += kWarpsR)
    topk_warp(a.rb.logits + (size_t)t * E, E, k, a.rb.topk_idx + t * k, a.rb.topk_w + t * k,
              a.out.topk_idx ? a.out.topk_idx + t * k : nullptr, a.out.topk_w ? a.out.topk_w + t * k : nullptr);
  // the expert kernels accumulate per-pair maxima with atomicMax: start them at zero
  if (a.h_amax)
    for (int i = tid; i < T * k; i += blockDim.x) a.h_amax[i] = 0u;
  if (a.hs_amax)
    for (int i = tid; i < T; i += blockDim.x) a.hs_amax[i] = 0u;
  __syncthreads();

  // dispatch (counting sort, stable in the pair id p = t*k + j)
  int32_t* s_cnt = reinterpret_cast<int32_t*>(smem);  // [E]
  int32_t* s_off = s_cnt + E;                         // [E + 1]
  int32_t* s_idx = s_off + E + 1;                     // [T*k]
  const int P = T * k;
  for (int i = tid; i < E; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += blockDim.x) {
    const int ex = __ldcg(a.rb.topk_idx + p);
    s_idx[p] = ex;
    atomicAdd(&s_cnt[ex], 1);
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive scan over E counts, and the compacted list of active experts
    int run = 0, run_act = 0;
    for (int base = 0; base < E; base += 32) {
      const int e2 = base + lane;
      const int c = (e2 < E) ? s_cnt[e2] : 0;
      int incl = c, act_incl = (c > 0);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        const int va = __shfl_up_sync(0xFFFFFFFFu, act_incl, o);
        if (lane >= o) { incl += v; act_incl += va; }
      }
      if (e2 < E) {
        s_off[e2] = run + incl - c;
        a.rb.cnt[e2] = c;
        if (a.out.cnt) a.out.cnt[e2] = c;
        if (c > 0) a.rb.act[run_act + act_incl - 1] = e2;
      }
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
      run_act += __shfl_sync(0xFFFFFFFFu, act_incl, 31);
    }
    if (lane == 0) {
      s_off[E] = run;
      a.rb.ctrl->n_active = run_act;
    }
  }
  __syncthreads();
  for (int i = tid; i <= E; i += blockDim.x) {
    a.rb.off[i] = s_off[i];
    if (a.out.off) a.out.off[i] = s_off[i];
  }
  for (int p = tid; p < P; p += blockDim.x) {
    const int ex = s_idx[p];
    int rank = 0;
    for (int q = 0; q < p; ++q) rank += (s_idx[q] == ex);
    const int pos = s_off[ex] + rank;
    a.rb.pair[pos] = p;
    if (a.out.pair) a.out.pair[pos] = p;
  }
  if (tid == 0) a.rb.ctrl->router_arrive = 0;  // leave the counter at zero for the next call
}

}  // namespace

// Warps sharing one expert row: split H while each warp keeps >= 256 columns.
int router_warps_per_row(int H) {
  int w = 1;
  while (w < kWarpsR && H % (4 * 32 * w * 2) == 0 && H / (w * 2) >= 256) w *= 2;
  return w;
}

cudaError_t launch_router_decode(const RouterArgs& a, cudaStream_t s) {
  const int rows_per_cta = kWarpsR / a.wpr;
  const int grid = (a.E + rows_per_cta - 1) / rows_per_cta;
  const size_t smem_x = (size_t)a.T * a.H * 2;
  const size_t smem_d = (size_t)(2 * a.E + 1 + a.T * a.k) * 4;
  const size_t smem = smem_x > smem_d ? smem_x : smem_d;
  cudaError_t err = cudaFuncSetAttribute(router_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  router_decode_kernel<<<grid, kRouterThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace qmoe
