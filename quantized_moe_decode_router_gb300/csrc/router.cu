// Router and dispatch for decode-sized batches (T <= 8).
//
// Logits: one warp per expert row, each lane accumulating the exact products
// x[t, h] * Wr[e, h] into a float-float pair (Dot2), so the final rounding
// gives the correctly rounded FP32 logit except when the exact value lies
// within ~2^-44 (relative) of an FP32 rounding midpoint.  The last CTA to
// finish (arrival counter, no spinning) computes softmax + top-k per token and
// the dispatch index: per-expert counts, offsets, the pair list as a stable
// counting sort, and the list of active experts.
//
// DGPP README "Execution and performance": engine.expert_tile_list (routed
// segments per expert); the top-k tie rule (logit descending, lower expert id
// first) keeps routing deterministic (DGPP README intro bullet "Exact").
#include "kernels.cuh"

namespace qmoe {

namespace {

constexpr int kMaxT = MOE_DECODE_MAX_TOKENS;

// Key order: larger logit first; equal logits -> smaller expert id first.
// A NaN logit ranks like -inf, so every untaken expert beats the empty state
// (-inf, INT_MAX) and k <= E selections always find a valid id.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  if (v != v) v = -__int_as_float(0x7F800000);
  return (v > bv) || (v == bv && i < bi);
}

__device__ void topk_warp(const float* __restrict__ logits_row, int E, int k, const float* __restrict__ bias,
                          int32_t* idx_out, float* w_out, int32_t* idx_out2, float* w_out2) {
  const int lane = threadIdx.x & 31;
  // each lane owns experts lane, lane + 32, ... (E <= 1024 -> at most 32); bit q marks a taken entry
  uint32_t taken = 0;
  const int per_lane = (E + 31) / 32;
  float sel_v[16];
  int sel_i[16];
  for (int j = 0; j < k; ++j) {
    float bv = -__int_as_float(0x7F800000);
    int bi = 0x7FFFFFFF;
    for (int q = 0; q < per_lane; ++q) {
      int e = q * 32 + lane;
      if (e < E && !((taken >> q) & 1u)) {
        float v = __ldcg(logits_row + e);
        if (better(v, e, bv, bi)) { bv = (v != v) ? -__int_as_float(0x7F800000) : v; bi = e; }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
      int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (better(ov, oi, bv, bi)) { bv = (ov != ov) ? bv : ov; bi = oi; }
    }
    if (bi < E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    sel_v[j] = bv;
    sel_i[j] = bi;
  }
  (void)bias;
  if (lane == 0) {
    // w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0), summed in j order
    float ex[16];
    float sum = 0.f;
    for (int j = 0; j < k; ++j) {
      ex[j] = expf(sel_v[j] - sel_v[0]);
      sum += ex[j];
    }
    for (int j = 0; j < k; ++j) {
      float w = ex[j] / sum;
      idx_out[j] = sel_i[j];
      w_out[j] = w;
      if (idx_out2) idx_out2[j] = sel_i[j];
      if (w_out2) w_out2[j] = w;
    }
  }
}

__global__ void __launch_bounds__(kRouterThreads) router_decode_kernel(RouterArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);  // bf16 [T][H]
  const int H = a.H, E = a.E, T = a.T, k = a.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the expert kernel that follows may be scheduled now: it stages the
  // activations and then waits for this grid's results (griddepcontrol.wait)
  asm volatile("griddepcontrol.launch_dependents;");

  // stage x (bf16) in shared memory
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.x);
    uint4* dst = reinterpret_cast<uint4*>(xs);
    const int n16 = T * H / 8;
    for (int i = tid; i < n16; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();

  const int e = blockIdx.x * (kRouterThreads / 32) + warp;
  if (e < E) {
    float hi[kMaxT], lo[kMaxT];
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) { hi[t] = 0.f; lo[t] = 0.f; }
    const float4* wrow = reinterpret_cast<const float4*>(a.w + (size_t)e * H);
    for (int h4 = lane; h4 < H / 4; h4 += 32) {
      float4 wv = __ldg(wrow + h4);
#pragma unroll
      for (int t = 0; t < kMaxT; ++t) {
        if (t < T) {
          uint2 xv = *reinterpret_cast<const uint2*>(xs + (size_t)t * H + h4 * 4);
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
          float h2 = __shfl_xor_sync(0xFFFFFFFFu, hi[t], o);
          float l2 = __shfl_xor_sync(0xFFFFFFFFu, lo[t], o);
          dot2_merge(hi[t], lo[t], h2, l2);
        }
        if (lane == 0) {
          float l = __fadd_rn(hi[t], lo[t]);
          if (a.bias) l = __fadd_rn(l, __ldg(a.bias + e));
          a.rb.logits[(size_t)t * E + e] = l;
        }
      }
    }
  }

  // ---- last CTA: top-k and dispatch ----
  __shared__ int is_last;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    uint32_t prev = atomicAdd(&a.rb.ctrl->router_arrive, 1u);
    is_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  for (int t = warp; t < T; t += kRouterThreads / 32) {
    topk_warp(a.rb.logits + (size_t)t * E, E, k, a.bias, a.rb.topk_idx + t * k, a.rb.topk_w + t * k,
              a.out.topk_idx ? a.out.topk_idx + t * k : nullptr, a.out.topk_w ? a.out.topk_w + t * k : nullptr);
  }
  __syncthreads();

  // dispatch (counting sort, stable in the pair id p = t*k + j)
  int32_t* s_cnt = reinterpret_cast<int32_t*>(smem);           // [E]
  int32_t* s_off = s_cnt + E;                                  // [E + 1]
  int32_t* s_idx = s_off + E + 1;                              // [T*k]
  const int P = T * k;
  for (int i = tid; i < E; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += blockDim.x) {
    int ex = __ldcg(a.rb.topk_idx + p);
    s_idx[p] = ex;
    atomicAdd(&s_cnt[ex], 1);
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive scan over E counts, and the compacted list of active experts
    int run = 0, run_act = 0;
    for (int base = 0; base < E; base += 32) {
      int e2 = base + lane;
      int c = (e2 < E) ? s_cnt[e2] : 0;
      int incl = c, act_incl = (c > 0);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        int va = __shfl_up_sync(0xFFFFFFFFu, act_incl, o);
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

cudaError_t launch_router_decode(const RouterArgs& a, cudaStream_t s) {
  const int grid = (a.E + kRouterThreads / 32 - 1) / (kRouterThreads / 32);
  size_t smem_x = (size_t)a.T * a.H * 2;
  size_t smem_d = (size_t)(2 * a.E + 1 + a.T * a.k) * 4;
  size_t smem = smem_x > smem_d ? smem_x : smem_d;
  cudaError_t err = cudaFuncSetAttribute(router_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  router_decode_kernel<<<grid, kRouterThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace qmoe
