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

// Selection key of a candidate: larger logit first, equal logits -> smaller
// expert id first, as one unsigned 64-bit maximum.  The float is mapped to
// an order-preserving unsigned integer (NaN ranks like -inf); the low half is
// the complemented expert id.  0 marks a taken or absent entry: every real
// candidate, even a -inf logit, has a larger key.
__device__ __forceinline__ unsigned long long sel_key(float v, int e) {
  uint32_t b = __float_as_uint(v);
  if (v != v) b = 0xFF800000u;  // -inf
  if (b == 0x80000000u) b = 0;  // -0 ties with +0
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)ord << 32) | (uint32_t)(~(uint32_t)e);
}

__device__ __forceinline__ float key_value(unsigned long long k) {
  const uint32_t ord = (uint32_t)(k >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}

__device__ __forceinline__ int key_id(unsigned long long k) { return (int)(~(uint32_t)k); }

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

// Largest of the lane's NQ keys, as a tournament (depth log2 NQ).
template <int NQ>
__device__ __forceinline__ unsigned long long lane_max(const unsigned long long (&key)[NQ]) {
  unsigned long long t[NQ / 2];
#pragma unroll
  for (int q = 0; q < NQ / 2; ++q) t[q] = umax64(key[2 * q], key[2 * q + 1]);
#pragma unroll
  for (int w = NQ / 4; w > 0; w >>= 1)
#pragma unroll
    for (int q = 0; q < w; ++q) t[q] = umax64(t[2 * q], t[2 * q + 1]);
  return t[0];
}

// Order-preserving unsigned image of a logit (larger logit -> larger key);
// NaN ranks like -inf, -0 like +0.  Every real logit maps above 0, the key of
// a taken or absent entry.
__device__ __forceinline__ uint32_t ord_key(float v) {
  uint32_t b = __float_as_uint(v);
  if (v != v) b = 0xFF800000u;  // -inf
  if (b == 0x80000000u) b = 0;  // -0 ties with +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float ord_value(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// Largest key of the lane and its slot; equal keys -> the lower slot (lower
// expert id).  A tournament: depth log2(NQ) instead of a chain of NQ - 1.
template <int NQ>
__device__ __forceinline__ void lane_best(const uint32_t (&key)[NQ], uint32_t& bk, int& bq) {
  uint32_t k2[NQ];
  int q2[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) { k2[q] = key[q]; q2[q] = q; }
#pragma unroll
  for (int w = NQ / 2; w > 0; w >>= 1)
#pragma unroll
    for (int q = 0; q < w; ++q) {
      const bool right = k2[2 * q + 1] > k2[2 * q];  // strictly larger: ties keep the lower slot
      k2[q] = right ? k2[2 * q + 1] : k2[2 * q];
      q2[q] = right ? q2[2 * q + 1] : q2[2 * q];
    }
  bk = k2[0];
  bq = q2[0];
}

// One warp: top-k of one token.  E <= 32 NQ: lane holds the keys of experts
// lane + 32 q in registers.  Each round takes the largest key over the warp
// (one redux), then the lowest expert id among the lanes holding it (a
// second redux): logit descending, ties to the lower id.  Only the winning
// lane rescans its keys.
template <int NQ>
__device__ void topk_warp(const float* __restrict__ logits_row, int E, int k, int32_t* idx_out, float* w_out,
                          int32_t* idx_out2, float* w_out2) {
  const int lane = threadIdx.x & 31;
  // lane holds experts lane * NQ + q (q < NQ): consecutive logits, loaded as float4 when whole
  uint32_t key[NQ];
  if (E == 32 * NQ) {
#pragma unroll
    for (int q4 = 0; q4 < NQ / 4; ++q4) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(logits_row + lane * NQ) + q4);
      key[4 * q4] = ord_key(v.x);
      key[4 * q4 + 1] = ord_key(v.y);
      key[4 * q4 + 2] = ord_key(v.z);
      key[4 * q4 + 3] = ord_key(v.w);
    }
  } else {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const int e = lane * NQ + q;
      key[q] = (e < E) ? ord_key(__ldcg(logits_row + e)) : 0u;
    }
  }
  uint32_t bk;
  int bq;
  lane_best<NQ>(key, bk, bq);
  uint32_t my_key = 0u, key0 = 0u;
  int my_i = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, bk);
    const uint32_t id = __reduce_min_sync(0xFFFFFFFFu, bk == m ? (uint32_t)(lane * NQ + bq) : 0xFFFFFFFFu);
    if ((int)(id / NQ) == lane) {  // this lane's candidate won: drop it, find the next one
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        if (q == bq) key[q] = 0u;
      lane_best<NQ>(key, bk, bq);
    }
    if (j == 0) key0 = m;
    if (lane == j) { my_key = m; my_i = (int)id; }
  }
  // w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0); lane j holds term j, the sum
  // is a fixed butterfly over the warp (lanes >= k contribute 0)
  const float my_ex = lane < k ? expf(ord_value(my_key) - ord_value(key0)) : 0.f;
  float sum = my_ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  if (lane < k) {
    const float w = my_ex / sum;
    idx_out[lane] = my_i;
    w_out[lane] = w;
    if (idx_out2) idx_out2[lane] = my_i;
    if (w_out2) w_out2[lane] = w;
  }
}

// Logits of this CTA's expert rows; returns after writing them to global memory.
// The tokens are staged once per CTA in shared memory (x_s, [T][H] bf16) and
// every lane holds its router-weight chunk in registers before the
// float-float loop, so the loop itself issues no global loads.
__device__ void router_logits_cta(const RouterArgs& a, const uint16_t* x_s, float (*s_hi)[kMaxT],
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
    const uint16_t* xp = x_s + (size_t)part * Hw;
    constexpr int kPre = 4;  // float4 chunks of the row held per lane at once
    for (int base = lane; base < Hw / 4; base += 32 * kPre) {
      float4 wv[kPre];
#pragma unroll
      for (int j = 0; j < kPre; ++j)
        if (base + 32 * j < Hw / 4) wv[j] = __ldg(wrow + base + 32 * j);
#pragma unroll
      for (int j = 0; j < kPre; ++j) {
        const int h4 = base + 32 * j;
        if (h4 < Hw / 4) {
#pragma unroll
          for (int t = 0; t < kMaxT; ++t) {
            if (t < T) {
              const uint2 xv = *reinterpret_cast<const uint2*>(xp + (size_t)t * H + h4 * 4);
              dot2_step(bf16_bits_to_float(xv.x & 0xFFFF), wv[j].x, hi[t], lo[t]);
              dot2_step(bf16_bits_to_float(xv.x >> 16), wv[j].y, hi[t], lo[t]);
              dot2_step(bf16_bits_to_float(xv.y & 0xFFFF), wv[j].z, hi[t], lo[t]);
              dot2_step(bf16_bits_to_float(xv.y >> 16), wv[j].w, hi[t], lo[t]);
            }
          }
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
  extern __shared__ __align__(16) uint8_t smem[];  // dispatch scratch of the last CTA
  __shared__ float s_hi[kWarpsR][kMaxT], s_lo[kWarpsR][kMaxT];
  __shared__ int is_last;
  const int H = a.H, E = a.E, T = a.T, k = a.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the expert kernel that follows may be scheduled now: it stages the
  // activations and then waits for this grid's results (griddepcontrol.wait)
  asm volatile("griddepcontrol.launch_dependents;");
  {
    // stage the tokens (bf16 [T][H]) in shared memory
    const uint4* xs = reinterpret_cast<const uint4*>(a.x);
    uint4* xd = reinterpret_cast<uint4*>(smem);
    for (int i = tid; i < T * H / 8; i += blockDim.x) xd[i] = __ldg(xs + i);
  }
  __syncthreads();
  router_logits_cta(a, reinterpret_cast<const uint16_t*>(smem), s_hi, s_lo);

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

  for (int t = warp; t < T; t += kWarpsR) {
    const float* lr = a.rb.logits + (size_t)t * E;
    int32_t* io = a.rb.topk_idx + t * k;
    float* wo = a.rb.topk_w + t * k;
    int32_t* io2 = a.out.topk_idx ? a.out.topk_idx + t * k : nullptr;
    float* wo2 = a.out.topk_w ? a.out.topk_w + t * k : nullptr;
    if (E <= 256) topk_warp<8>(lr, E, k, io, wo, io2, wo2);
    else if (E <= 512) topk_warp<16>(lr, E, k, io, wo, io2, wo2);
    else topk_warp<32>(lr, E, k, io, wo, io2, wo2);
  }
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
  {
    // exclusive scan over the E counts and over the active flags, by the whole
    // CTA: each thread owns up to four consecutive experts
    __shared__ int s_wsum[kWarpsR][2];
    const int per = (E + kRouterThreads - 1) / kRouterThreads;  // <= 4 for E <= 1024
    const int e0 = tid * per;
    int c4[4], tot = 0, act = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e2 = e0 + q;
      c4[q] = (q < per && e2 < E) ? s_cnt[e2] : 0;
      tot += c4[q];
      act += c4[q] > 0;
    }
    int incl = tot, ainc = act;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      const int va = __shfl_up_sync(0xFFFFFFFFu, ainc, o);
      if (lane >= o) { incl += v; ainc += va; }
    }
    if (lane == 31) { s_wsum[warp][0] = incl; s_wsum[warp][1] = ainc; }
    __syncthreads();
    int wbase = 0, abase = 0;
    for (int w2 = 0; w2 < warp; ++w2) { wbase += s_wsum[w2][0]; abase += s_wsum[w2][1]; }
    int run = wbase + incl - tot, run_act = abase + ainc - act;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e2 = e0 + q;
      if (q < per && e2 < E) {
        s_off[e2] = run;
        a.rb.cnt[e2] = c4[q];
        if (a.out.cnt) a.out.cnt[e2] = c4[q];
        if (c4[q] > 0) a.rb.act[run_act++] = e2;
        run += c4[q];
      }
    }
    if (tid == kRouterThreads - 1) {
      s_off[E] = run;
      a.rb.ctrl->n_active = run_act;
    }
  }
  __syncthreads();
  for (int i = tid; i <= E; i += blockDim.x) {
    a.rb.off[i] = s_off[i];
    if (a.out.off) a.out.off[i] = s_off[i];
  }
  __syncthreads();  // the offsets are out: s_off now serves as the running position
  // pair positions: one warp walks the pairs in order, 32 at a time; equal
  // experts within a batch are ranked by lane (match_any), s_off[e] advances
  if (warp == 0) {
    for (int b = 0; b < P; b += 32) {
      const int p = b + lane;
      const int ex = p < P ? s_idx[p] : -1 - lane;
      const uint32_t peers = __match_any_sync(0xFFFFFFFFu, ex);
      if (p < P) {
        const int pos = s_off[ex] + __popc(peers & ((1u << lane) - 1u));
        a.rb.pair[pos] = p;
        if (a.out.pair) a.out.pair[pos] = p;
      }
      __syncwarp();
      if (p < P && lane == 31 - __clz(peers)) s_off[ex] += __popc(peers);
      __syncwarp();
    }
  }
  if (tid == 0) {
    a.rb.ctrl->router_arrive = 0;  // leave the counter at zero for the next call
    a.rb.ctrl->gu_next = 0;        // task counter of the gate/up kernel that follows
  }
}

// ---------------------------------------------------------------- prefill --
// One warp per token.  The approximate logit a of expert e carries the bound
// eps = gamma_H ||x_t|| ||Wr_e|| (sequential FMA sum of exact products,
// Cauchy-Schwarz for sum |x w|), widened for the FP32 bias additions.  L is
// the k-th largest lower bound a - eps; an expert whose upper bound a + eps
// is below L has an exact logit below the k-th largest exact logit, so only
// the others (at least k) get exact float-float logits.  The row of the
// logits buffer then holds the exact logit of every candidate and -inf
// elsewhere, and the decode path's top-k runs on it.
template <int NQ>
__device__ void prefill_topk_token(const PrefillArgs& a, int t) {
  const int lane = threadIdx.x & 31;
  const int E = a.E, H = a.H, k = a.k;
  float* row = a.rb.logits + (size_t)t * E;
  const float u = 5.9604645e-8f;  // 2^-24
  const float gam = (float)H * u / (1.f - (float)H * u);
  const float xn = a.xnorm[t];
  float av[NQ], ev[NQ];
  unsigned long long lo_key[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int e = q * 32 + lane;
    av[q] = 0.f;
    ev[q] = 0.f;
    lo_key[q] = 0ull;
    if (e < E) {
      const float d = row[e];
      const float b = a.bias ? __ldg(a.bias + e) : 0.f;
      const float ab = __fadd_rn(d, b);
      // tensor-core logits: twice the FMA-chain bound plus the bf16 split residual
      const float g_e = a.logits_tc ? 2.f * gam + 7.62939453125e-06f : gam;
      const float eps0 = g_e * xn * a.wnorm[e] * 1.00390625f;
      const float eps = eps0 + 4.7683716e-7f * (fabsf(d) + fabsf(b) + eps0) + 1e-30f;
      av[q] = ab;
      ev[q] = eps;
      lo_key[q] = sel_key(ab - eps, e);
    }
  }
  // k-th largest lower bound
  unsigned long long mine = lane_max<NQ>(lo_key), kth = 0ull;
  for (int j = 0; j < k; ++j) {
    unsigned long long best = mine;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = umax64(best, __shfl_xor_sync(0xFFFFFFFFu, best, o));
    if (best == mine) {
      const int bi = key_id(best);
#pragma unroll
      for (int q = 0; q < NQ; ++q)
        if (q == (bi >> 5)) lo_key[q] = 0ull;
      mine = lane_max<NQ>(lo_key);
    }
    kth = best;
  }
  const float L = key_value(kth);
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int e_mine = q * 32 + lane;
    const bool cand = e_mine < E && !(av[q] + ev[q] < L);
    uint32_t bal = __ballot_sync(0xFFFFFFFFu, cand);
    if (e_mine < E && !cand) row[e_mine] = __int_as_float(0xFF800000);  // -inf
    while (bal) {
      const int src = __ffs(bal) - 1;
      bal &= bal - 1;
      const int e = q * 32 + src;
      // exact logit of expert e: float-float over H, lanes on consecutive float4 columns
      const float4* wrow = reinterpret_cast<const float4*>(a.rw + (size_t)e * H);
      const uint2* xp = reinterpret_cast<const uint2*>(a.x + (size_t)t * H);
      float hi = 0.f, lo = 0.f;
#pragma unroll 4
      for (int c = lane; c < H / 4; c += 32) {
        const float4 wv = __ldg(wrow + c);
        const uint2 xv = __ldg(xp + c);
        dot2_step(bf16_bits_to_float(xv.x & 0xFFFF), wv.x, hi, lo);
        dot2_step(bf16_bits_to_float(xv.x >> 16), wv.y, hi, lo);
        dot2_step(bf16_bits_to_float(xv.y & 0xFFFF), wv.z, hi, lo);
        dot2_step(bf16_bits_to_float(xv.y >> 16), wv.w, hi, lo);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xFFFFFFFFu, hi, o);
        const float l2 = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
        dot2_merge(hi, lo, h2, l2);
      }
      float lg = __fadd_rn(hi, lo);
      if (a.bias) lg = __fadd_rn(lg, __ldg(a.bias + e));
      const float aq = __shfl_sync(0xFFFFFFFFu, av[q], src), eq = __shfl_sync(0xFFFFFFFFu, ev[q], src);
      if (lane == 0) {
        row[e] = lg;
        if (fabsf(lg - aq) > eq && lg == lg) report_error(a.rb.ctrl, (uint32_t)MOE_ERR_DEVICE_BAD_INDEX, 0x200);
      }
    }
  }
  __syncwarp();
  int32_t* io = a.rb.topk_idx + (size_t)t * k;
  float* wo = a.rb.topk_w + (size_t)t * k;
  int32_t* io2 = a.out.topk_idx ? a.out.topk_idx + (size_t)t * k : nullptr;
  float* wo2 = a.out.topk_w ? a.out.topk_w + (size_t)t * k : nullptr;
  topk_warp<NQ>(row, E, k, io, wo, io2, wo2);
}

__global__ void __launch_bounds__(kRouterThreads, 1) prefill_topk_kernel(PrefillArgs a) {
  const int t = blockIdx.x * kWarpsR + (threadIdx.x >> 5);
  if (t >= a.T) return;
  if (a.E <= 256) prefill_topk_token<8>(a, t);
  else if (a.E <= 512) prefill_topk_token<16>(a, t);
  else prefill_topk_token<32>(a, t);
}

}  // namespace

// Warps sharing one expert row: split H (up to all 8 warps of a CTA) while
// every warp keeps at least 256 columns (two float4 per lane) and the grid
// (E * w / 8 CTAs) still fits one wave of two CTAs per SM.
int router_warps_per_row(int H, int E, int sms) {
  int w = 1;
  while (w < kWarpsR && H % (4 * 32 * w * 2) == 0 && H / (w * 2) >= 256 &&
         (long)E * (w * 2) <= (long)kWarpsR * 2 * sms)
    w *= 2;
  return w;
}

cudaError_t launch_router_decode(const RouterArgs& a, cudaStream_t s) {
  const int rows_per_cta = kWarpsR / a.wpr;
  const int grid = (a.E + rows_per_cta - 1) / rows_per_cta;
  // dispatch scratch of the last CTA, or the staged tokens before it (aliased)
  const size_t disp = (size_t)(2 * a.E + 1 + a.T * a.k) * 4, xbytes = (size_t)a.T * a.H * 2;
  const size_t smem = disp > xbytes ? disp : xbytes;
  cudaError_t err = cudaFuncSetAttribute(router_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  router_decode_kernel<<<grid, kRouterThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_topk(const PrefillArgs& a, cudaStream_t s) {
  prefill_topk_kernel<<<(a.T + kWarpsR - 1) / kWarpsR, kRouterThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace qmoe
