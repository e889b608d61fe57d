// Router and dispatch for decode-sized batches (T <= 8).
//
// Stage 1 (every SM): approximate FP32 logits by FMA with a rigorous error
// bound, and the router rows' norms.  Stage 2 (one CTA per token): the
// experts that can still reach the top-k (upper bound not below the k-th
// largest lower bound) get the correctly rounded FP32 logit, a float-float
// (Dot2) dot product rounded once; top-k with the fixed tie rule runs on those
// exact logits, and the last CTA to finish (arrival counter, no spinning)
// builds the dispatch index: per-expert counts, offsets, the pair list as a
// stable counting sort, and the active experts.  The result equals selecting
// from exact logits of every expert.
//
// DGPP README "Execution and performance": engine.expert_tile_list (routed
// segments per expert); the top-k tie rule (logit descending, lower expert
// id first) keeps routing deterministic (DGPP README intro bullet "Exact").
#include "kernels.cuh"

namespace qmoe {

namespace {

constexpr int kMaxT = MOE_DECODE_MAX_TOKENS;
constexpr int kWarpsR = kRouterThreads / 32;
constexpr int kSelThreads = 512;  // threads of the per-token selection and of the one-CTA dispatch kernels
constexpr int kSelWarps = kSelThreads / 32;

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
                          int32_t* idx_out2, float* w_out2, const float* __restrict__ wrow = nullptr) {
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
  // is a fixed butterfly over the warp (lanes >= k contribute 0).  With wrow
  // the weights use wrow's logits of the selected experts (bias_select).
  float lj = ord_value(my_key), l0 = ord_value(key0);
  if (wrow) {
    const int id0 = __shfl_sync(0xFFFFFFFFu, my_i, 0);
    lj = lane < k ? __ldcg(wrow + my_i) : 0.f;
    l0 = __ldcg(wrow + id0);
  }
  const float my_ex = lane < k ? expf(lj - l0) : 0.f;
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

// Bitonic sort of one 64-bit key per lane across the warp, descending: after
// it lane j holds the (j+1)-th largest key.  15 compare-exchange steps of a
// shuffle each, instead of one warp reduction per extracted element.
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, v, stride);
      // descending overall: within a bitonic block of `size`, the lower lane keeps the larger key when
      // the block sorts descending (bit `size` of the lane is 0), the smaller one otherwise
      const bool lower = (lane & stride) == 0;
      const bool desc = (lane & size) == 0;
      const bool keep_max = lower == desc;
      v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// Counting-sort dispatch of the T*k routed pairs (one CTA, any block size):
// per-expert counts, offsets (exclusive scan over E), the pair list grouped by
// expert in ascending pair id (a stable counting sort), and the active experts
// in ascending id.  Expert ids outside [0, E) are reported and left out.
// Scratch: s_cnt [E], s_off [E + 1], s_idx [T*k] in shared memory.
__device__ void dispatch_cta(const RouteBufs& rb, const RouteOut& out, int E, int P, int32_t* s_cnt,
                             int32_t* s_off, int32_t* s_idx) {
  __shared__ int s_wsum[32][2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x, nwarp = nthr >> 5;
  for (int i = tid; i < E; i += nthr) s_cnt[i] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += nthr) {
    int ex = __ldcg(rb.topk_idx + p);
    if ((unsigned)ex >= (unsigned)E) {
      report_error(rb.ctrl, (uint32_t)MOE_ERR_DEVICE_BAD_INDEX, 0x010);
      ex = -1;
    } else {
      atomicAdd(&s_cnt[ex], 1);
    }
    s_idx[p] = ex;
  }
  __syncthreads();
  {
    // exclusive scan over the counts and over the active flags; each thread owns up to four experts
    const int per = (E + nthr - 1) / nthr;  // <= 4 for E <= 1024 and >= 256 threads
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
        rb.cnt[e2] = c4[q];
        if (out.cnt) out.cnt[e2] = c4[q];
        if (c4[q] > 0) rb.act[run_act++] = e2;
        run += c4[q];
      }
    }
    if (tid == nthr - 1) {
      s_off[E] = run;
      rb.ctrl->n_active = run_act;
    }
    (void)nwarp;
  }
  __syncthreads();
  for (int i = tid; i <= E; i += nthr) {
    rb.off[i] = s_off[i];
    if (out.off) out.off[i] = s_off[i];
  }
  __syncthreads();  // the offsets are out: s_off now serves as the running position
  // pair positions: one warp walks the pairs in order, 32 at a time; equal
  // experts within a batch are ranked by lane (match_any), s_off[e] advances
  if (warp == 0) {
    for (int b = 0; b < P; b += 32) {
      const int p = b + lane;
      const int ex0 = p < P ? s_idx[p] : -1;
      const int ex = ex0 >= 0 ? ex0 : -1 - lane;
      const uint32_t peers = __match_any_sync(0xFFFFFFFFu, ex);
      if (ex >= 0) {
        const int pos = s_off[ex] + __popc(peers & ((1u << lane) - 1u));
        rb.pair[pos] = p;
        if (out.pair) out.pair[pos] = p;
      }
      __syncwarp();
      if (ex >= 0 && lane == 31 - __clz(peers)) s_off[ex] += __popc(peers);
      __syncwarp();
    }
  }
}

// ---- experts-only calls: the caller's routing -------------------------------
// One CTA: copies the caller's top-k indices and weights into the workspace
// and computes the shared expert's gate per token when the layer has one (one
// warp per token, the exact float-float dot product).  The gate/up kernel
// builds the dispatch index from the copied ids and reports any outside
// [0, E) as MOE_ERR_DEVICE_BAD_INDEX.
__global__ void __launch_bounds__(kSelThreads) dispatch_ext_kernel(RouterArgs a, const int32_t* idx_in,
                                                                    const float* w_in) {
  const int E = a.E, T = a.T, k = a.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  asm volatile("griddepcontrol.launch_dependents;");
  for (int p = tid; p < T * k; p += kSelThreads) {
    a.rb.topk_idx[p] = __ldg(idx_in + p);
    a.rb.topk_w[p] = __ldg(w_in + p);
  }
  if (a.sgate_w) {
    for (int t = warp; t < T; t += kSelWarps) {
      const float4* wrow = reinterpret_cast<const float4*>(a.sgate_w);
      const uint2* xp = reinterpret_cast<const uint2*>(a.x + (size_t)t * a.H);
      float hi = 0.f, lo = 0.f;
      for (int q = lane; q < a.H / 4; q += 32) {
        const float4 wv = __ldg(wrow + q);
        const uint2 xv = __ldg(xp + q);
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
      if (lane == 0) a.sgate[t] = 1.f / (1.f + expf(-__fadd_rn(hi, lo)));
    }
  }
  (void)E;
}

// ---- decode router, stage 1: exact logits of every expert on every SM -------
// Each expert row (and, as row E, the shared expert's gate vector) is split
// over `wpr` warps; a lane owns 8-column chunks of its warp's share, issues
// every weight load of the batch before using any, and accumulates each
// token's dot product as a float-float pair (Dot2: the product split exactly
// by FMA, the sum by TwoSum).  The pairs are merged across lanes and then
// across the row's warps in a fixed order and rounded once: the correctly
// rounded FP32 logit unless the exact sum lies within about 2^-44 (relative)
// of a rounding midpoint.
constexpr int kLogitChunks = 2;  // 8-column chunks a lane holds in flight at once

__global__ void __launch_bounds__(kRouterThreads) router_decode_kernel(RouterArgs a) {
  __shared__ float s_hi[kWarpsR][kMaxT], s_lo[kWarpsR][kMaxT];
  const int H = a.H, E = a.E, T = a.T, wpr = a.wpr;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the selection kernel may start now (it waits for these logits)
  asm volatile("griddepcontrol.launch_dependents;");
  const int rows = E + (a.sgate_w ? 1 : 0);
  const int rows_per_cta = kWarpsR / wpr;
  const int e = blockIdx.x * rows_per_cta + warp / wpr;
  const int part = warp % wpr;
  const int Hw = H / wpr, nch = Hw / 8;
  float hi[kMaxT], lo[kMaxT];
#pragma unroll
  for (int t = 0; t < kMaxT; ++t) { hi[t] = 0.f; lo[t] = 0.f; }
  if (e < rows) {
    const float* wrow = (e < E ? a.w + (size_t)e * H : a.sgate_w) + (size_t)part * Hw;
    const uint16_t* xp = a.x + (size_t)part * Hw;
    for (int c0 = lane; c0 < nch; c0 += 32 * kLogitChunks) {
      // every load of this batch (weights, and the tokens' matching columns, clamped to a
      // valid token so no load waits behind a branch) is issued before any is used
      float4 wv[kLogitChunks][2];
      uint4 xv[kLogitChunks][kMaxT];
#pragma unroll
      for (int j = 0; j < kLogitChunks; ++j) {
        const int c = min(c0 + 32 * j, nch - 1);
        wv[j][0] = __ldg(reinterpret_cast<const float4*>(wrow + 8 * c));
        wv[j][1] = __ldg(reinterpret_cast<const float4*>(wrow + 8 * c + 4));
#pragma unroll
        for (int t = 0; t < kMaxT; ++t)
          xv[j][t] = __ldg(reinterpret_cast<const uint4*>(xp + (size_t)min(t, T - 1) * H + 8 * c));
      }
#pragma unroll
      for (int j = 0; j < kLogitChunks; ++j) {
        if (c0 + 32 * j < nch) {
          const float w8[8] = {wv[j][0].x, wv[j][0].y, wv[j][0].z, wv[j][0].w,
                               wv[j][1].x, wv[j][1].y, wv[j][1].z, wv[j][1].w};
#pragma unroll
          for (int t = 0; t < kMaxT; ++t) {
            if (t < T) {
              const uint32_t xw[4] = {xv[j][t].x, xv[j][t].y, xv[j][t].z, xv[j][t].w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                dot2_step(bf16_bits_to_float(xw[i] & 0xFFFF), w8[2 * i], hi[t], lo[t]);
                dot2_step(bf16_bits_to_float(xw[i] >> 16), w8[2 * i + 1], hi[t], lo[t]);
              }
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int t = 0; t < kMaxT; ++t)
      if (t < T) {
        const float h2 = __shfl_xor_sync(0xFFFFFFFFu, hi[t], o);
        const float l2 = __shfl_xor_sync(0xFFFFFFFFu, lo[t], o);
        dot2_merge(hi[t], lo[t], h2, l2);
      }
  }
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) { s_hi[warp][t] = hi[t]; s_lo[warp][t] = lo[t]; }
  }
  __syncthreads();
  // the first warp of each row merges the row's parts in order and rounds once
  if (e < rows && part == 0 && lane < T) {
    float h = s_hi[warp][lane], l = s_lo[warp][lane];
    for (int p = 1; p < wpr; ++p) dot2_merge(h, l, s_hi[warp + p][lane], s_lo[warp + p][lane]);
    const float lg = __fadd_rn(h, l);
    if (e == E) {
      a.sgate[lane] = 1.f / (1.f + expf(-lg));  // the shared expert's sigmoid gate
    } else {
      const float lb = a.bias ? __fadd_rn(lg, __ldg(a.bias + e)) : lg;
      a.rb.logits[(size_t)lane * E + e] = lb;
      if (a.bias_select) a.approx[(size_t)lane * E + e] = lg;
    }
  }
}

// ---- decode router, stage 2: top-k of each token (one CTA per token) --------
// One thread per expert (two when E > 512), keys (logit descending, expert id
// ascending) from the exact logits of stage 1.  L = the k-th largest of the
// per-warp top-2 keys is at most the k-th largest key, so the keys >= L (at
// least k, typically a dozen) contain the top k; up to 32 of them are sorted
// by one warp bitonic sort, more (flat or tied logits) are taken by rounds of
// warp maxima.  The weights are the renormalised softmax of the chosen logits
// (the unbiased ones under bias_select).
__global__ void __launch_bounds__(kSelThreads) router_select_kernel(RouterArgs a) {
  __shared__ unsigned long long s_top2[kSelWarps][2];
  __shared__ unsigned long long s_cand[2 * kSelThreads];
  __shared__ unsigned long long s_L;
  __shared__ int s_ncand;
  const int E = a.E, k = a.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.x;
  asm volatile("griddepcontrol.launch_dependents;");
  if (tid == 0) s_ncand = 0;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  unsigned long long key[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int e = tid + r * kSelThreads;
    key[r] = e < E ? (((unsigned long long)ord_key(__ldcg(a.rb.logits + (size_t)t * E + e)) << 32) |
                      (uint32_t)~(uint32_t)e)
                   : 0ull;
  }
  {  // the warp's two largest keys
    unsigned long long best = key[0] > key[1] ? key[0] : key[1];
    const unsigned long long other = key[0] > key[1] ? key[1] : key[0];
    const uint32_t h1 = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(best >> 32));
    const uint32_t l1 = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(best >> 32) == h1 ? (uint32_t)best : 0u);
    const unsigned long long m1 = ((unsigned long long)h1 << 32) | l1;
    if (best == m1) best = other;  // keys are unique: the holder drops its maximum
    const uint32_t h2 = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(best >> 32));
    const uint32_t l2 = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(best >> 32) == h2 ? (uint32_t)best : 0u);
    if (lane == 0) { s_top2[warp][0] = m1; s_top2[warp][1] = ((unsigned long long)h2 << 32) | l2; }
  }
  __syncthreads();
  if (warp == 0) {
    const unsigned long long v = warp_sort_desc(lane < 2 * kSelWarps ? s_top2[lane >> 1][lane & 1] : 0ull);
    const unsigned long long L = __shfl_sync(0xFFFFFFFFu, v, k - 1);
    if (lane == 0) s_L = L;
  }
  __syncthreads();
  const unsigned long long L = s_L;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const bool cand = key[r] != 0ull && key[r] >= L;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, cand);
    int base = 0;
    if (lane == 0 && bal) base = atomicAdd(&s_ncand, __popc(bal));
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    if (cand) s_cand[base + __popc(bal & ((1u << lane) - 1u))] = key[r];
  }
  __syncthreads();
  if (warp != 0) return;
  const int nc = s_ncand;
  unsigned long long my_key = 0ull;
  if (nc <= 32) {
    my_key = warp_sort_desc(lane < nc ? s_cand[lane] : 0ull);  // lane j: the (j+1)-th largest
  } else {
    // flat or tied logits: rounds of the warp maximum; a lane holds candidates lane + 32 q
    for (int j = 0; j < k; ++j) {
      unsigned long long b = 0ull;
      int bc = -1;
      for (int c = lane; c < nc; c += 32)
        if (s_cand[c] > b) { b = s_cand[c]; bc = c; }
      const uint32_t mhi = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(b >> 32));
      const uint32_t mlo = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(b >> 32) == mhi ? (uint32_t)b : 0u);
      const unsigned long long m = ((unsigned long long)mhi << 32) | mlo;
      if (bc >= 0 && b == m) s_cand[bc] = 0ull;  // keys are unique: one lane holds the maximum
      __syncwarp();
      if (lane == j) my_key = m;
    }
  }
  const int my_e = (int)~(uint32_t)my_key;
  const int e0 = __shfl_sync(0xFFFFFFFFu, my_e, 0);
  float lj = ord_value((uint32_t)(my_key >> 32));
  float l0 = __shfl_sync(0xFFFFFFFFu, lj, 0);
  if (a.bias_select) {  // the bias steered the choice only: the weights use the unbiased logits
    lj = lane < k ? __ldcg(a.approx + (size_t)t * E + my_e) : 0.f;
    l0 = __ldcg(a.approx + (size_t)t * E + e0);
  }
  const float my_ex = lane < k ? expf(lj - l0) : 0.f;
  float sum = my_ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  if (lane < k) {
    const float w = my_ex / sum;
    a.rb.topk_idx[t * k + lane] = my_e;
    a.rb.topk_w[t * k + lane] = w;
    if (a.out.topk_idx) a.out.topk_idx[t * k + lane] = my_e;
    if (a.out.topk_w) a.out.topk_w[t * k + lane] = w;
  }
}


// moe_route (T <= 8): the dispatch index of the router's choices (one CTA)
__global__ void __launch_bounds__(kSelThreads) route_dispatch_kernel(RouterArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  int32_t* s_dcnt = reinterpret_cast<int32_t*>(smem);
  int32_t* s_doff = s_dcnt + a.E;
  int32_t* s_didx = s_doff + a.E + 1;
  dispatch_cta(a.rb, a.out, a.E, a.T * a.k, s_dcnt, s_doff, s_didx);
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
      const float lu = __fadd_rn(hi, lo);
      const float lg = a.bias ? __fadd_rn(lu, __ldg(a.bias + e)) : lu;
      const float aq = __shfl_sync(0xFFFFFFFFu, av[q], src), eq = __shfl_sync(0xFFFFFFFFu, ev[q], src);
      if (lane == 0) {
        row[e] = lg;
        if (a.bias_select) a.unbiased[(size_t)t * E + e] = lu;
        if (fabsf(lg - aq) > eq && lg == lg) report_error(a.rb.ctrl, (uint32_t)MOE_ERR_DEVICE_BAD_INDEX, 0x200);
      }
    }
  }
  __syncwarp();
  int32_t* io = a.rb.topk_idx + (size_t)t * k;
  float* wo = a.rb.topk_w + (size_t)t * k;
  int32_t* io2 = a.out.topk_idx ? a.out.topk_idx + (size_t)t * k : nullptr;
  float* wo2 = a.out.topk_w ? a.out.topk_w + (size_t)t * k : nullptr;
  __syncwarp();
  topk_warp<NQ>(row, E, k, io, wo, io2, wo2, a.bias_select ? a.unbiased + (size_t)t * E : nullptr);
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
  const int rows = a.E + (a.sgate_w ? 1 : 0);
  router_decode_kernel<<<(rows + rows_per_cta - 1) / rows_per_cta, kRouterThreads, 0, s>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.T);
  cfg.blockDim = dim3(kSelThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, router_select_kernel, a);
}

cudaError_t launch_dispatch_ext(const RouterArgs& a, const int32_t* idx, const float* w, cudaStream_t s) {
  dispatch_ext_kernel<<<1, kSelThreads, 0, s>>>(a, idx, w);
  return cudaGetLastError();
}

cudaError_t launch_route_dispatch(const RouterArgs& a, cudaStream_t s) {
  const size_t smem = ((size_t)2 * a.E + 1 + (size_t)a.T * a.k) * 4;
  route_dispatch_kernel<<<1, kSelThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_topk(const PrefillArgs& a, cudaStream_t s) {
  prefill_topk_kernel<<<(a.T + kWarpsR - 1) / kWarpsR, kRouterThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace qmoe
