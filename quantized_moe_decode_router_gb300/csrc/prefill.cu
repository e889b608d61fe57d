// Prefill-sized routing, dispatch and the element-wise steps around the
// expert GEMMs (any token count T).
//
// Router logits: an FP32 GEMM-like pass gives approximate logits a[t, e]
// with the classic bound for a sum of exact products accumulated by FMA in
// a fixed order, |a - dot| <= gamma_H * sum_h |x_h w_h| <= gamma_H *
// ||x_t|| ||Wr_e||.  Only experts whose interval can still reach the k-th
// largest lower bound are recomputed exactly (float-float, correctly
// rounded); every other expert provably ranks below the top-k (launch in
// router.cu).  Same result as the decode router: the exact FP32 logits
// decide the selection and the weights (DGPP README intro bullet "Exact";
// the tie rule logit descending, expert id ascending).
//
// Dispatch: per-chunk expert histograms, per-expert prefix over chunks and
// an exclusive scan over experts, then each chunk places its pairs in pair
// order, which gives the stable counting sort of the decode path for any T.
// The scan also emits the GEMM tile list: consecutive runs of at most
// kPfTokTile sorted positions of one expert (DGPP README "Execution and
// performance", engine.expert_tile_list).
#include <cuda_fp8.h>

#include "kernels.cuh"

namespace qmoe {

namespace {

constexpr int kThreads = 256;

// Exponent e with 2^e <= |v| < 2^(e+1) for the float bits of |v| (v != 0).
__device__ __forceinline__ int float_exponent(uint32_t abs_bits) {
  const int be = (int)(abs_bits >> 23);
  if (be > 0) return be - 127;
  return -127 - (__clz(abs_bits) - 9);  // subnormal
}

// Power-of-two exponent that lifts a row with largest magnitude amax into
// [2^14, 2^15): every element above 2^-31 of amax is exact in f16 after it.
__device__ __forceinline__ int f16_shift(uint32_t amax_bits) {
  if (amax_bits == 0) return 0;
  int s = 14 - float_exponent(amax_bits);
  return s > 100 ? 100 : s;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// One warp per token: max |x| (-> the f16 shift s) and ||x||_2.
__global__ void __launch_bounds__(kThreads) pf_prep_kernel(PrefillArgs a) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (t >= a.T) return;
  const int H = a.H;
  const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)t * H);
  uint32_t amax = 0;
  float ss = 0.f;
  for (int c = lane; c < H / 8; c += 32) {
    const uint4 v = __ldg(xr + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = bf16_bits_to_float(w[i] & 0xFFFF), hi = bf16_bits_to_float(w[i] >> 16);
      amax = max(amax, max(__float_as_uint(fabsf(lo)), __float_as_uint(fabsf(hi))));
      ss = fmaf(lo, lo, ss);
      ss = fmaf(hi, hi, ss);
    }
  }
  amax = __reduce_max_sync(0xFFFFFFFFu, amax);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  const int sft = f16_shift(amax);
  if (lane == 0) {
    a.xsig[t] = sft;
    a.xnorm[t] = sqrtf(ss);
  }
}

// One warp per expert: ||Wr_e||_2.
__global__ void __launch_bounds__(kThreads) pf_wnorm_kernel(PrefillArgs a) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (e >= a.E) return;
  const float4* wr = reinterpret_cast<const float4*>(a.rw + (size_t)e * a.H);
  float ss = 0.f;
  for (int c = lane; c < a.H / 4; c += 32) {
    const float4 v = __ldg(wr + c);
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  if (lane == 0) a.wnorm[e] = sqrtf(ss);
}

// Approximate logits: 64 tokens x 64 experts per CTA, each thread 4 x 4,
// every output a sequential FMA chain over h ascending (the order the error
// bound assumes).
constexpr int kLT = 64, kLE = 64, kLK = 32;

__global__ void __launch_bounds__(kThreads) pf_logits_kernel(PrefillArgs a) {
  __shared__ __align__(16) float sx[kLK][kLT + 4];
  __shared__ __align__(16) float sw[kLK][kLE + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.y * kLT, e0 = blockIdx.x * kLE;
  const int H = a.H, T = a.T, E = a.E;
  const int lr = tid >> 2, lc = (tid & 3) * 8;  // loader: row, first column
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < H; k0 += kLK) {
    {
      const int t = t0 + lr;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (t < T) v = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * H + k0 + lc));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sx[lc + 2 * i][lr] = bf16_bits_to_float(w[i] & 0xFFFF);
        sx[lc + 2 * i + 1][lr] = bf16_bits_to_float(w[i] >> 16);
      }
      const int e = e0 + lr;
      float4 w0 = make_float4(0.f, 0.f, 0.f, 0.f), w1 = w0;
      if (e < E) {
        const float4* wp = reinterpret_cast<const float4*>(a.rw + (size_t)e * H + k0 + lc);
        w0 = __ldg(wp);
        w1 = __ldg(wp + 1);
      }
      sw[lc + 0][lr] = w0.x; sw[lc + 1][lr] = w0.y; sw[lc + 2][lr] = w0.z; sw[lc + 3][lr] = w0.w;
      sw[lc + 4][lr] = w1.x; sw[lc + 5][lr] = w1.y; sw[lc + 6][lr] = w1.z; sw[lc + 7][lr] = w1.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kLK; ++kk) {
      const float4 xa = *reinterpret_cast<const float4*>(&sx[kk][ty * 4]);
      const float4 wb = *reinterpret_cast<const float4*>(&sw[kk][tx * 4]);
      const float xv[4] = {xa.x, xa.y, xa.z, xa.w}, wv[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) a.rb.logits[(size_t)t * E + e] = acc[i][j];
    }
  }
}

// Per-chunk expert histogram of the routed pairs.
__global__ void __launch_bounds__(kThreads) pf_hist_kernel(PrefillArgs a) {
  extern __shared__ int32_t s_h[];
  const int E = a.E, k = a.k;
  const int c = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_h[e] = 0;
  __syncthreads();
  const int p0 = c * kPfChunk * k;
  const int p1 = min(a.T, (c + 1) * kPfChunk) * k;
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = a.rb.topk_idx[p];
    if ((unsigned)e < (unsigned)E) atomicAdd(&s_h[e], 1);
    else report_error(a.rb.ctrl, (uint32_t)MOE_ERR_DEVICE_BAD_INDEX, 0x100);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) a.hist[(size_t)c * E + e] = s_h[e];
}

// One CTA: per-expert bases over chunks, counts, offsets, the GEMM tile
// list; clears the per-position |h| maxima of the gate/up epilogue.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) pf_scan_kernel(PrefillArgs a) {
  __shared__ int32_t s_wsum[kScanThreads / 32][2];
  const int E = a.E, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nchunk = (a.T + kPfChunk - 1) / kPfChunk;
  // E <= 1024: thread tid owns expert tid
  int cnt = 0;
  if (tid < E) {
    for (int c = 0; c < nchunk; ++c) {
      int32_t* hp = a.hist + (size_t)c * E + tid;
      const int v = *hp;
      *hp = cnt;
      cnt += v;
    }
  }
  const int ntile = (cnt + kPfTokTile - 1) / kPfTokTile;
  int inc = cnt, tinc = ntile;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, inc, o), tv = __shfl_up_sync(0xFFFFFFFFu, tinc, o);
    if (lane >= o) { inc += v; tinc += tv; }
  }
  if (lane == 31) { s_wsum[warp][0] = inc; s_wsum[warp][1] = tinc; }
  __syncthreads();
  int base = 0, tbase = 0;
  for (int w = 0; w < warp; ++w) { base += s_wsum[w][0]; tbase += s_wsum[w][1]; }
  const int off = base + inc - cnt, toff = tbase + tinc - ntile;
  if (tid < E) {
    a.rb.cnt[tid] = cnt;
    a.rb.off[tid] = off;
    if (a.out.cnt) a.out.cnt[tid] = cnt;
    if (a.out.off) a.out.off[tid] = off;
    for (int i = 0; i < ntile; ++i)
      if (toff + i < a.max_tiles) a.tiles[toff + i] = make_int2(tid, off + i * kPfTokTile);
    if (tid == E - 1) {
      a.rb.off[E] = off + cnt;
      if (a.out.off) a.out.off[E] = off + cnt;
      const int nt = toff + ntile;
      if (nt > a.max_tiles) report_error(a.rb.ctrl, (uint32_t)MOE_ERR_DEVICE_BAD_INDEX, 0x101);
      a.rb.ctrl->n_tiles = nt > a.max_tiles ? a.max_tiles : nt;
    }
  }
  if (a.h_amax)
    for (int i = tid; i < a.T * a.k; i += kScanThreads) a.h_amax[i] = 0u;
}

// One warp per chunk: place the chunk's pairs in pair order.
__global__ void __launch_bounds__(32) pf_place_kernel(PrefillArgs a) {
  extern __shared__ int32_t s_run[];
  const int E = a.E, k = a.k, lane = threadIdx.x;
  const int c = blockIdx.x;
  for (int e = lane; e < E; e += 32) s_run[e] = 0;
  __syncwarp();
  const int p0 = c * kPfChunk * k;
  const int p1 = min(a.T, (c + 1) * kPfChunk) * k;
  const int32_t* base = a.hist + (size_t)c * E;
  for (int b = p0; b < p1; b += 32) {
    const int p = b + lane;
    const bool valid = p < p1;
    int e = valid ? a.rb.topk_idx[p] : -1 - lane;
    if (valid && (unsigned)e >= (unsigned)E) e = -1 - lane;  // reported by the histogram pass
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0) {
      const int pos = a.rb.off[e] + base[e] + s_run[e] + rank;
      a.rb.pair[pos] = p;
      a.pos_of[p] = pos;
      if (a.out.pair) a.out.pair[pos] = p;
    }
    __syncwarp();
    if (e >= 0 && lane == 31 - __clz(peers)) s_run[e] += __popc(peers);
    __syncwarp();
  }
}

// One warp per sorted position: the GEMM operand row xg[pos] = f16( x[t] * 2^s_t ),
// t the token of the pair placed at pos (a contiguous copy per expert segment,
// so the gate/up GEMM loads its token tiles as plain 2-D boxes).  For the
// shared expert's argument block (dense_T > 0) position = token.
// Per-token 1x128 E4M3 quantisation of one BF16 row (the FP8-activation
// lever): per 128-element block s = amax / 448 and code = e4m3_rne_sat(v / s),
// both IEEE FP32 divisions (a negative value that rounds to zero keeps its
// sign: code 0x80); a zero block has scale 0 and +0 codes.  One warp, four
// elements per lane and block.  The result goes to ndst rows of the code and
// scale arrays: row r = the value of `dst` in lane r (ndst <= 32).
__device__ void quant_row_fp8(const uint16_t* src, int K, uint8_t* codes, float* scales, int dst, int ndst,
                              int lane) {
  for (int b = 0; b < K / 128; ++b) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(src + b * 128) + lane);
    const float v[4] = {bf16_bits_to_float(w.x & 0xFFFF), bf16_bits_to_float(w.x >> 16),
                        bf16_bits_to_float(w.y & 0xFFFF), bf16_bits_to_float(w.y >> 16)};
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const float sc = __fdiv_rn(m, 448.0f);
    uint32_t out = 0;
    if (sc > 0.f) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float q = __fdiv_rn(v[i], sc);
        uint32_t c = (uint32_t)__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3) & 0xFFu;
        c |= (__float_as_uint(q) >> 24) & 0x80u;  // the sign, also of a value that rounds to zero
        out |= c << (8 * i);
      }
    }
    for (int r = 0; r < ndst; ++r) {
      const int row = __shfl_sync(0xFFFFFFFFu, dst, r);
      reinterpret_cast<uint32_t*>(codes + (size_t)row * K + b * 128)[lane] = out;
      if (lane == 0) scales[(size_t)row * (K / 128) + b] = sc;
    }
  }
}

// The FP8-activation lever's token operand: one warp per token quantises its
// BF16 row once into E4M3 codes and scales and writes them to each of the
// token's sorted positions (dense: row t).
__global__ void __launch_bounds__(kThreads) pf_gather_fp8_kernel(PrefillArgs a) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (t >= a.T) return;
  const int rows = a.T * a.k;
  const int k = a.dense_T ? 1 : a.k;
  const int dst = a.dense_T ? t : (lane < k ? __ldg(a.pos_of + (size_t)t * k + lane) : 0);
  uint8_t* codes = reinterpret_cast<uint8_t*>(a.xg);
  quant_row_fp8(a.x + (size_t)t * a.H, a.H, codes, fp8_scales_after(codes, rows, a.H), dst, k, lane);
}

// The FP8-activation lever's h operand: each h row (BF16, after the gate/up
// epilogue) quantised into E4M3 codes and scales in the h16 buffer.
__global__ void __launch_bounds__(kThreads) pf_hquant_fp8_kernel(PrefillArgs a) {
  const int lane = threadIdx.x & 31;
  const int pos = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  const int rows = a.T * a.k;
  if (pos >= rows) return;
  uint8_t* codes = reinterpret_cast<uint8_t*>(a.h16);
  quant_row_fp8(a.h + (size_t)pos * a.I, a.I, codes, fp8_scales_after(codes, rows, a.I), pos, 1, lane);
}

__global__ void __launch_bounds__(kThreads) pf_gather_kernel(PrefillArgs a) {
  const int lane = threadIdx.x & 31;
  const int pos = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (pos >= a.T * a.k) return;
  const int H = a.H;
  const int t = a.dense_T ? pos : a.rb.pair[pos] / a.k;
  const uint4* xr = reinterpret_cast<const uint4*>(a.x + (size_t)t * H);
  uint4* xo = reinterpret_cast<uint4*>(a.xg + (size_t)pos * H);
  if (fold_lever(a)) {
    // the fold-scales lever's B operand: the BF16 row as it is
    for (int c = lane; c < H / 8; c += 32) xo[c] = __ldg(xr + c);
    return;
  }
  const float mul = exp2i(a.xsig[t]);
  for (int c = lane; c < H / 8; c += 32) {
    const uint4 v = __ldg(xr + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = pack_f16x2(bf16_bits_to_float(w[i] & 0xFFFF) * mul, bf16_bits_to_float(w[i] >> 16) * mul);
    xo[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// W4A4: one warp per sorted position copies the FP4 codes and block scales of
// its token (16-byte chunks for the codes, 8-byte chunks for the scales:
// H / 16 of them for NVFP4, H / 32 for MXFP4).
__global__ void __launch_bounds__(kThreads) pf_gather_q_kernel(PrefillArgs a) {
  const int lane = threadIdx.x & 31;
  const int pos = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (pos >= a.T * a.k) return;
  const int H = a.H;
  const int t = a.rb.pair[pos] / a.k;
  const uint4* cs = reinterpret_cast<const uint4*>(a.xq + (size_t)t * (H / 2));
  uint4* cd = reinterpret_cast<uint4*>(a.xqg + (size_t)pos * (H / 2));
  for (int c = lane; c < H / 32; c += 32) cd[c] = cs[c];
  const int sb = a.act_quant == 2 ? H / 32 : H / 16;  // scale bytes per row
  const uint2* ss = reinterpret_cast<const uint2*>(a.xsf + (size_t)t * sb);
  uint2* sd = reinterpret_cast<uint2*>(a.xsfg + (size_t)pos * sb);
  for (int c = lane; c < sb / 8; c += 32) sd[c] = ss[c];
}

// One warp per sorted position: h (bf16) -> f16 * 2^s, s from the row's max |h|
// (found here: the row spans several gate/up tiles).
__global__ void __launch_bounds__(kThreads) pf_hconv_kernel(PrefillArgs a) {
  const int lane = threadIdx.x & 31;
  const int pos = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (pos >= a.T * a.k) return;
  const int I = a.I;
  const uint4* hr = reinterpret_cast<const uint4*>(a.h + (size_t)pos * I);
  uint32_t amax = 0;
  for (int c = lane; c < I / 8; c += 32) {
    const uint4 v = hr[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = max(amax, max((w[i] & 0x7FFFu) << 16, (w[i] >> 16 & 0x7FFFu) << 16));
  }
  amax = __reduce_max_sync(0xFFFFFFFFu, amax);
  const int sft = f16_shift(amax);
  const float mul = exp2i(sft);
  uint4* ho = reinterpret_cast<uint4*>(a.h16 + (size_t)pos * I);
  for (int c = lane; c < I / 8; c += 32) {
    const uint4 v = hr[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = pack_f16x2(bf16_bits_to_float(w[i] & 0xFFFF) * mul, bf16_bits_to_float(w[i] >> 16) * mul);
    ho[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (lane == 0) a.hsig[pos] = sft;
}

// One warp per token: the sigmoid gate of a gated shared expert, from the
// correctly rounded FP32 logit x_t . w_gate (float-float dot, one rounding).
__global__ void __launch_bounds__(kThreads) pf_sgate_kernel(PrefillArgs a) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (t >= a.T) return;
  const int H = a.H;
  const uint2* xr = reinterpret_cast<const uint2*>(a.x + (size_t)t * H);
  const float4* wr = reinterpret_cast<const float4*>(a.sgate_w);
  float hi = 0.f, lo = 0.f;
  for (int q = lane; q < H / 4; q += 32) {
    const uint2 xv = __ldg(xr + q);
    const float4 wv = __ldg(wr + q);
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

// y[t] = bf16( sum_j w[t, j] * P[pos_of[t*k + j]] + g_t * S[t] ), j ascending, the
// shared term last (g_t = 1 unless the shared expert is gated); P and S in FP32,
// or in BF16 under the bf16-partials lever.
__global__ void __launch_bounds__(kThreads) pf_combine_kernel(PrefillArgs a) {
  const int t = blockIdx.x, H = a.H, k = a.k;
  const float* wt = a.rb.topk_w + (size_t)t * k;
  for (int c = threadIdx.x; c < H / 4; c += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float w = __ldg(wt + j);
      const int pos = __ldg(a.pos_of + (size_t)t * k + j);
      float4 p;
      if (a.p_bf16) {  // the bf16-partials lever: partials stored as BF16
        const uint2 v = __ldcs(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(a.P) + (size_t)pos * H) + c);
        p = make_float4(bf16_bits_to_float(v.x & 0xFFFF), bf16_bits_to_float(v.x >> 16), bf16_bits_to_float(v.y & 0xFFFF),
                        bf16_bits_to_float(v.y >> 16));
      } else {
        p = __ldcs(reinterpret_cast<const float4*>(a.P + (size_t)pos * H) + c);
      }
      acc.x = fmaf(w, p.x, acc.x);
      acc.y = fmaf(w, p.y, acc.y);
      acc.z = fmaf(w, p.z, acc.z);
      acc.w = fmaf(w, p.w, acc.w);
    }
    if (a.S) {
      const float g = a.sgate_w ? __ldg(a.sgate + t) : 1.f;
      float4 sv;
      if (a.p_bf16) {
        const uint2 v = __ldcs(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(a.S) + (size_t)t * H) + c);
        sv = make_float4(bf16_bits_to_float(v.x & 0xFFFF), bf16_bits_to_float(v.x >> 16), bf16_bits_to_float(v.y & 0xFFFF),
                         bf16_bits_to_float(v.y >> 16));
      } else {
        sv = __ldcs(reinterpret_cast<const float4*>(a.S + (size_t)t * H) + c);
      }
      acc.x = fmaf(g, sv.x, acc.x);
      acc.y = fmaf(g, sv.y, acc.y);
      acc.z = fmaf(g, sv.z, acc.z);
      acc.w = fmaf(g, sv.w, acc.w);
    }
    const uint32_t lo = (uint32_t)float_to_bf16_bits(acc.x) | ((uint32_t)float_to_bf16_bits(acc.y) << 16);
    const uint32_t hi = (uint32_t)float_to_bf16_bits(acc.z) | ((uint32_t)float_to_bf16_bits(acc.w) << 16);
    reinterpret_cast<uint2*>(a.y + (size_t)t * H)[c] = make_uint2(lo, hi);
  }
}

}  // namespace

cudaError_t launch_prefill_route(const PrefillArgs& a, cudaStream_t s, Marks mk) {
  const int wpb = kThreads / 32;
  pf_prep_kernel<<<(a.T + wpb - 1) / wpb, kThreads, 0, s>>>(a);
  pf_wnorm_kernel<<<(a.E + wpb - 1) / wpb, kThreads, 0, s>>>(a);
  if (a.logits_tc) {
    cudaError_t e1 = launch_prefill_logits_tc(a, s);
    if (e1 != cudaSuccess) return e1;
  } else {
    pf_logits_kernel<<<dim3((a.E + kLE - 1) / kLE, (a.T + kLT - 1) / kLT), kThreads, 0, s>>>(a);
  }
  mk(1);
  cudaError_t err = launch_prefill_topk(a, s);
  if (err != cudaSuccess) return err;
  mk(2);
  const int nchunk = (a.T + kPfChunk - 1) / kPfChunk;
  pf_hist_kernel<<<nchunk, kThreads, a.E * 4, s>>>(a);
  pf_scan_kernel<<<1, kScanThreads, 0, s>>>(a);
  pf_place_kernel<<<nchunk, 32, a.E * 4, s>>>(a);
  if (a.act_quant) {
    cudaError_t e2 = a.act_quant == 2 ? launch_quantize_act_mxfp4(a.x, a.T, a.H, a.xq, a.xsf, s)
                                      : launch_quantize_act_nvfp4(a.x, a.T, a.H, a.xq, a.xsf, s);
    if (e2 != cudaSuccess) return e2;
    pf_gather_q_kernel<<<(a.T * a.k + wpb - 1) / wpb, kThreads, 0, s>>>(a);
  } else if (a.xg) {
    if (fp8_lever(a)) pf_gather_fp8_kernel<<<(a.T + wpb - 1) / wpb, kThreads, 0, s>>>(a);
    else pf_gather_kernel<<<(a.T * a.k + wpb - 1) / wpb, kThreads, 0, s>>>(a);
  }
  mk(3);
  return cudaGetLastError();
}

cudaError_t launch_prefill_experts(const PrefillArgs& a, int sms, cudaStream_t s, Marks mk) {
  const int wpb = kThreads / 32;
  cudaError_t err;
  if (a.act_quant) {
    if ((err = launch_prefill_gemm_w4a4(false, a, sms, s)) != cudaSuccess) return err;
    mk(4);
    mk(5);
    if ((err = launch_prefill_gemm_w4a4(true, a, sms, s)) != cudaSuccess) return err;
    mk(6);
    pf_combine_kernel<<<a.T, kThreads, 0, s>>>(a);
    mk(7);
    return cudaGetLastError();
  }
  // the shared expert: one weight set over all T tokens in token order (its own argument block)
  PrefillArgs sa = a;
  if (a.sfmt) {
    sa.fmt = a.sfmt; sa.I = a.Is; sa.E = 1; sa.k = 1; sa.dense_T = a.T;
    sa.gate = a.s_gate; sa.up = a.s_up; sa.down = a.s_down;
    sa.xg = a.xs16; sa.h = a.hs; sa.h16 = a.hs16; sa.hsig = a.hssig; sa.P = a.S;
    if (fp8_lever(sa)) pf_gather_fp8_kernel<<<(a.T + wpb - 1) / wpb, kThreads, 0, s>>>(sa);
    else pf_gather_kernel<<<(a.T + wpb - 1) / wpb, kThreads, 0, s>>>(sa);
    if (a.sgate_w) pf_sgate_kernel<<<(a.T + wpb - 1) / wpb, kThreads, 0, s>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  err = launch_prefill_gemm(false, a, sms, s);
  if (err != cudaSuccess) return err;
  if (a.sfmt && (err = launch_prefill_gemm(false, sa, sms, s)) != cudaSuccess) return err;
  mk(4);
  // h -> f16 with a power-of-two row scale (the down GEMM's B); the fold-scales lever reads h as it is,
  // the FP8-activation lever quantises it to E4M3 blocks
  if (fp8_lever(a)) pf_hquant_fp8_kernel<<<(a.T * a.k + wpb - 1) / wpb, kThreads, 0, s>>>(a);
  else if (!fold_lever(a)) pf_hconv_kernel<<<(a.T * a.k + wpb - 1) / wpb, kThreads, 0, s>>>(a);
  if (a.sfmt && fp8_lever(sa)) pf_hquant_fp8_kernel<<<(a.T + wpb - 1) / wpb, kThreads, 0, s>>>(sa);
  else if (a.sfmt && !fold_lever(sa)) pf_hconv_kernel<<<(a.T + wpb - 1) / wpb, kThreads, 0, s>>>(sa);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  mk(5);
  if ((err = launch_prefill_gemm(true, a, sms, s)) != cudaSuccess) return err;
  if (a.sfmt && (err = launch_prefill_gemm(true, sa, sms, s)) != cudaSuccess) return err;
  mk(6);
  pf_combine_kernel<<<a.T, kThreads, 0, s>>>(a);
  mk(7);
  return cudaGetLastError();
}

}  // namespace qmoe
