// Decode-path expert projections (T <= 8 tokens).
//
//   gate/up: for every active expert e and every 16-row tile of its gate and
//            up matrices, h[p, rows] = bf16( silu(g) * u ) for the pairs p
//            routed to e (gate and up in one pass: DGPP README "Execution and
//            performance", engine.expert_gemm_pair).
//   down:    P[p, rows] = W_down_e h_p (FP32 partials, DGPP README row
//            engine.prefill_bf16_partials: fp32 partials by default); the last
//            CTA to finish a row block combines y = bf16( sum_j w_j P_j + S ).
//
// The weights stream from HBM with 128-bit non-allocating loads and are
// decoded in registers (DGPP forum post 15 "Lossless bf12": decode reads the
// weights at the memory line rate, rebuilding values in registers).  Decoded
// weights are exact in f16 (E2M1, E2M1 x E4M3, E4M3, int4, int8), and feed
// warp-level m16n8k16 MMAs with the tokens as the N=8 side, so one decode
// serves every token routed to the expert.  Activations enter as f16 scaled by
// a per-token power of two (exact for every element above 2^-32 of the
// token's largest magnitude), undone in the FP32 epilogue.
//
// Per-block scales: NVFP4's E4M3 block scale is folded into the f16 weights
// (e2m1 * e4m3 has at most 6 significant bits and stays inside f16's normal
// range); MXFP4, int4/int8 g64 and FP8 b128 scales multiply the FP32 partial
// sum of each 16-byte unit (the per-group FMA of the default chain, DGPP
// README row engine.prefill_fold_scales).
#include "kernels.cuh"

namespace qmoe {

namespace {

constexpr int kMaxT = MOE_DECODE_MAX_TOKENS;
constexpr int kWarps = kExpertThreads / 32;

// Per-format work unit.  The four lanes c = 0..3 of a row group always work
// inside one unit of kUnitK consecutive columns, lane c on its chunk of
// kChunkBytes bytes at byte offset c * kChunkBytes.  An m16n8k16 MMA reduces
// over K across those four lanes, so a unit never spans two scale blocks
// whose scale is applied after the MMA: MXFP4 units are one 32-element
// block, int4/int8 units one 64-element group, FP8 units lie inside one
// 128x128 block.  NVFP4 folds its 16-element block scales into the f16
// weights before the MMA, so its units may span several blocks.
template <int F> struct Fm;
template <> struct Fm<MOE_FMT_NVFP4> { static constexpr int kBits = 4, kChunkBytes = 16, kPrefetch = 2; };
template <> struct Fm<MOE_FMT_MXFP4> { static constexpr int kBits = 4, kChunkBytes = 4, kPrefetch = 8; };
template <> struct Fm<MOE_FMT_INT4_G64> { static constexpr int kBits = 4, kChunkBytes = 8, kPrefetch = 4; };
template <> struct Fm<MOE_FMT_INT8_G64> { static constexpr int kBits = 8, kChunkBytes = 16, kPrefetch = 2; };
template <> struct Fm<MOE_FMT_FP8_B128> { static constexpr int kBits = 8, kChunkBytes = 16, kPrefetch = 2; };
template <int F> constexpr int unit_k() { return 4 * Fm<F>::kChunkBytes * 8 / Fm<F>::kBits; }
template <int F> constexpr int chunk_k() { return Fm<F>::kChunkBytes * 8 / Fm<F>::kBits; }

// One expert matrix W[N, K] seen by a warp.
struct Mat {
  const uint8_t* data;
  const uint8_t* scales;
  int K;
};

__device__ __forceinline__ Mat mat_of(const QW& w, int fmt, int e, int N, int K) {
  Mat m;
  m.data = w.data + (size_t)e * data_bytes(fmt, N, K);
  m.scales = w.scales + (size_t)e * scale_bytes(fmt, N, K);
  m.K = K;
  return m;
}

// The raw scale bits of row R that lane chunk starting at column k needs.
template <int F>
__device__ __forceinline__ uint32_t load_scale(const Mat& m, int R, int k) {
  if constexpr (F == MOE_FMT_NVFP4) return ldg_nc_u16(m.scales + (size_t)R * (m.K / 16) + k / 16);
  else if constexpr (F == MOE_FMT_MXFP4) return ldg_nc_u8(m.scales + (size_t)R * (m.K / 32) + k / 32);
  else if constexpr (F == MOE_FMT_INT4_G64 || F == MOE_FMT_INT8_G64)
    return ldg_nc_u16(m.scales + ((size_t)R * (m.K / 64) + k / 64) * 2);
  else return ldg_nc_u32(m.scales + ((size_t)(R / 128) * (m.K / 128) + k / 128) * 4);
}

template <int F>
__device__ __forceinline__ float unit_scale(uint32_t s) {
  if constexpr (F == MOE_FMT_MXFP4) return e8m0_to_float(s);
  else if constexpr (F == MOE_FMT_INT4_G64 || F == MOE_FMT_INT8_G64) return __uint_as_float(s << 16);
  else return __uint_as_float(s);
}

template <int NM>
struct Unit {
  uint4 d[NM][2];      // this lane's chunk of rows r and r+8 (only the first kChunkBytes used)
  uint32_t s[NM][2];
};

template <int F, int NM>
__device__ __forceinline__ void load_unit(Unit<NM>& u, const Mat (&m)[NM], int R0, int kc) {
  constexpr int kB = Fm<F>::kBits, kC = Fm<F>::kChunkBytes;
#pragma unroll
  for (int i = 0; i < NM; ++i) {
    const size_t rb = (size_t)m[i].K * kB / 8;
    const uint8_t* p0 = m[i].data + (size_t)R0 * rb + (size_t)kc * kB / 8;
    if constexpr (kC == 16) {
      u.d[i][0] = ldg_nc_v4(p0);
      u.d[i][1] = ldg_nc_v4(p0 + 8 * rb);
    } else if constexpr (kC == 8) {
      const uint2 a = ldg_nc_v2(p0), b = ldg_nc_v2(p0 + 8 * rb);
      u.d[i][0] = make_uint4(a.x, a.y, 0, 0);
      u.d[i][1] = make_uint4(b.x, b.y, 0, 0);
    } else {
      u.d[i][0] = make_uint4(ldg_nc_u32(p0), 0, 0, 0);
      u.d[i][1] = make_uint4(ldg_nc_u32(p0 + 8 * rb), 0, 0, 0);
    }
    u.s[i][0] = load_scale<F>(m[i], R0, kc);
    u.s[i][1] = load_scale<F>(m[i], R0 + 8, kc);
  }
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// MMA over one unit of NM matrices; xl: this lane's activations (f16) at its
// chunk's first column.  Every lane of the warp executes every MMA.
template <int F, int NM>
__device__ __forceinline__ void compute_unit(const Unit<NM>& u, const __half* xl, float (&acc)[NM][4]) {
  if constexpr (Fm<F>::kBits == 4) {
    constexpr int kWords = Fm<F>::kChunkBytes / 4;  // 8 columns per word
    float d[NM][4];
    uint32_t s2[NM][2][2];
#pragma unroll
    for (int i = 0; i < NM; ++i) {
#pragma unroll
      for (int j = 0; j < 4; ++j) d[i][j] = 0.f;
      if constexpr (F == MOE_FMT_NVFP4) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          s2[i][r][0] = e4m3_bcast_f16x2(u.s[i][r] & 0xFF);
          s2[i][r][1] = e4m3_bcast_f16x2(u.s[i][r] >> 8);
        }
      }
    }
#pragma unroll
    for (int wd = 0; wd < kWords; ++wd) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xl + wd * 8);  // x[k .. k+8) as f16 pairs
      uint32_t bA0, bA1, bB0, bB1;
      if constexpr (F == MOE_FMT_INT4_G64) {
        bA0 = prmt(xv.x, xv.z, 0x5410u);  // (x0, x4)
        bA1 = prmt(xv.x, xv.z, 0x7632u);  // (x1, x5)
        bB0 = prmt(xv.y, xv.w, 0x5410u);  // (x2, x6)
        bB1 = prmt(xv.y, xv.w, 0x7632u);  // (x3, x7)
      } else {
        bA0 = xv.x; bA1 = xv.y; bB0 = xv.z; bB1 = xv.w;
      }
#pragma unroll
      for (int i = 0; i < NM; ++i) {
        uint32_t v0[4], v1[4];
        if constexpr (F == MOE_FMT_INT4_G64) {
          int4x8_to_f16x2_paired(word(u.d[i][0], wd), v0);
          int4x8_to_f16x2_paired(word(u.d[i][1], wd), v1);
        } else {
          e2m1x8_to_f16x2(word(u.d[i][0], wd), v0);
          e2m1x8_to_f16x2(word(u.d[i][1], wd), v1);
        }
        if constexpr (F == MOE_FMT_NVFP4) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v0[j] = hmul2_u32(v0[j], s2[i][0][wd >> 1]);
            v1[j] = hmul2_u32(v1[j], s2[i][1][wd >> 1]);
          }
        }
        const uint32_t aA[4] = {v0[0], v1[0], v0[1], v1[1]};
        const uint32_t aB[4] = {v0[2], v1[2], v0[3], v1[3]};
        if constexpr (F == MOE_FMT_NVFP4) {
          mma_f16_16816(acc[i], aA, bA0, bA1);
          mma_f16_16816(acc[i], aB, bB0, bB1);
        } else {
          mma_f16_16816(d[i], aA, bA0, bA1);
          mma_f16_16816(d[i], aB, bB0, bB1);
        }
      }
    }
    if constexpr (F != MOE_FMT_NVFP4) {
#pragma unroll
      for (int i = 0; i < NM; ++i) {
        const float sa = unit_scale<F>(u.s[i][0]), sb = unit_scale<F>(u.s[i][1]);
        acc[i][0] = __fmaf_rn(d[i][0], sa, acc[i][0]);
        acc[i][1] = __fmaf_rn(d[i][1], sa, acc[i][1]);
        acc[i][2] = __fmaf_rn(d[i][2], sb, acc[i][2]);
        acc[i][3] = __fmaf_rn(d[i][3], sb, acc[i][3]);
      }
    }
  } else {
    // 8-bit codes: a 16-byte chunk is 16 columns = four words of four codes
    float d[NM][4];
#pragma unroll
    for (int i = 0; i < NM; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) d[i][j] = 0.f;
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
      const uint2 xv = *reinterpret_cast<const uint2*>(xl + wd * 4);
#pragma unroll
      for (int i = 0; i < NM; ++i) {
        uint32_t lo0, hi0, lo1, hi1;
        if constexpr (F == MOE_FMT_INT8_G64) {
          int8x4_to_f16x2(word(u.d[i][0], wd), lo0, hi0);
          int8x4_to_f16x2(word(u.d[i][1], wd), lo1, hi1);
        } else {
          e4m3x4_to_f16x2(word(u.d[i][0], wd), lo0, hi0);
          e4m3x4_to_f16x2(word(u.d[i][1], wd), lo1, hi1);
        }
        const uint32_t a[4] = {lo0, lo1, hi0, hi1};
        mma_f16_16816(d[i], a, xv.x, xv.y);
      }
    }
#pragma unroll
    for (int i = 0; i < NM; ++i) {
      const float sa = unit_scale<F>(u.s[i][0]), sb = unit_scale<F>(u.s[i][1]);
      acc[i][0] = __fmaf_rn(d[i][0], sa, acc[i][0]);
      acc[i][1] = __fmaf_rn(d[i][1], sa, acc[i][1]);
      acc[i][2] = __fmaf_rn(d[i][2], sb, acc[i][2]);
      acc[i][3] = __fmaf_rn(d[i][3], sb, acc[i][3]);
    }
  }
}

// One warp: rows [row0, row0 + 16) of NM matrices over columns [kb, kb + Kw),
// Kw a multiple of the unit.  Lane (r = lane/4, c = lane%4) takes rows r and
// r+8 and chunk c of every unit; units stream through a register ring of
// kPrefetch entries.  The trip count is the same for every lane (mma.sync
// needs the whole warp).  xrow: this lane's token row (f16) in shared memory.
template <int F, int NM>
__device__ __forceinline__ void warp_tile(const Mat (&m)[NM], int row0, int kb, int Kw, const __half* xrow,
                                          float (&acc)[NM][4]) {
  constexpr int UK = unit_k<F>(), CK = chunk_k<F>(), PF = Fm<F>::kPrefetch;
  const int lane = threadIdx.x & 31;
  const int R0 = row0 + (lane >> 2);
  const int koff = kb + (lane & 3) * CK;
  const int nU = Kw / UK;
  Unit<NM> buf[PF];
#pragma unroll
  for (int p = 0; p < PF; ++p)
    if (p < nU) load_unit<F, NM>(buf[p], m, R0, koff + p * UK);
  for (int u0 = 0; u0 < nU; u0 += PF) {
#pragma unroll
    for (int p = 0; p < PF; ++p) {
      const int u = u0 + p;
      if (u < nU) {
        compute_unit<F, NM>(buf[p], xrow + koff + u * UK, acc);
        if (u + PF < nU) load_unit<F, NM>(buf[p], m, R0, koff + (u + PF) * UK);
      }
    }
  }
}

template <int NM>
__device__ __forceinline__ void warp_tile_any(int fmt, const Mat (&m)[NM], int row0, int kb, int Kw,
                                              const __half* xrow, float (&acc)[NM][4]) {
  switch (fmt) {
    case MOE_FMT_NVFP4: warp_tile<MOE_FMT_NVFP4, NM>(m, row0, kb, Kw, xrow, acc); break;
    case MOE_FMT_MXFP4: warp_tile<MOE_FMT_MXFP4, NM>(m, row0, kb, Kw, xrow, acc); break;
    case MOE_FMT_INT4_G64: warp_tile<MOE_FMT_INT4_G64, NM>(m, row0, kb, Kw, xrow, acc); break;
    case MOE_FMT_INT8_G64: warp_tile<MOE_FMT_INT8_G64, NM>(m, row0, kb, Kw, xrow, acc); break;
    case MOE_FMT_FP8_B128: warp_tile<MOE_FMT_FP8_B128, NM>(m, row0, kb, Kw, xrow, acc); break;
    default: break;
  }
}

// Largest-magnitude element -> power-of-two exponent p with amax * 2^-p in [2^14, 2^15).
__device__ __forceinline__ int scale_exponent(float amax) {
  if (!(amax > 0.f) || !(amax < __int_as_float(0x7F800000))) return 0;
  int e = ((__float_as_uint(amax) >> 23) & 0xFF) - 127;
  int p = e - 14;
  return max(-100, min(100, p));
}

// Stage rows (bf16, length K, source stride K) into shared memory as f16
// scaled by 2^-p per row.  Row `nrows` is zero-filled (the MMA column of an
// absent token).  Uses the whole CTA.
__device__ void stage_rows_f16(const uint16_t* const* src_rows, int nrows, int K, __half* dst, int dst_stride,
                               int* pexp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int r = warp; r < nrows; r += kWarps) {
    const uint16_t* s = src_rows[r];
    float amax = 0.f;
    for (int k = lane * 8; k < K; k += 256) {
      uint4 v = *reinterpret_cast<const uint4*>(s + k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(w[j] & 0xFFFF)), fabsf(bf16_bits_to_float(w[j] >> 16))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const int p = scale_exponent(amax);
    if (lane == 0) pexp[r] = p;
    const float inv = exp2i(-p);
    __half* d = dst + (size_t)r * dst_stride;
    for (int k = lane * 8; k < K; k += 256) {
      uint4 v = *reinterpret_cast<const uint4*>(s + k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        __half2 hh = __floats2half2_rn(bf16_bits_to_float(w[j] & 0xFFFF) * inv, bf16_bits_to_float(w[j] >> 16) * inv);
        o[j] = *reinterpret_cast<uint32_t*>(&hh);
      }
      *reinterpret_cast<uint4*>(d + k) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  __half* z = dst + (size_t)nrows * dst_stride;
  for (int k = tid * 8; k < K; k += kExpertThreads * 8) *reinterpret_cast<uint4*>(z + k) = make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// --------------------------------------------------------------- gate / up --

__global__ void __launch_bounds__(kExpertThreads, 1) gateup_decode_kernel(ExpertArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int T = a.T, H = a.H, I = a.I;
  const int WK = a.wk_gu, WR = a.wr_gu;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int xs_stride = a.xs_tok_stride;  // halfs per token row
  __half* xs = reinterpret_cast<__half*>(smem);
  float* red = reinterpret_cast<float*>(smem + (size_t)(T + 1) * xs_stride * 2);  // [kWarps][2][32][4]
  __shared__ int s_pexp[kMaxT + 1];
  __shared__ int s_col_tok[8];
  __shared__ int s_col_out[8];
  __shared__ const uint16_t* s_src[kMaxT];

  pdl_launch_dependents();
  // activations are an input of the call: stage them before waiting on the router
  if (tid < T) s_src[tid] = a.x + (size_t)tid * H;
  __syncthreads();
  stage_rows_f16(s_src, T, H, xs, xs_stride, s_pexp);
  if (tid == 0) s_pexp[T] = 0;
  pdl_wait();
  const int n_active = *reinterpret_cast<volatile int*>(&a.rb.ctrl->n_active);
  const int rows_item = 16 * WR;
  const int tiles = I / rows_item;
  const int stiles = a.sfmt ? a.Is / rows_item : 0;
  const int n_items = n_active * tiles + stiles;
  const int it0 = (int)((long long)blockIdx.x * n_items / gridDim.x);
  const int it1 = (int)((long long)(blockIdx.x + 1) * n_items / gridDim.x);
  const int wk = warp % WK, wr = warp / WK;
  const int Kw = H / WK;
  __syncthreads();

  for (int it = it0; it < it1; ++it) {
    const bool shared_item = it >= n_active * tiles;
    int e = 0, tile, ncols;
    if (!shared_item) {
      const int slot = it / tiles;
      tile = it - slot * tiles;
      e = a.rb.act[slot];
      ncols = a.rb.cnt[e];
      if (tid < 8) {
        if (tid < ncols) {
          const int p = a.rb.pair[a.rb.off[e] + tid];
          s_col_tok[tid] = p / a.k;
          s_col_out[tid] = p;
        } else {
          s_col_tok[tid] = T;
          s_col_out[tid] = -1;
        }
      }
    } else {
      tile = it - n_active * tiles;
      ncols = T;
      if (tid < 8) {
        s_col_tok[tid] = tid < T ? tid : T;
        s_col_out[tid] = tid < T ? tid : -1;
      }
    }
    __syncthreads();
    const int fmt = shared_item ? a.sfmt : a.fmt;
    const int N = shared_item ? a.Is : I;
    const QW& qg = shared_item ? a.sgate : a.gate;
    const QW& qu = shared_item ? a.sup : a.up;
    const Mat m[2] = {mat_of(qg, fmt, e, N, H), mat_of(qu, fmt, e, N, H)};
    const int row0 = tile * rows_item + wr * 16;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const __half* xrow = xs + (size_t)s_col_tok[lane >> 2] * xs_stride;
    warp_tile_any<2>(fmt, m, row0, wk * Kw, Kw, xrow, acc);
    float* rw = red + ((size_t)warp * 2 * 32 + lane) * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) { rw[j] = acc[0][j]; rw[32 * 4 + j] = acc[1][j]; }
    __syncthreads();
    if (wk == 0) {
      float g[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
      for (int w2 = 0; w2 < WK; ++w2) {  // fixed order: deterministic
        const float* rr = red + ((size_t)(wr * WK + w2) * 2 * 32 + lane) * 4;
#pragma unroll
        for (int j = 0; j < 4; ++j) { g[j] += rr[j]; u[j] += rr[32 * 4 + j]; }
      }
      const float tsg = (fmt == MOE_FMT_NVFP4) ? __ldg(qg.ts + e) : 1.f;
      const float tsu = (fmt == MOE_FMT_NVFP4) ? __ldg(qu.ts + e) : 1.f;
      const int r = lane >> 2, c = lane & 3;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = 2 * c + (j & 1);
        const int row = row0 + r + ((j & 2) ? 8 : 0);
        const int out = s_col_out[col];
        if (out >= 0) {
          const float sc = exp2i(s_pexp[s_col_tok[col]]);
          const float gv = g[j] * sc * tsg, uv = u[j] * sc * tsu;
          const uint16_t hb = float_to_bf16_bits(silu_f(gv) * uv);
          if (shared_item) a.hs[(size_t)out * a.Is + row] = hb;
          else a.h[(size_t)out * I + row] = hb;
        }
      }
    }
    __syncthreads();
  }
}

// -------------------------------------------------------- down + combine --

__global__ void __launch_bounds__(kExpertThreads, 1) down_decode_kernel(ExpertArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int T = a.T, H = a.H, I = a.I, k = a.k;
  const int WK = a.wk_dn, WR = a.wr_dn;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hs_stride = a.hs_tok_stride;
  __half* hsm = reinterpret_cast<__half*>(smem);  // [9][hs_stride]
  float* red = reinterpret_cast<float*>(smem + (size_t)(8 + 1) * hs_stride * 2);  // [kWarps][32][4]
  __shared__ int s_pexp[9];
  __shared__ int s_col_out[8];
  __shared__ const uint16_t* s_src[8];
  __shared__ int s_cur;
  __shared__ int s_last;
  __shared__ int s_ncols;

  pdl_launch_dependents();
  pdl_wait();
  const int n_active = *reinterpret_cast<volatile int*>(&a.rb.ctrl->n_active);
  const int rows_item = 16 * WR;
  const int tiles = H / rows_item;
  const int n_items = n_active * tiles + (a.sfmt ? tiles : 0);
  const int needed = n_active + (a.sfmt ? 1 : 0);
  const int it0 = (int)((long long)blockIdx.x * n_items / gridDim.x);
  const int it1 = (int)((long long)(blockIdx.x + 1) * n_items / gridDim.x);
  const int wk = warp % WK, wr = warp / WK;
  if (tid == 0) s_cur = -2;
  __syncthreads();

  for (int it = it0; it < it1; ++it) {
    const bool shared_item = it >= n_active * tiles;
    int e = 0, tile, who;
    if (!shared_item) {
      const int slot = it / tiles;
      tile = it - slot * tiles;
      e = a.rb.act[slot];
      who = e;
    } else {
      tile = it - n_active * tiles;
      who = -1;
    }
    const int K = shared_item ? a.Is : I;
    if (who != s_cur) {  // stage the hidden activations of this expert's pairs
      __syncthreads();
      int ncols;
      if (!shared_item) {
        ncols = a.rb.cnt[e];
        if (tid < 8) {
          if (tid < ncols) {
            const int p = a.rb.pair[a.rb.off[e] + tid];
            s_src[tid] = a.h + (size_t)p * I;
            s_col_out[tid] = p;
          } else {
            s_col_out[tid] = -1;
          }
        }
      } else {
        ncols = T;
        if (tid < 8) {
          if (tid < T) s_src[tid] = a.hs + (size_t)tid * a.Is;
          s_col_out[tid] = tid < T ? tid : -1;
        }
      }
      __syncthreads();
      stage_rows_f16(s_src, ncols, K, hsm, hs_stride, s_pexp);  // row ncols is the zero row
      if (tid == 0) { s_cur = who; s_ncols = ncols; }
      __syncthreads();
    }
    const int fmt = shared_item ? a.sfmt : a.fmt;
    const QW& qd = shared_item ? a.sdown : a.down;
    const Mat m[1] = {mat_of(qd, fmt, e, H, K)};
    const int row0 = tile * rows_item + wr * 16;
    float acc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
    const int col_b = lane >> 2;
    const __half* xrow = hsm + (size_t)(s_col_out[col_b] >= 0 ? col_b : s_ncols) * hs_stride;
    const int Kw = K / WK;
    warp_tile_any<1>(fmt, m, row0, wk * Kw, Kw, xrow, acc);
    float* rw = red + ((size_t)warp * 32 + lane) * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) rw[j] = acc[0][j];
    __syncthreads();
    if (wk == 0) {
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      for (int w2 = 0; w2 < WK; ++w2) {
        const float* rr = red + ((size_t)(wr * WK + w2) * 32 + lane) * 4;
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] += rr[j];
      }
      const float ts = (fmt == MOE_FMT_NVFP4) ? __ldg(qd.ts + e) : 1.f;
      const int r = lane >> 2, c = lane & 3;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = 2 * c + (j & 1);
        const int row = row0 + r + ((j & 2) ? 8 : 0);
        const int out = s_col_out[col];
        if (out >= 0) {
          const float val = v[j] * exp2i(s_pexp[col]) * ts;
          if (shared_item) a.S[(size_t)out * H + row] = val;
          else a.P[(size_t)out * H + row] = val;
        }
      }
    }
    // completion of this row block by this expert; the last of the `needed`
    // contributions combines the block (no floating-point atomics)
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const uint32_t prev = atomicAdd(&a.rb_cnt[tile], 1u);
      s_last = (prev == (uint32_t)needed - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      const int r0 = tile * rows_item;
      for (int q = tid; q < T * rows_item; q += kExpertThreads) {
        const int t = q / rows_item, row = r0 + (q - t * rows_item);
        float y = 0.f;
        for (int j = 0; j < k; ++j)
          y = __fmaf_rn(__ldcg(a.rb.topk_w + t * k + j), __ldcg(a.P + (size_t)(t * k + j) * H + row), y);
        if (a.sfmt) y = __fadd_rn(y, __ldcg(a.S + (size_t)t * H + row));
        a.y[(size_t)t * H + row] = float_to_bf16_bits(y);
      }
      if (tid == 0) a.rb_cnt[tile] = 0;
    }
  }
}

cudaError_t launch_pdl(void (*kern)(ExpertArgs), const ExpertArgs& a, int grid, size_t smem, cudaStream_t s) {
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kExpertThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

cudaError_t launch_gateup_decode(const ExpertArgs& a, int grid, size_t smem, cudaStream_t s) {
  return launch_pdl(gateup_decode_kernel, a, grid, smem, s);
}

cudaError_t launch_down_decode(const ExpertArgs& a, int grid, size_t smem, cudaStream_t s) {
  return launch_pdl(down_decode_kernel, a, grid, smem, s);
}

}  // namespace qmoe
