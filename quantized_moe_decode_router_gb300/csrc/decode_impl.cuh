// Decode-path expert projections (T <= 8 tokens), templated on the routed
// and shared expert formats.  Included by one translation unit per routed
// format (decode_<fmt>.cu).
//
//   gate/up: h[p, rows] = bf16( silu(g) * u ) for every pair p routed to an
//            expert, gate and up in one pass (DGPP README "Execution and
//            performance", engine.expert_gemm_pair).
//   down:    P[p, rows] = W_down_e h_p (FP32 partials, DGPP README row
//            engine.prefill_bf16_partials), S for the shared expert.
//   combine: y = bf16( sum_j w_j P_j + S ) in j order, chained after down.
//
// Work is split into independent warp tasks (expert, 16-row tile, K slice)
// so that every warp streams its own weights without CTA barriers; K slices
// of one tile are summed by the last slice to finish, in slice order
// (deterministic, no floating-point atomics).  Weights stream from HBM in
// 16-byte cp.async copies (L2 only) through a warp-private shared-memory ring
// and are decoded in registers (DGPP forum post
// 15 "Lossless bf12": decode reads weights at the memory line rate,
// rebuilding them in registers) into f16 MMA fragments; the tokens are the
// N=8 side of m16n8k16, so one decode serves every token of the expert.
//
// Lane layout: lane (r = lane/4, c = lane%4) holds rows r and r+8 of the
// tile and the 16-byte chunk c of every unit (4-bit formats: 128 columns per
// unit, 32 per lane; 8-bit formats: 64 and 16).  An MMA reduces K across the
// four lanes of a row group, so scales that differ between those lanes are
// folded into the f16 weights before the MMA:
//   NVFP4   e2m1 * e4m3 (at most 6 significant bits, f16-normal): exact.
//   MXFP4   e2m1 * 2^(c - cmax), cmax the largest scale code of the four
//           lanes; 2^(cmax-127) multiplies the FP32 partial.  Exact while
//           c - cmax >= -20; otherwise the unit takes a 4-MMA path that
//           applies each lane's scale in FP32.
//   INT4    q * M * 2^(e - emax) with the BF16 scale s = M * 2^e (M an 8-bit
//           integer): |q * M| <= 2040 fits f16's 11-bit significand; exact
//           while e - emax >= -24, else the 4-MMA path.
//   INT8, FP8: one scale per unit for all four lanes, applied to the FP32
//           partial of the unit (the per-group FMA of the default chain,
//           DGPP README row engine.prefill_fold_scales).
// Activations enter as f16 scaled by a per-token (per-pair for h) power of
// two, exact for every element above 2^-32 of the row's largest magnitude.
#pragma once

#include "kernels.cuh"

namespace qmoe {
namespace dec {

constexpr int kMaxT = MOE_DECODE_MAX_TOKENS;
constexpr int kWarps = kExpertThreads / 32;

template <int F> struct Fm;
template <> struct Fm<MOE_FMT_NVFP4> { static constexpr int kBits = 4; };
template <> struct Fm<MOE_FMT_MXFP4> { static constexpr int kBits = 4; };
template <> struct Fm<MOE_FMT_INT4_G64> { static constexpr int kBits = 4; };
template <> struct Fm<MOE_FMT_INT8_G64> { static constexpr int kBits = 8; };
template <> struct Fm<MOE_FMT_FP8_B128> { static constexpr int kBits = 8; };
template <> struct Fm<MOE_FMT_INT4_G128> { static constexpr int kBits = 4; };
template <int F> constexpr int unit_k() { return Fm<F>::kBits == 4 ? 128 : 64; }
__device__ __forceinline__ int Fm_bits(int fmt) {
  return (fmt == MOE_FMT_INT8_G64 || fmt == MOE_FMT_FP8_B128) ? 8 : 4;
}
template <int F> constexpr int chunk_k() { return unit_k<F>() / 4; }

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

// Byte offset of the scale bits for column k inside one row's scales.
template <int F>
__device__ __forceinline__ uint32_t scale_col(int k) {
  if constexpr (F == MOE_FMT_NVFP4) return (uint32_t)k / 16;
  else if constexpr (F == MOE_FMT_MXFP4) return (uint32_t)k / 32;
  else if constexpr (F == MOE_FMT_INT4_G64 || F == MOE_FMT_INT8_G64) return (uint32_t)k / 64 * 2;
  else if constexpr (F == MOE_FMT_INT4_G128) return (uint32_t)k / 128 * 2;
  else return (uint32_t)k / 128 * 4;
}

// Start of row R's scales (FP8: of its 128-row block).
template <int F>
__device__ __forceinline__ const uint8_t* scale_row(const Mat& m, int R) {
  if constexpr (F == MOE_FMT_NVFP4) return m.scales + (size_t)R * (m.K / 16);
  else if constexpr (F == MOE_FMT_MXFP4) return m.scales + (size_t)R * (m.K / 32);
  else if constexpr (F == MOE_FMT_INT4_G64 || F == MOE_FMT_INT8_G64) return m.scales + (size_t)R * (m.K / 64) * 2;
  else if constexpr (F == MOE_FMT_INT4_G128) return m.scales + (size_t)R * (m.K / 128) * 2;
  else return m.scales + (size_t)(R / 128) * (m.K / 128) * 4;
}

// The scale bits inside the aligned 32-bit word that holds them (byte offset lo2 = address & 3).
template <int F>
__device__ __forceinline__ uint32_t scale_bits(uint32_t w, uint32_t lo2) {
  if constexpr (F == MOE_FMT_MXFP4) return (w >> (8 * lo2)) & 0xFFu;
  else if constexpr (F == MOE_FMT_FP8_B128) return w;
  else return (w >> (8 * lo2)) & 0xFFFFu;
}

// Per-task view of a warp's rows: data pointers at the lane's first chunk and
// scale-row pointers; units advance the data by 64 bytes.
template <int NM>
struct Stream {
  const uint8_t* d[NM][2];
  const uint8_t* s[NM][2];
};

template <int F, int NM>
__device__ __forceinline__ Stream<NM> make_stream(const Mat (&m)[NM], int R0, int koff) {
  constexpr int kB = Fm<F>::kBits;
  Stream<NM> st;
#pragma unroll
  for (int i = 0; i < NM; ++i) {
    const size_t rb = (size_t)m[i].K * kB / 8;
    const uint8_t* p0 = m[i].data + (size_t)R0 * rb + (size_t)koff * kB / 8;
    st.d[i][0] = p0;
    st.d[i][1] = p0 + 8 * rb;
    st.s[i][0] = scale_row<F>(m[i], R0);
    st.s[i][1] = scale_row<F>(m[i], R0 + 8);
  }
  return st;
}

template <int NM>
struct Unit {
  uint4 d[NM][2];  // rows r and r+8
  uint32_t s[NM][2];
};

// Warp-private shared-memory ring: one stage holds a unit of every lane,
// data [NM][2 rows][32 lanes] x 16 B followed by scale words [NM][2][32] x 4 B.
template <int NM>
constexpr int stage_bytes() { return dec_stage_bytes(NM); }

template <int F, int NM>
__device__ __forceinline__ void issue_unit(uint8_t* stage, const Stream<NM>& st, int u, int kc) {
  const int lane = threadIdx.x & 31;
  const uint32_t sc = scale_col<F>(kc);
#pragma unroll
  for (int i = 0; i < NM; ++i)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      cp_async16(stage + ((i * 2 + r) * 32 + lane) * 16, st.d[i][r] + (size_t)u * 64);
      const uintptr_t sp = reinterpret_cast<uintptr_t>(st.s[i][r]) + sc;
      cp_async4(stage + NM * 2 * 32 * 16 + ((i * 2 + r) * 32 + lane) * 4,
                reinterpret_cast<const void*>(sp & ~(uintptr_t)3));
    }
}

// Bit offset of the lane's scale bits inside their aligned 32-bit word.  For
// 4-bit codes a unit advances the scale column by a multiple of 4 bytes (and
// slices and row steps keep that alignment), so the offset of the first unit
// (column koff) holds for every unit of the stream.
template <int F, int NM>
__device__ __forceinline__ void scale_shifts(const Stream<NM>& st, int koff, uint32_t (&sh)[NM][2]) {
#pragma unroll
  for (int i = 0; i < NM; ++i)
#pragma unroll
    for (int r = 0; r < 2; ++r)
      sh[i][r] = 8u * (((uint32_t)reinterpret_cast<uintptr_t>(st.s[i][r]) + scale_col<F>(koff)) & 3u);
}

template <int F, int NM>
__device__ __forceinline__ void read_unit(Unit<NM>& u, const uint8_t* stage, const Stream<NM>& st, int kc,
                                          const uint32_t (&sh)[NM][2]) {
  const int lane = threadIdx.x & 31;
  const uint32_t sc = scale_col<F>(kc);
#pragma unroll
  for (int i = 0; i < NM; ++i)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      u.d[i][r] = *reinterpret_cast<const uint4*>(stage + ((i * 2 + r) * 32 + lane) * 16);
      const uint32_t w = *reinterpret_cast<const uint32_t*>(stage + NM * 2 * 32 * 16 + ((i * 2 + r) * 32 + lane) * 4);
      if constexpr (Fm<F>::kBits == 4 && F != MOE_FMT_INT4_G128) {
        u.s[i][r] = (w >> sh[i][r]) & (F == MOE_FMT_MXFP4 ? 0xFFu : 0xFFFFu);
      } else {
        const uint32_t lo2 = ((uint32_t)reinterpret_cast<uintptr_t>(st.s[i][r]) + sc) & 3u;
        u.s[i][r] = scale_bits<F>(w, lo2);
      }
    }
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ int max4(int v) {
  v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
  return max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
}

__device__ __forceinline__ uint32_t f16x2_bcast(float v) {
  __half2 h = __float2half2_rn(v);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Decoded (unscaled) f16 fragments of one 32-bit word of row r / r+8.
template <int F>
__device__ __forceinline__ void decode_word4(uint32_t w, uint32_t (&v)[4]) {
  if constexpr (F == MOE_FMT_INT4_G64) int4x8_to_f16x2_paired(w, v);
  else if constexpr (F == MOE_FMT_INT4_G128) int4x8_to_f16x2_paired(w ^ 0x88888888u, v);  // u - 8: flip the top bit
  else e2m1x8_to_f16x2(w, v);
}

// Per-lane scale folding of a 4-bit unit.  fac[i][r][b]: f16x2 factor for
// row r (0 -> r, 1 -> r+8) and 16-element half b of the lane's chunk;
// us[i][r]: FP32 unit scale applied after the MMA.  Returns false if the
// fold would not be exact for some lane of the warp (-> 4-MMA path).
template <int F, int NM>
__device__ __forceinline__ bool fold4(const Unit<NM>& u, uint32_t (&fac)[NM][2][2], float (&us)[NM][2]) {
  bool ok = true;
#pragma unroll
  for (int i = 0; i < NM; ++i) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint32_t s = u.s[i][r];
      if constexpr (F == MOE_FMT_NVFP4) {
        // both E4M3 scales in one conversion (byte 0 -> low half), each half then broadcast
        const uint32_t f2 = e4m3x2_to_f16x2(s & 0xFFFFu);
        fac[i][r][0] = prmt(f2, f2, 0x1010u);
        fac[i][r][1] = prmt(f2, f2, 0x3232u);
        us[i][r] = 1.f;
      } else if constexpr (F == MOE_FMT_MXFP4) {
        const int c = (int)(s & 0xFF);
        const int cm = max4(c);
        const int d = c - cm;
        ok = ok && d >= -20 && cm != 255;
        fac[i][r][0] = fac[i][r][1] = f16x2_bcast(exp2i(max(d, -20)));
        us[i][r] = e8m0_to_float((uint32_t)cm);
      } else {  // INT4_G64: bf16 scale = M * 2^e, M the integer significand
        const uint32_t E8 = (s >> 7) & 0xFF;
        const int M = (int)((s & 0x7F) | (E8 ? 0x80u : 0u));
        const int e = (E8 ? (int)E8 : 1) - 134;
        const int ev = M ? e : -100000;
        const int em = max4(ev);
        const int d = e - em;
        ok = ok && E8 != 255 && (M == 0 || d >= -24);
        const float f = (float)M * exp2i(max(d, -24));  // exact: an 8-bit integer times a power of two
        fac[i][r][0] = fac[i][r][1] = f16x2_bcast((s & 0x8000) ? -f : f);
        us[i][r] = ldexpf(1.0f, em < -1000 ? 0 : em);
      }
    }
  }
  return __all_sync(0xFFFFFFFFu, ok);
}

template <int F>
__device__ __forceinline__ float unscaled_scale(uint32_t s) {
  if constexpr (F == MOE_FMT_MXFP4) return e8m0_to_float(s & 0xFF);
  else if constexpr (F == MOE_FMT_INT4_G128) return __half2float(__ushort_as_half((unsigned short)s));
  else if constexpr (F == MOE_FMT_INT4_G64 || F == MOE_FMT_INT8_G64) return __uint_as_float(s << 16);
  else return __uint_as_float(s);
}

// B fragments (activations) of word wd of the lane's chunk.
template <int F>
__device__ __forceinline__ void b_frags(const uint4& xv, uint32_t& a0, uint32_t& a1, uint32_t& b0, uint32_t& b1) {
  if constexpr (F == MOE_FMT_INT4_G64 || F == MOE_FMT_INT4_G128) {
    a0 = prmt(xv.x, xv.z, 0x5410u);  // (x0, x4)
    a1 = prmt(xv.x, xv.z, 0x7632u);  // (x1, x5)
    b0 = prmt(xv.y, xv.w, 0x5410u);  // (x2, x6)
    b1 = prmt(xv.y, xv.w, 0x7632u);  // (x3, x7)
  } else {
    a0 = xv.x; a1 = xv.y; b0 = xv.z; b1 = xv.w;
  }
}

// One unit of NM matrices: MMA into acc (even words of the lane's chunk) and
// acc2 (odd words): two independent accumulation chains, so consecutive MMAs
// of a matrix do not wait for each other.  xl: this lane's activations (f16)
// at its chunk's first column.  Every lane executes every MMA.
template <int F, int NM>
__device__ __forceinline__ void compute_unit(const Unit<NM>& u, const __half* xl, float (&acc)[NM][4],
                                             float (&acc2)[NM][4]) {
  if constexpr (F == MOE_FMT_INT4_G128) {
    // one FP16 scale per row covers the whole 128-column unit for all four lanes: the integer codes
    // go through the MMA unscaled (exact in f16) and the scale multiplies the FP32 partial
    float d[NM][4], d2[NM][4];
#pragma unroll
    for (int i = 0; i < NM; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) { d[i][j] = 0.f; d2[i][j] = 0.f; }
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xl + wd * 8);
      uint32_t bA0, bA1, bB0, bB1;
      b_frags<F>(xv, bA0, bA1, bB0, bB1);
#pragma unroll
      for (int i = 0; i < NM; ++i) {
        uint32_t v0[4], v1[4];
        decode_word4<F>(word(u.d[i][0], wd), v0);
        decode_word4<F>(word(u.d[i][1], wd), v1);
        const uint32_t aA[4] = {v0[0], v1[0], v0[1], v1[1]};
        const uint32_t aB[4] = {v0[2], v1[2], v0[3], v1[3]};
        float (&dst)[4] = (wd & 1) ? d2[i] : d[i];
        mma_f16_16816(dst, aA, bA0, bA1);
        mma_f16_16816(dst, aB, bB0, bB1);
      }
    }
#pragma unroll
    for (int i = 0; i < NM; ++i) {
      const float sa = unscaled_scale<F>(u.s[i][0]), sb = unscaled_scale<F>(u.s[i][1]);
      acc[i][0] = __fmaf_rn(d[i][0], sa, acc[i][0]);
      acc[i][1] = __fmaf_rn(d[i][1], sa, acc[i][1]);
      acc[i][2] = __fmaf_rn(d[i][2], sb, acc[i][2]);
      acc[i][3] = __fmaf_rn(d[i][3], sb, acc[i][3]);
      acc2[i][0] = __fmaf_rn(d2[i][0], sa, acc2[i][0]);
      acc2[i][1] = __fmaf_rn(d2[i][1], sa, acc2[i][1]);
      acc2[i][2] = __fmaf_rn(d2[i][2], sb, acc2[i][2]);
      acc2[i][3] = __fmaf_rn(d2[i][3], sb, acc2[i][3]);
    }
  } else if constexpr (Fm<F>::kBits == 4) {
    uint32_t fac[NM][2][2];
    float us[NM][2];
    const bool fast = fold4<F, NM>(u, fac, us);
    if (fast) {
      float d[NM][4], d2[NM][4];
#pragma unroll
      for (int i = 0; i < NM; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) { d[i][j] = 0.f; d2[i][j] = 0.f; }
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xl + wd * 8);
        uint32_t bA0, bA1, bB0, bB1;
        b_frags<F>(xv, bA0, bA1, bB0, bB1);
#pragma unroll
        for (int i = 0; i < NM; ++i) {
          uint32_t v0[4], v1[4];
          decode_word4<F>(word(u.d[i][0], wd), v0);
          decode_word4<F>(word(u.d[i][1], wd), v1);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v0[j] = hmul2_u32(v0[j], fac[i][0][wd >> 1]);
            v1[j] = hmul2_u32(v1[j], fac[i][1][wd >> 1]);
          }
          const uint32_t aA[4] = {v0[0], v1[0], v0[1], v1[1]};
          const uint32_t aB[4] = {v0[2], v1[2], v0[3], v1[3]};
          float (&dst)[4] = (F == MOE_FMT_NVFP4) ? ((wd & 1) ? acc2[i] : acc[i]) : ((wd & 1) ? d2[i] : d[i]);
          mma_f16_16816(dst, aA, bA0, bA1);
          mma_f16_16816(dst, aB, bB0, bB1);
        }
      }
      if constexpr (F != MOE_FMT_NVFP4) {
#pragma unroll
        for (int i = 0; i < NM; ++i) {
          acc[i][0] = __fmaf_rn(d[i][0], us[i][0], acc[i][0]);
          acc[i][1] = __fmaf_rn(d[i][1], us[i][0], acc[i][1]);
          acc[i][2] = __fmaf_rn(d[i][2], us[i][1], acc[i][2]);
          acc[i][3] = __fmaf_rn(d[i][3], us[i][1], acc[i][3]);
          acc2[i][0] = __fmaf_rn(d2[i][0], us[i][0], acc2[i][0]);
          acc2[i][1] = __fmaf_rn(d2[i][1], us[i][0], acc2[i][1]);
          acc2[i][2] = __fmaf_rn(d2[i][2], us[i][1], acc2[i][2]);
          acc2[i][3] = __fmaf_rn(d2[i][3], us[i][1], acc2[i][3]);
        }
      }
    } else if constexpr (F != MOE_FMT_NVFP4) {
      // exact slow path: one MMA pass per lane column c', applying that lane's scale in FP32
      const int lane = threadIdx.x & 31, c = lane & 3;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        float d[NM][4];
#pragma unroll
        for (int i = 0; i < NM; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) d[i][j] = 0.f;
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xl + wd * 8);
          uint32_t bA0, bA1, bB0, bB1;
          b_frags<F>(xv, bA0, bA1, bB0, bB1);
#pragma unroll
          for (int i = 0; i < NM; ++i) {
            uint32_t v0[4], v1[4];
            decode_word4<F>(c == cc ? word(u.d[i][0], wd) : 0u, v0);
            decode_word4<F>(c == cc ? word(u.d[i][1], wd) : 0u, v1);
            const uint32_t aA[4] = {v0[0], v1[0], v0[1], v1[1]};
            const uint32_t aB[4] = {v0[2], v1[2], v0[3], v1[3]};
            mma_f16_16816(d[i], aA, bA0, bA1);
            mma_f16_16816(d[i], aB, bB0, bB1);
          }
        }
        const int src = (lane & ~3) | cc;
#pragma unroll
        for (int i = 0; i < NM; ++i) {
          const float sa = unscaled_scale<F>(__shfl_sync(0xFFFFFFFFu, u.s[i][0], src));
          const float sb = unscaled_scale<F>(__shfl_sync(0xFFFFFFFFu, u.s[i][1], src));
          acc[i][0] = __fmaf_rn(d[i][0], sa, acc[i][0]);
          acc[i][1] = __fmaf_rn(d[i][1], sa, acc[i][1]);
          acc[i][2] = __fmaf_rn(d[i][2], sb, acc[i][2]);
          acc[i][3] = __fmaf_rn(d[i][3], sb, acc[i][3]);
        }
      }
    }
  } else {
    // 8-bit codes: the four lanes' chunks are one scale block; four words of four codes
    float d[NM][4], d2[NM][4];
#pragma unroll
    for (int i = 0; i < NM; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) { d[i][j] = 0.f; d2[i][j] = 0.f; }
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
        mma_f16_16816((wd & 1) ? d2[i] : d[i], a, xv.x, xv.y);
      }
    }
#pragma unroll
    for (int i = 0; i < NM; ++i) {
      const float sa = unscaled_scale<F>(u.s[i][0]), sb = unscaled_scale<F>(u.s[i][1]);
      acc[i][0] = __fmaf_rn(d[i][0], sa, acc[i][0]);
      acc[i][1] = __fmaf_rn(d[i][1], sa, acc[i][1]);
      acc[i][2] = __fmaf_rn(d[i][2], sb, acc[i][2]);
      acc[i][3] = __fmaf_rn(d[i][3], sb, acc[i][3]);
      acc2[i][0] = __fmaf_rn(d2[i][0], sa, acc2[i][0]);
      acc2[i][1] = __fmaf_rn(d2[i][1], sa, acc2[i][1]);
      acc2[i][2] = __fmaf_rn(d2[i][2], sb, acc2[i][2]);
      acc2[i][3] = __fmaf_rn(d2[i][3], sb, acc2[i][3]);
    }
  }
}

// One warp: rows [row0, row0 + 16) of NM matrices over columns [kb, kb + Kw)
// (Kw a multiple of the block).  Units stream from HBM into the warp's
// private shared-memory ring of PF stages with cp.async (PF - 1 units in
// flight while one is decoded), so the bytes in flight do not cost
// registers.  Each lane copies and reads back only its own chunk, so the
// per-thread cp.async groups are the only synchronisation needed.  The trip
// count is warp-uniform (mma.sync needs the whole warp).  The K range is
// summed as blocks of `bu` units, each block from zero; block sums are either
// added to acc in block order (bpart == nullptr) or stored to bpart[b] for
// the tile's last slice to add in the same order, so the association of the
// sum depends only on K, never on how K is split between warps.
template <int F, int NM, int PF>
__device__ __forceinline__ void warp_tile(const Mat (&m)[NM], int row0, int kb, int Kw, int bu, const __half* xrow,
                                          float (&acc)[NM][4], float* bpart, uint8_t* ring) {
  constexpr int UK = unit_k<F>(), CK = chunk_k<F>(), SB = stage_bytes<NM>();
  const int lane = threadIdx.x & 31;
  const int R0 = row0 + (lane >> 2);
  const int koff = kb + (lane & 3) * CK;
  const int nU = Kw / UK;
  float blk[NM][4], blk2[NM][4];
#pragma unroll
  for (int i = 0; i < NM; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) { blk[i][j] = 0.f; blk2[i][j] = 0.f; }
  const Stream<NM> st = make_stream<F, NM>(m, R0, koff);
  uint32_t sh[NM][2];
  scale_shifts<F, NM>(st, koff, sh);
#pragma unroll
  for (int p = 0; p < PF - 1; ++p) {
    if (p < nU) issue_unit<F, NM>(ring + p * SB, st, p, koff + p * UK);
    cp_async_commit();
  }
  int slot_issue = PF - 1, slot_read = 0;
  for (int u = 0; u < nU; ++u) {
    const int un = u + PF - 1;
    if (un < nU) issue_unit<F, NM>(ring + slot_issue * SB, st, un, koff + un * UK);
    cp_async_commit();
    cp_async_wait<PF - 1>();  // unit u has landed
    Unit<NM> cur;
    read_unit<F, NM>(cur, ring + slot_read * SB, st, koff + u * UK, sh);
    slot_issue = (slot_issue + 1 == PF) ? 0 : slot_issue + 1;
    slot_read = (slot_read + 1 == PF) ? 0 : slot_read + 1;
    compute_unit<F, NM>(cur, xrow + koff + u * UK, blk, blk2);
    if (bu == 1 || (u & 1)) {  // block complete (bu is 1 or 2): its sum is blk + blk2
      if (bpart) {
        float* d = bpart + (size_t)(bu == 1 ? u : u >> 1) * (32 * 4 * NM) + lane * 4 * NM;
#pragma unroll
        for (int i = 0; i < NM; ++i)
          *reinterpret_cast<float4*>(d + 4 * i) = make_float4(blk[i][0] + blk2[i][0], blk[i][1] + blk2[i][1],
                                                              blk[i][2] + blk2[i][2], blk[i][3] + blk2[i][3]);
      } else {
#pragma unroll
        for (int i = 0; i < NM; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] += blk[i][j] + blk2[i][j];
      }
#pragma unroll
      for (int i = 0; i < NM; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) { blk[i][j] = 0.f; blk2[i][j] = 0.f; }
    }
  }
  cp_async_wait<0>();
}

// ntile tiles of one matrix set, rows row0 + t * row_step (t < ntile), each
// over the whole K range [0, Kw) with no split: one continuous cp.async
// stream, so the next tile's first units are in flight while this tile
// finishes.  Every block is summed from zero and added in block order, as in
// warp_tile; epi(t, acc) runs when tile t is complete.
template <int F, int NM, int PF, class Epi>
__device__ __forceinline__ void warp_tiles(const Mat (&m)[NM], int row0, int row_step, int ntile, int Kw, int bu,
                                           const __half* xrow, uint8_t* ring, Epi epi) {
  constexpr int UK = unit_k<F>(), CK = chunk_k<F>(), SB = stage_bytes<NM>();
  const int lane = threadIdx.x & 31;
  const int R = lane >> 2;
  const int koff = (lane & 3) * CK;
  const int nU = Kw / UK;
  const int total = ntile * nU;
  float blk[NM][4], blk2[NM][4], acc[NM][4];
#pragma unroll
  for (int i = 0; i < NM; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) { blk[i][j] = 0.f; blk2[i][j] = 0.f; acc[i][j] = 0.f; }
  // the streams of tile t are those of tile 0 moved by t row steps (every
  // format's code and scale addresses are linear in the row step used here)
  const Stream<NM> st0 = make_stream<F, NM>(m, row0 + R, koff);
  const Stream<NM> st1 = make_stream<F, NM>(m, row0 + row_step + R, koff);
  uint32_t sh[NM][2];  // the same for every tile: a row step moves the scales by a multiple of 4 bytes
  scale_shifts<F, NM>(st0, koff, sh);
  auto stream_of = [&](int t) {
    Stream<NM> st;
#pragma unroll
    for (int i = 0; i < NM; ++i)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        st.d[i][r] = st0.d[i][r] + (ptrdiff_t)t * (st1.d[i][r] - st0.d[i][r]);
        st.s[i][r] = st0.s[i][r] + (ptrdiff_t)t * (st1.s[i][r] - st0.s[i][r]);
      }
    return st;
  };
  // (tile, unit) of the next unit to issue, kept as running counters
  int ti = 0, ui = 0;
  auto issue_next = [&](int slot) {
    issue_unit<F, NM>(ring + slot * SB, stream_of(ti), ui, koff + ui * UK);
    if (++ui == nU) { ui = 0; ++ti; }
  };
#pragma unroll
  for (int p = 0; p < PF - 1; ++p) {
    if (p < total) issue_next(p);
    cp_async_commit();
  }
  int slot_issue = PF - 1, slot_read = 0;
  int t = 0, u = 0;  // the unit read in this iteration
  for (int g = 0; g < total; ++g) {
    if (g + PF - 1 < total) issue_next(slot_issue);
    cp_async_commit();
    cp_async_wait<PF - 1>();  // unit g has landed
    Unit<NM> cur;
    read_unit<F, NM>(cur, ring + slot_read * SB, stream_of(t), koff + u * UK, sh);
    slot_issue = (slot_issue + 1 == PF) ? 0 : slot_issue + 1;
    slot_read = (slot_read + 1 == PF) ? 0 : slot_read + 1;
    compute_unit<F, NM>(cur, xrow + koff + u * UK, blk, blk2);
    if (bu == 1 || (u & 1)) {  // block complete (bu is 1 or 2): its sum is blk + blk2
#pragma unroll
      for (int i = 0; i < NM; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) { acc[i][j] += blk[i][j] + blk2[i][j]; blk[i][j] = 0.f; blk2[i][j] = 0.f; }
    }
    if (u == nU - 1) {
      epi(t, acc);
#pragma unroll
      for (int i = 0; i < NM; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
      u = 0;
      ++t;
    } else {
      ++u;
    }
  }
  cp_async_wait<0>();
}

// Largest-magnitude element -> exponent p with amax * 2^-p in [2^14, 2^15).
__device__ __forceinline__ int scale_exponent_bits(uint32_t amax_bits) {
  amax_bits &= 0x7FFFFFFFu;
  if (amax_bits == 0 || amax_bits >= 0x7F800000u) return 0;
  int e = (int)(amax_bits >> 23) - 127;
  return max(-100, min(100, e - 14));
}

// Stage bf16 rows into shared memory as f16 scaled by 2^-p (p from the row's
// amax, computed here when amax_bits is null).  Row `nrows` is zero-filled.
// Loads are issued in batches of eight per lane so a row costs about one
// memory round trip per 2048 elements.
static __device__ void stage_rows_f16(const uint16_t* const* src, const uint32_t* amax_bits, int nrows, int K,
                                      __half* dst, int stride, int* pexp) {
  constexpr int kBatch = 8;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int r = warp; r < nrows; r += kWarps) {
    const uint16_t* s = src[r];
    uint32_t am;
    if (amax_bits) {
      am = amax_bits[r];
    } else {
      float amax = 0.f;
      for (int k0 = 0; k0 < K; k0 += kBatch * 256) {
        uint4 v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int k = k0 + j * 256 + lane * 8;
          v[j] = (k < K) ? *reinterpret_cast<const uint4*>(s + k) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(w[q] & 0xFFFF)), fabsf(bf16_bits_to_float(w[q] >> 16))));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      am = __float_as_uint(amax);
    }
    const int p = scale_exponent_bits(am);
    if (lane == 0) pexp[r] = p;
    const float inv = exp2i(-p);
    __half* d = dst + (size_t)r * stride;
    for (int k0 = 0; k0 < K; k0 += kBatch * 256) {
      uint4 v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int k = k0 + j * 256 + lane * 8;
        v[j] = (k < K) ? *reinterpret_cast<const uint4*>(s + k) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int k = k0 + j * 256 + lane * 8;
        if (k < K) {
          const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            __half2 hh = __floats2half2_rn(bf16_bits_to_float(w[q] & 0xFFFF) * inv,
                                           bf16_bits_to_float(w[q] >> 16) * inv);
            o[q] = *reinterpret_cast<uint32_t*>(&hh);
          }
          *reinterpret_cast<uint4*>(d + k) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }
  __half* z = dst + (size_t)nrows * stride;
  for (int k = tid * 8; k < K; k += kExpertThreads * 8) *reinterpret_cast<uint4*>(z + k) = make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Tiles split into S > 1 slices: every slice has stored its block sums
// (tile_part[b], b < nblk); the slice that arrives last adds all of them in
// block order and returns true with the sum in acc.  S == 1: acc already
// holds the sum, return true.
template <int NM>
__device__ __forceinline__ bool block_reduce(float (&acc)[NM][4], const float* tile_part, uint32_t* cnt, int S,
                                             int nblk) {
  const int lane = threadIdx.x & 31;
  if (S == 1) return true;
  __threadfence();
  __syncwarp();
  uint32_t prev = 0;
  if (lane == 0) prev = atomicAdd(cnt, 1u);
  prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
  if (prev != (uint32_t)S - 1) return false;
  __threadfence();
#pragma unroll
  for (int i = 0; i < NM; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int bl = 0; bl < nblk; ++bl) {
    const float* p = tile_part + (size_t)bl * (32 * 4 * NM) + lane * 4 * NM;
#pragma unroll
    for (int i = 0; i < NM; ++i) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(p + 4 * i));
      acc[i][0] += v.x; acc[i][1] += v.y; acc[i][2] += v.z; acc[i][3] += v.w;
    }
  }
  if (lane == 0) *cnt = 0;
  return true;
}

// ------------------------------------------------------------ local dispatch --
// Every gate/up and down CTA builds the dispatch index of the call in shared
// memory from the T * k top-k ids (at most 128 pairs): pairs sorted by
// (expert, pair id) - the stable counting sort of the router's dispatch - the
// active experts in ascending id, and each one's segment of the sorted list.
// A group of nthr >= 128 threads does it (tid: the index in the group),
// synchronised on named barrier `bar`.  Gate/up CTA 0 also writes the index
// to the workspace (counts and offsets of every expert, the pair list, the
// active list): the routing outputs of the call.  Ids outside [0, E), or an
// expert named twice by one token (a top-k choice names distinct experts),
// are reported as MOE_ERR_DEVICE_BAD_INDEX and their pairs left out.
constexpr int kMaxPairs = kMaxT * 16;

struct LocalDispatch {
  int pe[kMaxPairs];        // expert of pair p (-1: left out)
  int sorted[kMaxPairs];    // pair ids by (expert, pair id); the valid ones first
  int act[kMaxPairs];       // active experts, ascending
  int aoff[kMaxPairs + 1];  // segment of active expert i: sorted[aoff[i] .. aoff[i + 1])
  int wcnt[kExpertThreads / 32];
  int n_active, n_valid;
};

static __device__ void local_dispatch(const ExpertArgs& a, LocalDispatch& d, bool write_global, int tid, int nthr,
                                      uint32_t bar) {
  const int lane = tid & 31, warp = tid >> 5;
  const int P = a.T * a.k, E = a.E, k = a.k;
  if (tid < P) {
    int e = __ldcg(a.rb.topk_idx + tid);
    if ((unsigned)e >= (unsigned)E) {
      report_error(a.rb.ctrl, (uint32_t)MOE_ERR_DEVICE_BAD_INDEX, 0x040);
      e = -1;
    }
    d.pe[tid] = e;
  }
  bar_sync_n(bar, nthr);
  bool dup = false;  // the same expert twice in one token: keep the first
  if (tid < P && d.pe[tid] >= 0)
    for (int q = tid / k * k; q < tid; ++q) dup = dup || d.pe[q] == d.pe[tid];
  bar_sync_n(bar, nthr);
  if (dup) {
    report_error(a.rb.ctrl, (uint32_t)MOE_ERR_DEVICE_BAD_INDEX, 0x041);
    d.pe[tid] = -1;
  }
  bar_sync_n(bar, nthr);
  // rank of each pair under the key (expert, pair id), left-out pairs last
  if (tid < P) {
    const int ep = d.pe[tid] >= 0 ? d.pe[tid] : E;
    const long kp = (long)ep * kMaxPairs + tid;
    int rank = 0;
    for (int q = 0; q < P; ++q) {
      const int eq = d.pe[q] >= 0 ? d.pe[q] : E;
      rank += ((long)eq * kMaxPairs + q) < kp;
    }
    d.sorted[rank] = tid;
  }
  bar_sync_n(bar, nthr);
  // segment starts: the first sorted entry of each expert (ballots over the pair warps)
  bool first = false;
  int e = -1;
  if (tid < P) {
    e = d.pe[d.sorted[tid]];
    first = e >= 0 && (tid == 0 || d.pe[d.sorted[tid - 1]] != e);
  }
  const uint32_t bal = __ballot_sync(0xFFFFFFFFu, first);
  const uint32_t valid = __ballot_sync(0xFFFFFFFFu, tid < P && e >= 0);
  if (lane == 0) d.wcnt[warp] = __popc(bal) | (__popc(valid) << 16);
  bar_sync_n(bar, nthr);
  int base = 0, nact = 0, nvalid = 0;
  for (int w = 0; w < nthr / 32; ++w) {
    if (w < warp) base += d.wcnt[w] & 0xFFFF;
    nact += d.wcnt[w] & 0xFFFF;
    nvalid += d.wcnt[w] >> 16;
  }
  if (first) {
    const int slot = base + __popc(bal & ((1u << lane) - 1u));
    d.act[slot] = e;
    d.aoff[slot] = tid;
  }
  if (tid == 0) {
    d.n_active = nact;
    d.n_valid = nvalid;
    d.aoff[nact] = nvalid;
  }
  bar_sync_n(bar, nthr);
  if (!write_global) return;
  for (int i = tid; i < d.n_valid; i += nthr) a.rb.pair[i] = d.sorted[i];
  for (int i = tid; i < d.n_active; i += nthr) a.rb.act[i] = d.act[i];
  // counts and offsets of every expert: binary search of the sorted valid pairs
  for (int x = tid; x <= E; x += nthr) {
    int lo = 0, hi = d.n_valid;  // first sorted position whose expert is >= x
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (d.pe[d.sorted[mid]] < x) lo = mid + 1; else hi = mid;
    }
    a.rb.off[x] = lo;
    if (x < E) {
      int lo2 = lo, hi2 = d.n_valid;  // first position whose expert is > x
      while (lo2 < hi2) {
        const int mid = (lo2 + hi2) >> 1;
        if (d.pe[d.sorted[mid]] <= x) lo2 = mid + 1; else hi2 = mid;
      }
      a.rb.cnt[x] = lo2 - lo;
    }
  }
  if (tid == 0) a.rb.ctrl->n_active = d.n_active;
}

// --------------------------------------------------------------- gate / up --

template <int FR, int FS, int PF>
__device__ __forceinline__ void gu_tile(int fmt_is_shared, const Mat (&m)[2], int row0, int kb, int Kw, int bu,
                                        const __half* xrow, float (&acc)[2][4], float* bpart, uint8_t* ring) {
  if (fmt_is_shared) {
    if constexpr (FS != 0) warp_tile<FS, 2, PF>(m, row0, kb, Kw, bu, xrow, acc, bpart, ring);
  } else {
    warp_tile<FR, 2, PF>(m, row0, kb, Kw, bu, xrow, acc, bpart, ring);
  }
}

// MINB CTAs per SM: 2 with three ring stages per warp (large batches: about
// one task per warp, each streaming with more bytes in flight), 3 with two
// (small batches: more warps in flight).
template <int FR, int FS, int MINB>
__global__ void __launch_bounds__(kExpertThreads, MINB) gateup_kernel(ExpertArgs a) {
  constexpr int PF = gu_stages(MINB);
  extern __shared__ __align__(16) uint8_t smem[];
  const int T = a.T, H = a.H, I = a.I, k = a.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int xs_stride = a.xs_tok_stride;
  // [T][xs_stride]; columns without a token read row 0 (their results are discarded)
  __half* xs = reinterpret_cast<__half*>(smem);
  uint8_t* ring = smem + (size_t)T * xs_stride * 2 + (size_t)warp * PF * stage_bytes<2>();
  __shared__ int s_pexp[kMaxT + 1];
  __shared__ const uint16_t* s_src[kMaxT];

  // the activations are an input of the call: stage them before waiting on the router
  if (tid < T) s_src[tid] = a.x + (size_t)tid * H;
  __syncthreads();
  stage_rows_f16(s_src, nullptr, T, H, xs, xs_stride, s_pexp);
  if (tid == 0) s_pexp[T] = 0;
  __syncthreads();

  const int tpe = I / 16;
  const int stiles = FS ? a.Is / 16 : 0;
  const int S = a.gu_slices, Ss = FS ? a.gu_slices_s : 1, St = a.gu_slices_t;
  const int Br = dec_blocks(FR, H), bur = dec_block_units(FR, H);
  const int Bs = FS ? dec_blocks(FS, H) : 1, bus = FS ? dec_block_units(FS, H) : 1;
  const int r = lane >> 2, c = lane & 3;
  // Tasks: the shared expert's tiles first (numbered 0 .. n_shared_tasks - 1,
  // their split counters and block sums at the start of the buffers), then
  // the routed tiles.  Every warp starts on task warp * grid + CTA, so
  // consecutive tasks (the shared expert's first of all) land on different
  // SMs; later tasks are handed out one at a time from a global counter, so
  // warps that finish early take more.  The shared expert depends on the
  // tokens only, so a warp whose first task is a shared one runs it before
  // waiting for the router.  Routed tiles that do not fit in the first wave
  // (the tail) are split into St > S slices, so the warps that finish the
  // first wave share them in short pieces.
  const int n_shared_tasks = stiles * Ss;
  const int nw = gridDim.x * kWarps;
  const size_t shared_blocks = Ss > 1 ? (size_t)stiles * Bs : 0;  // block sums of the shared tiles
  __shared__ LocalDispatch ld;
  int n_rtiles = 0, n_tail = 0, n_head = 0, n_tasks = n_shared_tasks;
  bool routed_known = false;
  uint32_t* next = &a.rb.ctrl->gu_next;

  // one task: shared tile q < n_shared_tasks, else a routed tile (after the local dispatch)
  auto run_task = [&](int q) {
    const bool shared_item = q < n_shared_tasks;
    int Si, tile_id, slice;  // K slices of this tile, tile (shared tiles first), slice
    if (shared_item) {
      Si = Ss; tile_id = q / Ss; slice = q % Ss;
    } else if (q - n_shared_tasks < n_head * S) {
      const int qq = q - n_shared_tasks;
      Si = S; tile_id = stiles + qq / S; slice = qq % S;
    } else {
      const int qt = q - n_shared_tasks - n_head * S;
      Si = St; tile_id = stiles + n_head + qt / St; slice = qt % St;
    }
    const int Kw = H / Si;
    int e = 0, tile, col_tok = 0, col_pair[2] = {-1, -1}, col_tokc[2] = {0, 0};
    if (!shared_item) {
      const int rt = tile_id - stiles;  // routed tile index
      const int slot = rt / tpe;
      tile = rt - slot * tpe;
      e = ld.act[slot];
      const int off = ld.aoff[slot], ncols = ld.aoff[slot + 1] - off;  // <= T: distinct experts per token
      if (r < ncols) col_tok = ld.sorted[off + r] / k;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int n = 2 * c + j;
        if (n < ncols) {
          col_pair[j] = ld.sorted[off + n];
          col_tokc[j] = col_pair[j] / k;
        }
      }
    } else {
      tile = tile_id;
      if (r < T) col_tok = r;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int n = 2 * c + j;
        if (n < T) { col_pair[j] = n; col_tokc[j] = n; }
      }
    }
    const int fmt = shared_item ? FS : FR;
    const int N = shared_item ? a.Is : I;
    const QW& qg = shared_item ? a.sgate : a.gate;
    const QW& qu = shared_item ? a.sup : a.up;
    const Mat m[2] = {mat_of(qg, fmt, e, N, H), mat_of(qu, fmt, e, N, H)};
    const int row0 = tile * 16;
    const int B = shared_item ? Bs : Br;
    // block sums: shared tiles first, then the routed ones (all when S > 1, else the tail only)
    float* tile_part;
    if (shared_item) {
      tile_part = a.gu_part + (size_t)tile * Bs * (32 * 8);
    } else {
      const int rt = tile_id - stiles;
      const int rslot = S > 1 ? rt : max(rt - n_head, 0);  // (unused for unsplit tiles)
      tile_part = a.gu_part + (shared_blocks + (size_t)rslot * Br) * (32 * 8);
    }
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    gu_tile<FR, FS, PF>(shared_item, m, row0, slice * Kw, Kw, shared_item ? bus : bur, xs + (size_t)col_tok * xs_stride,
                    acc, Si > 1 ? tile_part + (size_t)slice * (B / Si) * (32 * 8) : nullptr, ring);
    if (block_reduce<2>(acc, tile_part, a.gu_cnt + tile_id, Si, B)) {
      const float tsg = (fmt == MOE_FMT_NVFP4) ? __ldg(qg.ts + e) : 1.f;
      const float tsu = (fmt == MOE_FMT_NVFP4) ? __ldg(qu.ts + e) : 1.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int cj = j & 1;
        const int row = row0 + r + ((j & 2) ? 8 : 0);
        const int out = col_pair[cj];
        if (out >= 0) {
          const float sc = exp2i(s_pexp[col_tokc[cj]]);
          const float gv = acc[0][j] * sc * tsg, uv = acc[1][j] * sc * tsu;
          const uint16_t hb = float_to_bf16_bits(silu_f(gv) * uv);
          if (shared_item) a.hs[(size_t)out * a.Is + row] = hb;
          else a.h[(size_t)out * I + row] = hb;
        }
      }
    }
  };

  // The shared expert depends on the tokens only: warps [0, ws) of this CTA start on a shared task
  // (q0 < n_shared_tasks) and run it before the router's results are needed, while the other warps
  // (at least four) wait for the router and build the dispatch; the shared-task warps then take it
  // over a named barrier, so a routed task never waits for a shared one.
  const int q0 = warp * gridDim.x + blockIdx.x;
  const int ws = n_shared_tasks > (int)blockIdx.x
                     ? min(kWarps, (n_shared_tasks - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x)
                     : 0;
  const bool early = ws <= kWarps - 4;
  const bool ran_first = early && warp < ws;
  if (ran_first) {
    run_task(q0);
    pdl_wait();
    bar_sync_n(2, kExpertThreads);  // the dispatch is built
  } else {
    pdl_wait();
    const int g0 = early ? 32 * ws : 0;
    local_dispatch(a, ld, blockIdx.x == 0, tid - g0, kExpertThreads - g0, 1);
    // the down kernel may start now: the router has completed, so its prologue can read the top-k ids
    pdl_launch_dependents();
    if (early && ws > 0) bar_arrive_n(2, kExpertThreads);
  }
  {
    n_rtiles = ld.n_active * tpe;
    if (St > S) {
      const long first = (long)n_shared_tasks + (long)n_rtiles * S;
      if (first > nw) n_tail = (int)min((long)min(n_rtiles, a.gu_tail_cap), (first - nw + S - 1) / S);
    }
    n_head = n_rtiles - n_tail;
    n_tasks = n_shared_tasks + n_head * S + n_tail * St;
    routed_known = true;
  }
  (void)routed_known;
  // later tasks one at a time from the counter, each fetched while the previous one runs
  int qn = 0;
  int q = q0;
  if (ran_first) {
    if (lane == 0) qn = nw + (int)atomicAdd(next, 1u);
    q = __shfl_sync(0xFFFFFFFFu, qn, 0);
  }
  while (q < n_tasks) {
    if (lane == 0) qn = nw + (int)atomicAdd(next, 1u);
    run_task(q);
    q = __shfl_sync(0xFFFFFFFFu, qn, 0);
  }
}

// -------------------------------------------------------------------- down --

// One element of a down projection's output: P[pair, row] (routed) or S[token, row]
// (shared), FP32, or rounded to BF16 under the bf16-partials lever.
__device__ __forceinline__ void store_partial(const ExpertArgs& a, bool shared_item, int out, int row, float v) {
  const size_t i = (size_t)out * a.H + row;
  if (a.p_bf16) {
    uint16_t* d = reinterpret_cast<uint16_t*>(shared_item ? a.S : a.P);
    d[i] = float_to_bf16_bits(v);
  } else {
    (shared_item ? a.S : a.P)[i] = v;
  }
}

template <int FR, int FS>
__global__ void __launch_bounds__(kExpertThreads, 2) down_kernel(ExpertArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int T = a.T, H = a.H, I = a.I, k = a.k;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hs_stride = a.hs_tok_stride;
  const int SG = a.dn_segs;  // segments staged at once
  const size_t seg_halfs = (size_t)(kMaxT + 1) * hs_stride;
  __half* hsm = reinterpret_cast<__half*>(smem);  // [SG][kMaxT + 1][hs_stride]
  uint8_t* ring = smem + (size_t)SG * seg_halfs * 2 + (size_t)warp * kStagesDN * stage_bytes<1>();
  __shared__ int s_pexp[kMaxDnSegs][kMaxT + 1];
  __shared__ int s_col_out[kMaxDnSegs][kMaxT];
  __shared__ int s_ncols[kMaxDnSegs];
  __shared__ const uint16_t* s_src[kMaxT];

  __shared__ LocalDispatch ld;
  pdl_launch_dependents();
  // The gate/up kernel let this grid start only after its own wait on the router, so the top-k
  // ids are complete: the dispatch, the task range and the L2 prefetch of this CTA's weights run
  // before the wait for gate/up's h.
  local_dispatch(a, ld, false, tid, kExpertThreads, 1);
  const int n_active = ld.n_active;
  const int tpe = H / 16;
  const int S = a.dn_slices;
  const int Br = dec_blocks(FR, I), Bs = FS ? dec_blocks(FS, a.Is) : 1;
  const int sh = FS ? 1 : 0;
  const int n_seg = n_active + sh;                 // expert segments, the shared one first
  const int tasks_per_seg = tpe * S;
  const int n_tasks = n_seg * tasks_per_seg;
  // contiguous task range per CTA, split by weight bytes (a shared-expert task
  // can cost more than a routed one)
  const long long cr = (long long)(data_bytes(FR, H, I) + scale_bytes(FR, H, I)) / tasks_per_seg;
  const long long cs = FS ? (long long)(data_bytes(FS, H, a.Is) + scale_bytes(FS, H, a.Is)) / tasks_per_seg : 0;
  const long long ns = (long long)sh * tasks_per_seg;
  const long long total = ns * cs + (long long)n_active * tasks_per_seg * cr;
  auto task_at = [&](long long cost) -> int {
    if (cost <= 0) return 0;
    if (cost >= total) return n_tasks;
    if (cost < ns * cs) return (int)((cost + cs - 1) / cs);
    return (int)(ns + (cost - ns * cs + cr - 1) / cr);
  };
  const int q0 = task_at(total * blockIdx.x / gridDim.x);
  const int q1 = task_at(total * (blockIdx.x + 1) / gridDim.x);
  const int r = lane >> 2, c = lane & 3;
  // this CTA's weight bytes (one contiguous row range per segment) are brought into L2 while
  // gate/up runs; the warps' rings then read them from L2
  if (q0 < q1 && tid < 32) {
    const int seg_a = q0 / tasks_per_seg, seg_b = (q1 - 1) / tasks_per_seg;
    for (int seg = seg_a + lane; seg <= seg_b; seg += 32) {
      const bool shared_item = FS && seg == 0;
      const int fmt = shared_item ? FS : FR;
      const int K = shared_item ? a.Is : I;
      const int e = shared_item ? 0 : ld.act[seg - sh];
      const QW& qd = shared_item ? a.sdown : a.down;
      const int t_a = max(q0, seg * tasks_per_seg) - seg * tasks_per_seg;
      const int t_b = min(q1, (seg + 1) * tasks_per_seg) - seg * tasks_per_seg;  // tasks [t_a, t_b)
      const int tile_a = t_a / S, tile_b = (t_b + S - 1) / S;                    // row tiles they touch
      const size_t rb = (size_t)K * Fm_bits(fmt) / 8;                            // bytes of one row
      const uint8_t* d0 = qd.data + (size_t)e * data_bytes(fmt, H, K) + (size_t)tile_a * 16 * rb;
      prefetch_l2_share(d0, (size_t)(tile_b - tile_a) * 16 * rb, 0, 1);
      if (fmt != MOE_FMT_FP8_B128) {
        const size_t sr = scale_bytes(fmt, H, K) / H;                            // scale bytes of one row
        prefetch_l2_share(qd.scales + (size_t)e * scale_bytes(fmt, H, K) + (size_t)tile_a * 16 * sr,
                          (size_t)(tile_b - tile_a) * 16 * sr, 0, 1);
      }
    }
  }

  pdl_wait();
  // the gate/up kernel has finished: leave its task counter at zero for the next call
  if (blockIdx.x == 0 && tid == 0) a.rb.ctrl->gu_next = 0;
  if (q0 >= q1) return;

  // the segments of [q0, q1), staged SG at a time; inside a group the warps
  // take the tasks in turn with no barrier between segments
  const int seg_lo = q0 / tasks_per_seg, seg_hi = (q1 - 1) / tasks_per_seg;
  for (int sg = seg_lo; sg <= seg_hi; sg += SG) {
    const int sg_end = min(seg_hi + 1, sg + SG);
    __syncthreads();  // the previous group's rows are no longer read
    for (int seg = sg; seg < sg_end; ++seg) {
      const int i = seg - sg;
      const bool shared_item = FS && seg == 0;
      int ncols;
      if (!shared_item) {
        const int slot = seg - sh;
        ncols = min(ld.aoff[slot + 1] - ld.aoff[slot], kMaxT);
        if (tid < kMaxT) {
          if (tid < ncols) {
            const int p = ld.sorted[ld.aoff[slot] + tid];
            s_src[tid] = a.h + (size_t)p * I;
            s_col_out[i][tid] = p;
          } else {
            s_col_out[i][tid] = -1;
          }
        }
      } else {
        ncols = T;
        if (tid < kMaxT) {
          if (tid < T) s_src[tid] = a.hs + (size_t)tid * a.Is;
          s_col_out[i][tid] = tid < T ? tid : -1;
        }
      }
      if (tid == 0) s_ncols[i] = ncols;
      __syncthreads();
      // each staged row's largest magnitude is found here (the rows are h, just written to L2)
      stage_rows_f16(s_src, nullptr, ncols, shared_item ? a.Is : I, hsm + (size_t)i * seg_halfs, hs_stride,
                     s_pexp[i]);
      __syncthreads();  // s_src / s_amax are reused by the next segment
    }
    const int t_lo = max(q0, sg * tasks_per_seg), t_hi = min(q1, sg_end * tasks_per_seg);
    if (S == 1) {
      // this warp's tiles of each segment (every kWarps-th task) as one stream
      for (int seg = sg; seg < sg_end; ++seg) {
        const int a0 = max(t_lo, seg * tasks_per_seg), a1 = min(t_hi, (seg + 1) * tasks_per_seg);
        if (a0 >= a1) continue;
        const int qs = a0 + (((t_lo + warp - a0) % kWarps) + kWarps) % kWarps;
        if (qs >= a1) continue;
        const int ntile = (a1 - 1 - qs) / kWarps + 1;
        const int i = seg - sg;
        const bool shared_item = FS && seg == 0;
        const int e = shared_item ? 0 : ld.act[seg - sh];
        const int ncols = s_ncols[i];
        const int K = shared_item ? a.Is : I;
        const int fmt = shared_item ? FS : FR;
        const QW& qd = shared_item ? a.sdown : a.down;
        const Mat m[1] = {mat_of(qd, fmt, e, H, K)};
        const int bu = dec_block_units(fmt, K);
        const __half* xrow = hsm + (size_t)i * seg_halfs + (size_t)(r < ncols ? r : ncols) * hs_stride;
        const int tile0 = qs - seg * tasks_per_seg;
        const float ts = (fmt == MOE_FMT_NVFP4) ? __ldg(qd.ts + e) : 1.f;
        auto epi = [&](int t, float (&acc)[1][4]) {
          const int tile = tile0 + t * kWarps;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int col = 2 * c + (j & 1);
            const int row = tile * 16 + r + ((j & 2) ? 8 : 0);
            const int out = s_col_out[i][col];
            if (out >= 0) store_partial(a, shared_item, out, row, acc[0][j] * exp2i(s_pexp[i][col]) * ts);
          }
        };
        if (shared_item) {
          if constexpr (FS != 0) warp_tiles<FS, 1, kStagesDN>(m, tile0 * 16, 16 * kWarps, ntile, K, bu, xrow, ring, epi);
        } else {
          warp_tiles<FR, 1, kStagesDN>(m, tile0 * 16, 16 * kWarps, ntile, K, bu, xrow, ring, epi);
        }
      }
      continue;
    }
    for (int q = t_lo + warp; q < t_hi; q += kWarps) {
      const int seg = q / tasks_per_seg, i = seg - sg;
      const bool shared_item = FS && seg == 0;
      const int e = shared_item ? 0 : ld.act[seg - sh];
      const int ncols = s_ncols[i];
      const int K = shared_item ? a.Is : I;
      const int fmt = shared_item ? FS : FR;
      const QW& qd = shared_item ? a.sdown : a.down;
      const Mat m[1] = {mat_of(qd, fmt, e, H, K)};
      const int Kw = K / S;
      const int B = dec_blocks(fmt, K), bu = dec_block_units(fmt, K);
      const __half* xrow = hsm + (size_t)i * seg_halfs + (size_t)(r < ncols ? r : ncols) * hs_stride;
      const int local = q - seg * tasks_per_seg;
      const int tile = local / S, slice = local - tile * S;
      float acc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
      const int tile_id = shared_item ? n_active * tpe + tile : (seg - sh) * tpe + tile;
      float* tile_part = a.dn_part + (shared_item ? (size_t)n_active * tpe * Br + (size_t)tile * Bs
                                                  : (size_t)tile_id * Br) * (32 * 4);
      float* bpart = S > 1 ? tile_part + (size_t)slice * (B / S) * (32 * 4) : nullptr;
      if (shared_item) {
        if constexpr (FS != 0) warp_tile<FS, 1, kStagesDN>(m, tile * 16, slice * Kw, Kw, bu, xrow, acc, bpart, ring);
      } else {
        warp_tile<FR, 1, kStagesDN>(m, tile * 16, slice * Kw, Kw, bu, xrow, acc, bpart, ring);
      }
      if (!block_reduce<1>(acc, tile_part, a.dn_cnt + tile_id, S, B)) continue;
      const float ts = (fmt == MOE_FMT_NVFP4) ? __ldg(qd.ts + e) : 1.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = 2 * c + (j & 1);
        const int row = tile * 16 + r + ((j & 2) ? 8 : 0);
        const int out = s_col_out[i][col];
        if (out >= 0) store_partial(a, shared_item, out, row, acc[0][j] * exp2i(s_pexp[i][col]) * ts);
      }
    }
  }
}

// y[t] = bf16( sum_j w[t, j] * P[t*k + j] (+ g_t S[t]) ), j ascending, after the
// down kernel (programmatic dependent launch; waits for its completion).  g_t
// is the shared expert's sigmoid gate when the layer has one, else 1.
__device__ __forceinline__ float4 load_partial4(const float* base, size_t row, int H, int c4, int bf16) {
  if (!bf16) return __ldcg(reinterpret_cast<const float4*>(base + row * H) + c4);
  const uint2 v = __ldcg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(base) + row * H) + c4);
  return make_float4(bf16_bits_to_float(v.x & 0xFFFF), bf16_bits_to_float(v.x >> 16), bf16_bits_to_float(v.y & 0xFFFF),
                     bf16_bits_to_float(v.y >> 16));
}

template <int FS>
__global__ void __launch_bounds__(256) combine_kernel(ExpertArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int H = a.H, k = a.k;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;  // (token, 4 columns)
  if (i >= a.T * (H / 4)) return;
  const int t = i / (H / 4), c4 = i - t * (H / 4);
  // all k partial rows are loaded before the j-ordered fma chain (k <= 16)
  float wj[16];
  float4 pj[16];
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j < k) {
      wj[j] = __ldcg(a.rb.topk_w + t * k + j);
      pj[j] = load_partial4(a.P, (size_t)(t * k + j), H, c4, a.p_bf16);
    }
  float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j < k) {
      y[0] = __fmaf_rn(wj[j], pj[j].x, y[0]);
      y[1] = __fmaf_rn(wj[j], pj[j].y, y[1]);
      y[2] = __fmaf_rn(wj[j], pj[j].z, y[2]);
      y[3] = __fmaf_rn(wj[j], pj[j].w, y[3]);
    }
  if (FS) {
    const float4 sv = load_partial4(a.S, (size_t)t, H, c4, a.p_bf16);
    const float g = a.shared_g ? __ldcg(a.shared_g + t) : 1.f;
    y[0] = __fmaf_rn(g, sv.x, y[0]);
    y[1] = __fmaf_rn(g, sv.y, y[1]);
    y[2] = __fmaf_rn(g, sv.z, y[2]);
    y[3] = __fmaf_rn(g, sv.w, y[3]);
  }
  const uint32_t lo = (uint32_t)float_to_bf16_bits(y[0]) | ((uint32_t)float_to_bf16_bits(y[1]) << 16);
  const uint32_t hi = (uint32_t)float_to_bf16_bits(y[2]) | ((uint32_t)float_to_bf16_bits(y[3]) << 16);
  reinterpret_cast<uint2*>(a.y + (size_t)t * H)[c4] = make_uint2(lo, hi);
}

template <int FR, int FS>
cudaError_t launch_pdl_kernel(void (*kern)(ExpertArgs), const ExpertArgs& a, size_t smem, cudaStream_t s) {
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kExpertThreads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms * per_sm);
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

template <int FR>
cudaError_t launch_expert_pair(int sfmt, bool down, const ExpertArgs& a, size_t smem, cudaStream_t s) {
  switch (sfmt) {
#define QMOE_CASE(FS)                                                                              \
  case FS:                                                                                         \
    return down ? launch_pdl_kernel<FR, FS>(down_kernel<FR, FS>, a, smem, s)                       \
                : (a.T <= kGuSmallT ? launch_pdl_kernel<FR, FS>(gateup_kernel<FR, FS, 3>, a, smem, s)    \
                                    : launch_pdl_kernel<FR, FS>(gateup_kernel<FR, FS, 2>, a, smem, s));
    QMOE_CASE(0)
    QMOE_CASE(MOE_FMT_NVFP4)
    QMOE_CASE(MOE_FMT_MXFP4)
    QMOE_CASE(MOE_FMT_INT4_G64)
    QMOE_CASE(MOE_FMT_INT8_G64)
    QMOE_CASE(MOE_FMT_FP8_B128)
    QMOE_CASE(MOE_FMT_INT4_G128)
#undef QMOE_CASE
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dec
}  // namespace qmoe
