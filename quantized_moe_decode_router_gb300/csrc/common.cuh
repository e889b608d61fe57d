// Device-side building blocks shared by the MoE kernels (sm_103a).
//
// Format decoding in registers (DGPP forum post 15 "Lossless bf12": weights
// are rebuilt in registers, never as a dequantized copy), tensor-core MMA
// wrappers, and the float-float arithmetic of the router.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace qmoe {

constexpr int kWarp = 32;

// ---------------------------------------------------------------- workspace --

// Control block at the start of every workspace (zeroed by moe_workspace_init;
// every kernel leaves the counters it uses back at zero).
struct Ctrl {
  uint32_t error;          // MOE_ERR_DEVICE_* code of the first device-side error, 0 if none
  uint32_t error_info;     // where it happened (kernel-specific)
  uint32_t router_arrive;  // CTAs of the router kernel that finished their logits
  int32_t n_active;        // experts with at least one routed pair
  int32_t n_tiles;         // prefill: token tiles in the GEMM tile list
  uint32_t gu_next;        // decode gate/up: next task to hand out (zeroed by the router)
  uint32_t pad[2];
};

__device__ __forceinline__ void report_error(Ctrl* ctrl, uint32_t code, uint32_t info) {
  if (atomicCAS(&ctrl->error, 0u, code) == 0u) ctrl->error_info = info;
}

// ------------------------------------------------------------ small helpers --

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ldg_nc_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ldg_nc_u16(const void* p) {
  unsigned short r;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t ldg_nc_u8(const void* p) {
  unsigned short r;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(r) : "l"(p));
  return r & 0xFF;
}

// Asynchronous global -> shared copies (cp.async), completion tracked per thread.
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Hint: bring [p, p + bytes) into L2 (bulk prefetch, no completion to wait for).
// p 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Prefetch the 16-byte aligned part of share `part` of `parts` equal shares of [base, base + len).
__device__ __forceinline__ void prefetch_l2_share(const uint8_t* base, size_t len, int part, int parts) {
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(base);
  uintptr_t lo = b0 + len * (size_t)part / (size_t)parts, hi = b0 + len * (size_t)(part + 1) / (size_t)parts;
  lo = (lo + 15) & ~(uintptr_t)15;
  hi &= ~(uintptr_t)15;
  constexpr uintptr_t kMax = 1u << 20;  // one request at most 1 MiB
  while (lo < hi) {
    const uintptr_t n = hi - lo < kMax ? hi - lo : kMax;
    prefetch_l2_bulk(reinterpret_cast<const void*>(lo), (uint32_t)n);
    lo += n;
  }
}

// Named barrier `id` over n threads (a multiple of 32): wait for all, or arrive only.
__device__ __forceinline__ void bar_sync_n(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive_n(uint32_t id, uint32_t n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// E8M0 scale code of an MXFP4 activation block with largest magnitude amax:
// e = the smallest integer with 6 * 2^e >= amax (0 for amax = 0), code e + 127
// clamped to [0, 254].  amax = f 2^p with f in [0.5, 1) puts log2(amax / 6) in
// [p - 3.585, p - 2.585), so e is p - 3 or p - 2; the comparison is exact.
__device__ __forceinline__ int mxfp4_act_scale_code(float amax) {
  if (!(amax > 0.f)) return 127;
  int p;
  frexpf(amax, &p);
  const int e = (6.0f * ldexpf(1.0f, p - 3) >= amax) ? p - 3 : p - 2;
  return min(max(e + 127, 0), 254);
}

// 2^e as a float for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// E8M0 code -> float (2^(c-127); 255 is NaN).
__device__ __forceinline__ float e8m0_to_float(uint32_t c) {
  if (c == 0) return __uint_as_float(0x00400000u);  // 2^-127, a binary32 subnormal
  if (c == 255) return __uint_as_float(0x7FC00000u);
  return __uint_as_float(c << 23);
}

// ------------------------------------------------------- format conversions --

// Two E2M1 codes in one byte -> f16x2 (low nibble -> low half), exact.
// Returns the four f16x2 pairs of a 32-bit word of eight codes, in K order.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&out)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(w));
}

// f32 -> E4M3 code, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t f32_to_e4m3_sat(float x) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(x));
  return r & 0xFF;
}

// Two f32 -> two E2M1 codes in one byte (lo -> low nibble), RNE, saturating to +-6.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2_sat(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}" : "=r"(r) : "f"(hi), "f"(lo));
  return r & 0xFF;
}

// Two E4M3 codes (low byte -> low half) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  unsigned short s = (unsigned short)two_bytes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(s));
  return r;
}

// One E4M3 code broadcast to both halves of an f16x2.
__device__ __forceinline__ uint32_t e4m3_bcast_f16x2(uint32_t byte) {
  return e4m3x2_to_f16x2((byte & 0xFF) * 0x0101u);
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                      *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t mask, uint32_t x) {
  uint32_t r;  // (a & mask) ^ x
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(a), "r"(mask), "r"(x));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Eight two's-complement int4 codes (low nibble = even k) -> four f16x2 of the
// exact integers, paired as (k0,k4), (k1,k5), (k2,k6), (k3,k7).  Uses the
// 1024 + u f16 encoding of a small unsigned integer u in the mantissa.
__device__ __forceinline__ void int4x8_to_f16x2_paired(uint32_t w, uint32_t (&out)[4]) {
  const uint32_t w8 = w >> 8;
  const uint32_t k1032 = 0x64086408u;  // f16x2 (1032, 1032)
  const uint32_t k1_16 = 0x2C002C00u;  // f16x2 (1/16, 1/16)
  const uint32_t km72 = 0xD480D480u;   // f16x2 (-72, -72)
  out[0] = hsub2_u32(lop3_and_xor(w, 0x000F000Fu, 0x64086408u), k1032);
  out[1] = hfma2_u32(lop3_and_xor(w, 0x00F000F0u, 0x64806480u), k1_16, km72);
  out[2] = hsub2_u32(lop3_and_xor(w8, 0x000F000Fu, 0x64086408u), k1032);
  out[3] = hfma2_u32(lop3_and_xor(w8, 0x00F000F0u, 0x64806480u), k1_16, km72);
}

// Four int8 codes -> two f16x2 of the exact integers, pairs (k0,k1), (k2,k3).
__device__ __forceinline__ void int8x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t wx = w ^ 0x80808080u;  // offset binary: u = q + 128
  const uint32_t k1152 = 0x64806480u;   // f16x2 (1152, 1152)
  lo = hsub2_u32(prmt(wx, 0x64646464u, 0x5140u), k1152);
  hi = hsub2_u32(prmt(wx, 0x64646464u, 0x5342u), k1152);
}

// Four E4M3 codes -> two f16x2, pairs (k0,k1), (k2,k3), exact.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = e4m3x2_to_f16x2(w & 0xFFFFu);
  hi = e4m3x2_to_f16x2(w >> 16);
}

// ------------------------------------------------------------ tensor cores --

// D = A(16x16, f16, row) * B(16x8, f16, col) + C, FP32 accumulate (legacy
// warp-level MMA; used where the problem is a matrix-vector product and the
// tensor pipe only relieves the CUDA cores of the FMAs).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------ float-float (router) --

// Knuth's TwoSum: s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bp = __fsub_rn(s, a);
  float ap = __fsub_rn(s, bp);
  e = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

// Accumulate the exact product a*b into the unevaluated sum (hi + lo):
// TwoProd via FMA, then TwoSum (Ogita, Rump and Oishi, "Accurate sum and dot
// product", SIAM J. Sci. Comput. 26(6), 2005, algorithm Dot2).
__device__ __forceinline__ void dot2_step(float a, float b, float& hi, float& lo) {
  float p = __fmul_rn(a, b);
  float q = __fmaf_rn(a, b, -p);
  float s, e;
  two_sum(hi, p, s, e);
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(q, e));
}

// Merge two float-float partial sums.
__device__ __forceinline__ void dot2_merge(float& hi, float& lo, float hi2, float lo2) {
  float s, e;
  two_sum(hi, hi2, s, e);
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(lo2, e));
}

}  // namespace qmoe
