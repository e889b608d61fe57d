// Format decode to FP32 (the register decode of every projection kernel,
// exposed for bit-exact checking) and the NVFP4 activation quantizer of the
// W4A4 lever (DGPP forum, weekly update on page 5: NVFP4 W4A4 prefill is
// opt-in).
#include "decode_impl.cuh"

namespace qmoe {

namespace {

__device__ __forceinline__ float h2lo(uint32_t v) { return __low2float(*reinterpret_cast<__half2*>(&v)); }
__device__ __forceinline__ float h2hi(uint32_t v) { return __high2float(*reinterpret_cast<__half2*>(&v)); }

// One thread decodes eight consecutive columns [k, k+8) of row R.
__global__ void dequantize_kernel(int fmt, QW w, int N, int K, int expert, int row0, int nrows, float* out) {
  const int groups = K / 8;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (long long)nrows * groups) return;
  const int r = (int)(gid / groups), k = (int)(gid - (long long)r * groups) * 8;
  const int R = row0 + r;
  const uint8_t* data = w.data + (size_t)expert * data_bytes(fmt, N, K);
  const uint8_t* sc = w.scales + (size_t)expert * scale_bytes(fmt, N, K);
  float v[8];
  if (fmt == MOE_FMT_NVFP4 || fmt == MOE_FMT_MXFP4 || fmt == MOE_FMT_INT4_G64 || fmt == MOE_FMT_INT4_G128) {
    const uint32_t wd = *reinterpret_cast<const uint32_t*>(data + (size_t)R * (K / 2) + k / 2);
    uint32_t f[4];
    if (fmt == MOE_FMT_INT4_G64) {
      int4x8_to_f16x2_paired(wd, f);  // pairs (k0,k4), (k1,k5), (k2,k6), (k3,k7)
      for (int j = 0; j < 4; ++j) { v[j] = h2lo(f[j]); v[j + 4] = h2hi(f[j]); }
      const uint32_t sb = *reinterpret_cast<const uint16_t*>(sc + ((size_t)R * (K / 64) + k / 64) * 2);
      const float s = __uint_as_float(sb << 16);
      for (int j = 0; j < 8; ++j) v[j] = v[j] * s;
    } else if (fmt == MOE_FMT_INT4_G128) {
      int4x8_to_f16x2_paired(wd ^ 0x88888888u, f);  // u - 8 (zero point 8)
      for (int j = 0; j < 4; ++j) { v[j] = h2lo(f[j]); v[j + 4] = h2hi(f[j]); }
      const uint16_t sb = *reinterpret_cast<const uint16_t*>(sc + ((size_t)R * (K / 128) + k / 128) * 2);
      const float s = __half2float(__ushort_as_half(sb));
      for (int j = 0; j < 8; ++j) v[j] = v[j] * s;
    } else {
      e2m1x8_to_f16x2(wd, f);
      if (fmt == MOE_FMT_NVFP4) {
        const uint32_t sb = sc[(size_t)R * (K / 16) + k / 16];
        const uint32_t s2 = e4m3_bcast_f16x2(sb);
        const float ts = w.ts[expert];
        for (int j = 0; j < 4; ++j) {
          const uint32_t p = hmul2_u32(f[j], s2);  // exact: at most 6 significant bits
          v[2 * j] = h2lo(p) * ts;
          v[2 * j + 1] = h2hi(p) * ts;
        }
      } else {
        const float s = e8m0_to_float(sc[(size_t)R * (K / 32) + k / 32]);
        for (int j = 0; j < 4; ++j) { v[2 * j] = h2lo(f[j]) * s; v[2 * j + 1] = h2hi(f[j]) * s; }
      }
    }
  } else {
    const uint2 wd = *reinterpret_cast<const uint2*>(data + (size_t)R * K + k);
    uint32_t lo0, hi0, lo1, hi1;
    float s;
    if (fmt == MOE_FMT_INT8_G64) {
      int8x4_to_f16x2(wd.x, lo0, hi0);
      int8x4_to_f16x2(wd.y, lo1, hi1);
      s = __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(sc + ((size_t)R * (K / 64) + k / 64) * 2))
                          << 16);
    } else {
      e4m3x4_to_f16x2(wd.x, lo0, hi0);
      e4m3x4_to_f16x2(wd.y, lo1, hi1);
      s = *reinterpret_cast<const float*>(sc + ((size_t)(R / 128) * (K / 128) + k / 128) * 4);
    }
    const uint32_t q[4] = {lo0, hi0, lo1, hi1};
    for (int j = 0; j < 4; ++j) { v[2 * j] = h2lo(q[j]) * s; v[2 * j + 1] = h2hi(q[j]) * s; }
  }
  float4* o = reinterpret_cast<float4*>(out + (size_t)r * K + k);
  o[0] = make_float4(v[0], v[1], v[2], v[3]);
  o[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// One thread per 16-element block.
__global__ void quantize_act_nvfp4_kernel(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales) {
  const int nb = K / 16;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (long long)rows * nb) return;
  const int r = (int)(gid / nb), b = (int)(gid - (long long)r * nb);
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)r * K + b * 16);
  const uint4 v0 = src[0], v1 = src[1];
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float a[16];
  float amax = 0.f;
  for (int j = 0; j < 8; ++j) {
    a[2 * j] = bf16_bits_to_float(w[j] & 0xFFFF);
    a[2 * j + 1] = bf16_bits_to_float(w[j] >> 16);
    amax = fmaxf(amax, fmaxf(fabsf(a[2 * j]), fabsf(a[2 * j + 1])));
  }
  const uint32_t sc = f32_to_e4m3_sat(__fdiv_rn(amax, 6.0f));
  const float s = h2lo(e4m3_bcast_f16x2(sc));
  uint32_t out[2] = {0, 0};
  if (s > 0.f) {
    for (int j = 0; j < 8; ++j) {
      const uint32_t byte = f32x2_to_e2m1x2_sat(__fdiv_rn(a[2 * j], s), __fdiv_rn(a[2 * j + 1], s));
      out[j >> 2] |= byte << (8 * (j & 3));
    }
  }
  *reinterpret_cast<uint2*>(codes + (size_t)r * (K / 2) + b * 8) = make_uint2(out[0], out[1]);
  scales[(size_t)r * nb + b] = (uint8_t)sc;
}

// MXFP4 activations, one thread per 32-element block: e = the smallest integer with 6 * 2^e >= amax
// (from amax = f 2^p, f in [0.5, 1): e is p - 3 or p - 2, decided by one exact comparison), scale
// code e + 127 clamped to [0, 254], codes e2m1_rne_sat(a * 2^-e) (exact scaling by a power of two).
__global__ void quantize_act_mxfp4_kernel(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales) {
  const int nb = K / 32;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (long long)rows * nb) return;
  const int r = (int)(gid / nb), b = (int)(gid - (long long)r * nb);
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)r * K + b * 32);
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = src[i];
    w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
  }
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j)
    amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(w[j] & 0xFFFF)), fabsf(bf16_bits_to_float(w[j] >> 16))));
  const int sc = mxfp4_act_scale_code(amax);
  const float inv = exp2i(127 - sc);  // 2^-e
  uint32_t out[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint32_t byte = f32x2_to_e2m1x2_sat(bf16_bits_to_float(w[j] & 0xFFFF) * inv,
                                              bf16_bits_to_float(w[j] >> 16) * inv);
    out[j >> 2] |= byte << (8 * (j & 3));
  }
  *reinterpret_cast<uint4*>(codes + (size_t)r * (K / 2) + b * 16) = make_uint4(out[0], out[1], out[2], out[3]);
  scales[(size_t)r * nb + b] = (uint8_t)sc;
}

}  // namespace

cudaError_t launch_quantize_act_mxfp4(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales,
                                      cudaStream_t s) {
  const long long n = (long long)rows * (K / 32);
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  quantize_act_mxfp4_kernel<<<(unsigned)blocks, threads, 0, s>>>(x, rows, K, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(int fmt, QW w, int N, int K, int expert, int row0, int nrows, float* out,
                              cudaStream_t s) {
  const long long n = (long long)nrows * (K / 8);
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  dequantize_kernel<<<(unsigned)blocks, threads, 0, s>>>(fmt, w, N, K, expert, row0, nrows, out);
  return cudaGetLastError();
}

cudaError_t launch_quantize_act_nvfp4(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales,
                                      cudaStream_t s) {
  const long long n = (long long)rows * (K / 16);
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  quantize_act_nvfp4_kernel<<<(unsigned)blocks, threads, 0, s>>>(x, rows, K, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_combine_decode(const ExpertArgs& a, cudaStream_t s) {
  const int n = a.T * (a.H / 4);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n + 255) / 256);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.sfmt ? cudaLaunchKernelEx(&cfg, dec::combine_kernel<1>, a) : cudaLaunchKernelEx(&cfg, dec::combine_kernel<0>, a);
}

}  // namespace qmoe
