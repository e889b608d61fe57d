// Approximate router logits for large token counts on tcgen05 (bf16 MMA).
//
// x is BF16, so x * w is exact in FP32 for a BF16 w.  The FP32 router matrix
// is split as Wr = hi + lo + r with hi = bf16(Wr), lo = bf16(Wr - hi) and
// |r| <= 2^-18 |Wr|; a[t, e] = x_t . hi_e + x_t . lo_e accumulates in the
// tensor core's FP32 accumulator.  The selection (prefill top-k) treats a as
// an approximation with the bound eps = (2 gamma_H + 2^-17) ||x_t|| ||Wr_e||
// (twice the bound of a sequential FP32 FMA sum, plus the split residual)
// and recomputes every expert that may reach the top-k exactly, so the
// routing is that of the correctly rounded FP32 logits (DGPP README intro
// bullet "Exact").
//
// One CTA per tile of 128 tokens x 128 experts, K in steps of 64 (three TMA
// stages of x, hi and lo, 128-byte swizzle), accumulator in TMEM; the
// epilogue stages the tile and writes each token's 128 logits with one bulk
// copy.
#include <cuda.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace qmoe {

namespace {

constexpr int TT = 128;   // tokens per tile (MMA M)
constexpr int TE = 128;   // experts per tile (MMA N)
constexpr int BK = 64;    // K per stage
constexpr int NS = 3;     // stages
constexpr int TILE_BYTES = 128 * BK * 2;             // 16 KB per operand tile
constexpr int STAGE_BYTES = 3 * TILE_BYTES;          // x, hi, lo
constexpr int STG_OFF = NS * STAGE_BYTES;            // epilogue staging [TT][TE] f32
constexpr int SMEM = STG_OFF + TT * TE * 4 + 1024;
constexpr int kThreads = 256;                        // warp 0 TMA, warp 1 MMA, warps 4-7 epilogue
constexpr uint64_t kDrainLimit = 2000000000ull;  // 2 s: waits that drain copies and MMAs already issued

// hi = bf16(w), lo = bf16(w - hi), element-wise over the router matrix.
__global__ void __launch_bounds__(256) wsplit_kernel(const float* __restrict__ w, uint16_t* hi, uint16_t* lo, long n) {
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n / 4) return;
  const float4 v = __ldg(reinterpret_cast<const float4*>(w) + i);
  const float f[4] = {v.x, v.y, v.z, v.w};
  uint16_t h[4], l[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    h[j] = float_to_bf16_bits(f[j]);
    l[j] = float_to_bf16_bits(f[j] - bf16_bits_to_float(h[j]));
  }
  reinterpret_cast<uint2*>(hi)[i] = make_uint2(h[0] | (uint32_t)h[1] << 16, h[2] | (uint32_t)h[3] << 16);
  reinterpret_cast<uint2*>(lo)[i] = make_uint2(l[0] | (uint32_t)l[1] << 16, l[2] | (uint32_t)l[3] << 16);
}

__global__ void __launch_bounds__(kThreads, 1) logits_tc_kernel(PrefillArgs a, const __grid_constant__ CUtensorMap tmX,
                                                                const __grid_constant__ CUtensorMap tmHi,
                                                                const __grid_constant__ CUtensorMap tmLo) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[NS], empty[NS], done;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.y * TT, e0 = blockIdx.x * TE;
  const int nst = a.H / BK;
  Ctrl* ctrl = a.rb.ctrl;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      tc::bar_init(&full[i], 1);
      tc::bar_init(&empty[i], 1);
    }
    tc::bar_init(&done, 1);
    tc::bar_init_fence();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_slot, TE);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t issued = 0;
      for (int s = 0; s < nst; ++s) {
        const int st = s % NS;
        if (!tc::bar_wait(&empty[st], ((s / NS) & 1) ^ 1, a.wait_ns)) {
          report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x500);
          break;
        }
        uint8_t* b = smem + st * STAGE_BYTES;
        tc::bar_arrive_expect_tx(&full[st], STAGE_BYTES);
        tc::tma_load_2d(b, &tmX, s * BK, t0, &full[st]);
        tc::tma_load_2d(b + TILE_BYTES, &tmHi, s * BK, e0, &full[st]);
        tc::tma_load_2d(b + 2 * TILE_BYTES, &tmLo, s * BK, e0, &full[st]);
        ++issued;
      }
      // every load issued has landed before the CTA can exit (the MMA warp may have stopped early)
      tc::drain_loads(full, NS, issued, kDrainLimit);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_f16(TT, TE, 1);
      bool ok = true;
      for (int s = 0; s < nst; ++s) {
        const int st = s % NS;
        if (!tc::bar_wait(&full[st], (s / NS) & 1, a.wait_ns)) {
          report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x510);
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t b = tc::smem_u32(smem + st * STAGE_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t da = tc::smem_desc_sw128(b + kk * 32);
          tc::mma_f16(tmem, da, tc::smem_desc_sw128(b + TILE_BYTES + kk * 32), idesc, (s | kk) != 0);
          tc::mma_f16(tmem, da, tc::smem_desc_sw128(b + 2 * TILE_BYTES + kk * 32), idesc, 1);
        }
        tc::commit(&empty[st]);
      }
      (void)ok;
      tc::commit(&done);  // also the drain: every MMA of this CTA completes before TMEM is freed
      tc::bar_wait(&done, 0, kDrainLimit);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // epilogue: lanes = tokens of the tile, columns = experts
    const int q = warp & 3;
    float* stg = reinterpret_cast<float*>(smem + STG_OFF);
    // the four epilogue warps go on together or stop together (no warp left at the barrier below)
    const bool ready = tc::bar_wait(&done, 0, kDrainLimit);
    if (tc::named_all(2, 128, ready)) {
      tc::fence_after_sync();
      const int row = q * 32 + lane;
#pragma unroll 1
      for (int c0 = 0; c0 < TE; c0 += 32) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
        tc::tmem_ld_wait();
        float4* dst = reinterpret_cast<float4*>(stg + (size_t)row * TE + c0);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), __uint_as_float(v[4 * j + 2]),
                               __uint_as_float(v[4 * j + 3]));
      }
      tc::fence_proxy_async();
      tc::named_sync(1, 128);
      if (warp == 4) {
        for (int r = lane; r < TT; r += 32)
          if (t0 + r < a.T)
            tc::bulk_store(a.rb.logits + (size_t)(t0 + r) * a.E + e0, stg + (size_t)r * TE, TE * 4);
        tc::bulk_commit();
        tc::bulk_wait();
      }
    } else {
      report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x520);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TE);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

bool bf16_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, 128};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The tensor-core logits apply when whole 128 x 128 tiles and 64-column
// steps cover the problem; the caller falls back to the FP32 path otherwise.
bool prefill_logits_tc_ok(const PrefillArgs& a) {
  return a.rw_hi && a.E % TE == 0 && a.H % BK == 0 && a.T >= TT;
}

cudaError_t launch_prefill_logits_tc(const PrefillArgs& a, cudaStream_t s) {
  const long n = (long)a.E * a.H;
  wsplit_kernel<<<(unsigned)((n / 4 + 255) / 256), 256, 0, s>>>(a.rw, a.rw_hi, a.rw_lo, n);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  alignas(64) CUtensorMap tx, thi, tlo;
  if (!bf16_map(&tx, a.x, (uint64_t)a.H, (uint64_t)a.T) || !bf16_map(&thi, a.rw_hi, (uint64_t)a.H, (uint64_t)a.E) ||
      !bf16_map(&tlo, a.rw_lo, (uint64_t)a.H, (uint64_t)a.E))
    return cudaErrorInvalidValue;
  if ((err = cudaFuncSetAttribute(logits_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM)) != cudaSuccess)
    return err;
  logits_tc_kernel<<<dim3(a.E / TE, (a.T + TT - 1) / TT), kThreads, SMEM, s>>>(a, tx, thi, tlo);
  return cudaGetLastError();
}

}  // namespace qmoe
