// Prefill expert GEMMs on tcgen05 (exact chain, NVFP4 weights).
//
//   gate/up: for a token tile of one expert and 128 rows of I,
//            G = Wg x^T, U = Wu x^T (two TMEM accumulators), epilogue
//            h = bf16( silu(ts_g G) * (ts_u U) ) per sorted position.
//   down:    for a token tile and 128 rows of H, D = Wd h^T, epilogue
//            P[pair] = ts_d D (FP32 partials, DGPP README "Execution and
//            performance", engine.prefill_bf16_partials off by default).
//
// The MMA is kind::f16 with f16 operands.  Weights are decoded in shared
// memory, never in HBM (DGPP README intro "no dequantized copy"): e2m1 * e4m3
// has at most 6 significant bits and lies in f16's normal range, so the
// decoded operand is exact; the tensor scale multiplies the FP32
// accumulator.  Tokens enter as f16 scaled by a power of two per token (per
// sorted position for h), exact for every element above 2^-31 of the row's
// largest magnitude; the epilogue undoes the scale.  Products are exact in
// FP32 and accumulate in the tensor core's FP32 accumulator.
//
// CTA roles (persistent grid, one CTA per SM):
//   warps 0-7  decode the weight rows of each K step (cp.async ring of raw
//              codes per thread, e2m1/e4m3 conversion to f16) into the
//              stage's A tiles, then run the epilogue from TMEM;
//   warp 8     copies the stage's token rows (B tile) with cp.async and
//              signals their arrival through the stage's mbarrier;
//   warp 9     allocates TMEM and issues the MMAs from one thread;
//              tcgen05.commit releases each stage and publishes each tile.
// Every wait on an mbarrier is bounded; a wait that gives up records
// MOE_ERR_DEVICE_TIMEOUT and the CTA winds down (draining its MMAs before
// TMEM is released).
#include "kernels.cuh"
#include "tc.cuh"

namespace qmoe {

namespace {

constexpr int BM = kPfRowTile;  // weight rows per tile (MMA M)
constexpr int NT = kPfTokTile;  // tokens per tile (MMA N at most)
constexpr int BK = 64;          // K per step (f16: 128 bytes per row)
constexpr int KB = BK * 2;
constexpr int kDec = 256;       // decode / epilogue threads
constexpr int kRaw = 4;         // raw ring stages per decode thread
constexpr int kRawBytes = 48;   // per thread per raw stage
constexpr uint64_t kWaitLimit = 2000000000ull;  // 2 s of global timer per wait

template <bool DOWN>
struct Cfg {
  static constexpr int NMAT = DOWN ? 1 : 2;
  static constexpr int STAGES = DOWN ? 4 : 3;
  static constexpr int TPR = kDec / (NMAT * BM);  // decode threads per weight row
  static constexpr int KT = BK / TPR;             // columns per decode thread per step
  static constexpr int A_BYTES = BM * KB;
  static constexpr int B_BYTES = NT * KB;
  static constexpr int STAGE_BYTES = NMAT * A_BYTES + B_BYTES;
  static constexpr int RAW_OFF = STAGES * STAGE_BYTES;
  static constexpr int SMEM = RAW_OFF + kRaw * kDec * kRawBytes + 1024;
  static constexpr uint32_t TMEM_COLS = 256;
};

__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0));
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

template <bool DOWN>
__global__ void __launch_bounds__(kPfGemmThreads, 1) pf_gemm_kernel(PrefillArgs a) {
  using C = Cfg<DOWN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_a[C::STAGES], full_b[C::STAGES], empty[C::STAGES];
  __shared__ __align__(8) uint64_t acc_full, acc_empty, drain;
  __shared__ uint32_t tmem_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, I = a.I, k = a.k;
  const int K = DOWN ? I : H;          // reduction length
  const int N = DOWN ? H : I;          // rows of one weight matrix
  const int RT = N / BM;               // row tiles per token tile
  const int nsteps = K / BK;
  const int n_items = a.rb.ctrl->n_tiles * RT;
  Ctrl* ctrl = a.rb.ctrl;

  if (tid == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      tc::bar_init(&full_a[i], kDec);
      tc::bar_init(&full_b[i], 32);
      tc::bar_init(&empty[i], 1);
    }
    tc::bar_init(&acc_full, 1);
    tc::bar_init(&acc_empty, kDec);
    tc::bar_init(&drain, 1);
    tc::bar_init_fence();
  }
  if (warp == 9) tc::tmem_alloc(&tmem_slot, C::TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp < 8) {
    // ------------------------------------------------ decode + epilogue --
    const int d = tid;
    const int m = d / (BM * C::TPR);
    const int rr = (d % (BM * C::TPR)) / C::TPR;
    const int hh = d % C::TPR;
    const QW& W = DOWN ? a.down : (m == 0 ? a.gate : a.up);
    uint8_t* raw = smem + C::RAW_OFF + d * kRawBytes;
    uint32_t g = 0;
    bool ok = true;
    int item = 0;
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, ++item) {
      const int2 tile = a.tiles[it / RT];
      const int rt = it % RT, e = tile.x, pos0 = tile.y;
      const int row = rt * BM + rr;
      const uint8_t* crow = W.data + (size_t)e * data_bytes(MOE_FMT_NVFP4, N, K) + (size_t)row * (K / 2);
      const uint8_t* srow = W.scales + (size_t)e * scale_bytes(MOE_FMT_NVFP4, N, K) + (size_t)row * (K / 16);
      auto issue = [&](int s) {
        uint8_t* dst = raw + (s % kRaw) * (kDec * kRawBytes);
        const int k0 = s * BK + hh * C::KT;
        cp_async16(dst, crow + k0 / 2);
        if (C::KT == 64) cp_async16(dst + 16, crow + k0 / 2 + 16);
        cp_async4(dst + 32, srow + (s * BK) / 16);
      };
#pragma unroll 1
      for (int j = 0; j < kRaw - 1; ++j) {
        if (j < nsteps) issue(j);
        cp_async_commit();
      }
#pragma unroll 1
      for (int s = 0; s < nsteps; ++s, ++g) {
        if (s + kRaw - 1 < nsteps) issue(s + kRaw - 1);
        cp_async_commit();
        cp_async_wait<kRaw - 1>();
        const uint8_t* src = raw + (s % kRaw) * (kDec * kRawBytes);
        const uint32_t sw = *reinterpret_cast<const uint32_t*>(src + 32);
        uint4 out[C::KT / 8];
#pragma unroll
        for (int c = 0; c < C::KT / 8; ++c) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(src + 4 * c);
          const uint32_t sc = e4m3_bcast_f16x2(sw >> (8 * (hh * (C::KT / 16) + c / 2)));
          uint32_t v[4];
          e2m1x8_to_f16x2(w, v);
          out[c] = make_uint4(hmul2_u32(v[0], sc), hmul2_u32(v[1], sc), hmul2_u32(v[2], sc), hmul2_u32(v[3], sc));
        }
        const int stage = g % C::STAGES;
        if (!tc::bar_wait(&empty[stage], ((g / C::STAGES) & 1) ^ 1, kWaitLimit)) {
          report_error(ctrl, MOE_ERR_DEVICE_TIMEOUT, 0x300 | (DOWN ? 1 : 0));
          ok = false;
          break;
        }
        uint8_t* A = smem + stage * C::STAGE_BYTES + m * C::A_BYTES;
#pragma unroll
        for (int c = 0; c < C::KT / 8; ++c)
          *reinterpret_cast<uint4*>(A + tc::chunk_off(rr, hh * (C::KT / 8) + c, KB)) = out[c];
        tc::fence_proxy_async();
        tc::bar_arrive(&full_a[stage]);
      }
      cp_async_wait<0>();
      if (!ok) break;

      // ---- epilogue: warp (q, half) reads TMEM lanes 32q.. and half of the columns
      if (!tc::bar_wait(&acc_full, item & 1, kWaitLimit)) {
        report_error(ctrl, MOE_ERR_DEVICE_TIMEOUT, 0x310 | (DOWN ? 1 : 0));
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const int q = warp & 3, half = warp >> 2;
      const int n_valid = min(NT, a.rb.off[e + 1] - pos0);
      const int orow = rt * BM + q * 32 + lane;
      const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int cb = 0; cb < NT / 2; cb += 16) {
        const int c0 = half * (NT / 2) + cb;
        if (c0 >= n_valid) break;
        if (!DOWN) {
          uint32_t gv[16], uv[16];
          tc::tmem_ld16(tq + c0, gv);
          tc::tmem_ld16(tq + NT + c0, uv);
          tc::tmem_ld_wait();
          const float tsg = __ldg(a.gate.ts + e), tsu = __ldg(a.up.ts + e);
#pragma unroll 4
          for (int j = 0; j < 16; ++j) {
            if (c0 + j >= n_valid) break;
            const int pos = pos0 + c0 + j;
            const int tok = a.rb.pair[pos] / k;
            const float un = exp2i(-a.xsig[tok]);
            const float gg = __uint_as_float(gv[j]) * (tsg * un);
            const float uu = __uint_as_float(uv[j]) * (tsu * un);
            const uint16_t hb = float_to_bf16_bits(silu(gg) * uu);
            a.h[(size_t)pos * I + orow] = hb;
            const uint32_t mag = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(hb & 0x7FFF) << 16);
            if (lane == 0 && mag) atomicMax(&a.h_amax[pos], mag);
          }
        } else {
          uint32_t dv[16];
          tc::tmem_ld16(tq + c0, dv);
          tc::tmem_ld_wait();
          const float tsd = __ldg(a.down.ts + e);
#pragma unroll 4
          for (int j = 0; j < 16; ++j) {
            if (c0 + j >= n_valid) break;
            const int pos = pos0 + c0 + j;
            const float un = exp2i(-a.hsig[pos]);
            a.P[(size_t)a.rb.pair[pos] * H + orow] = __uint_as_float(dv[j]) * (tsd * un);
          }
        }
      }
      tc::fence_before_sync();
      tc::bar_arrive(&acc_empty);
    }
  } else if (warp == 8) {
    // --------------------------------------------------------- B loader --
    uint32_t g = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const int2 tile = a.tiles[it / RT];
      const int e = tile.x, pos0 = tile.y;
      const int n_valid = min(NT, a.rb.off[e + 1] - pos0);
      const uint16_t* src[NT / 32];
      bool val[NT / 32];
#pragma unroll
      for (int i = 0; i < NT / 32; ++i) {
        const int r = lane + 32 * i;
        val[i] = r < n_valid;
        const int pos = pos0 + (val[i] ? r : 0);
        src[i] = DOWN ? a.h16 + (size_t)pos * I : a.xs + (size_t)(a.rb.pair[pos] / k) * H;
      }
#pragma unroll 1
      for (int s = 0; s < nsteps; ++s, ++g) {
        const int stage = g % C::STAGES;
        if (!tc::bar_wait(&empty[stage], ((g / C::STAGES) & 1) ^ 1, kWaitLimit)) {
          report_error(ctrl, MOE_ERR_DEVICE_TIMEOUT, 0x320 | (DOWN ? 1 : 0));
          ok = false;
          break;
        }
        uint8_t* B = smem + stage * C::STAGE_BYTES + C::NMAT * C::A_BYTES;
#pragma unroll
        for (int i = 0; i < NT / 32; ++i) {
          if (!val[i]) continue;  // rows past the tile's tokens only feed discarded columns
          const int r = lane + 32 * i;
#pragma unroll
          for (int c = 0; c < 8; ++c) cp_async16_zfill(B + tc::chunk_off(r, c, KB), src[i] + s * BK + c * 8, true);
        }
        cp_async_arrive_noinc(&full_b[stage]);
      }
    }
    cp_async_wait<0>();
  } else {
    // -------------------------------------------------------------- MMA --
    if (lane == 0) {
      uint32_t g = 0;
      int item = 0;
      bool ok = true;
      for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, ++item) {
        const int2 tile = a.tiles[it / RT];
        const int n_valid = min(NT, a.rb.off[tile.x + 1] - tile.y);
        const int n_mma = (n_valid + 15) & ~15;
        const uint32_t idesc = tc::idesc_f16(BM, n_mma, 0);
        if (!tc::bar_wait(&acc_empty, (item & 1) ^ 1, kWaitLimit)) {
          report_error(ctrl, MOE_ERR_DEVICE_TIMEOUT, 0x330 | (DOWN ? 1 : 0));
          break;
        }
        tc::fence_after_sync();
#pragma unroll 1
        for (int s = 0; s < nsteps; ++s, ++g) {
          const int stage = g % C::STAGES;
          const uint32_t par = (g / C::STAGES) & 1;
          if (!tc::bar_wait(&full_a[stage], par, kWaitLimit) || !tc::bar_wait(&full_b[stage], par, kWaitLimit)) {
            report_error(ctrl, MOE_ERR_DEVICE_TIMEOUT, 0x340 | (DOWN ? 1 : 0));
            ok = false;
            break;
          }
          tc::fence_after_sync();
          tc::fence_proxy_async();
          const uint32_t base = tc::smem_u32(smem + stage * C::STAGE_BYTES);
          const uint32_t bB = base + C::NMAT * C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t db = tc::smem_desc(bB + kk * 256, 128, 1024);
#pragma unroll
            for (int mm = 0; mm < C::NMAT; ++mm) {
              const uint64_t da = tc::smem_desc(base + mm * C::A_BYTES + kk * 256, 128, 1024);
              tc::mma_f16(tmem + mm * NT, da, db, idesc, (s | kk) != 0);
            }
          }
          tc::commit(&empty[stage]);
        }
        if (!ok) break;
        tc::commit(&acc_full);
      }
      tc::commit(&drain);
      tc::bar_wait(&drain, 0, kWaitLimit);
    }
    __syncwarp();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace

size_t prefill_gemm_smem(bool down) { return down ? Cfg<true>::SMEM : Cfg<false>::SMEM; }

cudaError_t launch_prefill_gemm_nvfp4(bool down, const PrefillArgs& a, int grid, cudaStream_t s) {
  cudaError_t err;
  if (down) {
    err = cudaFuncSetAttribute(pf_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<true>::SMEM);
    if (err != cudaSuccess) return err;
    pf_gemm_kernel<true><<<grid, kPfGemmThreads, Cfg<true>::SMEM, s>>>(a);
  } else {
    err = cudaFuncSetAttribute(pf_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<false>::SMEM);
    if (err != cudaSuccess) return err;
    pf_gemm_kernel<false><<<grid, kPfGemmThreads, Cfg<false>::SMEM, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace qmoe
