// Prefill expert GEMMs, W4A4 lever (block-scaled FP4 tensor cores): NVFP4
// weights with NVFP4 activations, or MXFP4 weights with MXFP4 activations.
//
// The activation lever of the DGPP README ("Highlights", the W4A4 lever; the
// levers are explicit and off by default): the token rows x and h are
// quantised to NVFP4 (16-element blocks, E4M3 block scale, tensor scale 1)
// and both operands of each projection are FP4.  tcgen05.mma
// kind::mxf4nvf4 (scale_vec::4X) multiplies the packed E2M1 codes and
// applies the two UE4M3 block scales in hardware; the weights' FP32 tensor
// scale multiplies the FP32 accumulator in the epilogue.  For MXFP4 weights
// the activations are MXFP4 (32-element blocks, E8M0 scale) and the MMA is the
// same kind with scale_vec::2X and UE8M0 scales.
//
//   gate/up: G = Wg x^T, U = Wu x^T per (token tile, 128 rows of I);
//            h = bf16( silu(ts_g G) * (ts_u U) ), re-quantised to NVFP4 per
//            16 rows of I in the epilogue (the operand of the down GEMM): h is
//            staged first so the TMEM accumulator is released early.
//   down:    P[pos] = ts_d (Wd h^T), FP32 partials by sorted position.
//
// Operands: packed codes as 2-D TMA boxes of 128 rows x 128 bytes (256 K),
// 128-byte swizzle, three stages.  Block scales go to TMEM: for every K=64
// MMA, 4 columns per operand, where lane l of every quadrant, column c,
// holds the scale bytes of row (l mod 32) + 32 c for that MMA's K range:
// four UE4M3 bytes (NVFP4), or two UE8M0 bytes in the low half (MXFP4).
//
// CTA roles (persistent grid, one CTA per SM):
//   warp 0       TMA producer (weights and token codes);
//   warp 1       TMEM allocation and MMA issue (the whole warp runs the loop, one elected lane issues);
//   warps 4-7    scale writers: load the stage's block scales, tcgen05.st
//                them into the stage's TMEM scale slot (one quadrant each);
//   warps 8-15   epilogue (two warps per TMEM lane quadrant).
// Every mbarrier wait is bounded (MOE_ERR_DEVICE_TIMEOUT).
#include <cuda.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace qmoe {

namespace {

constexpr int BM = kPfRowTile;
constexpr int NT = kPfTokTile;
constexpr int KS = 256;        // K per stage
constexpr int KSB = KS / 2;    // bytes of codes per row per stage
constexpr int ST = 3;          // stages
constexpr uint64_t kDrainLimit = 2000000000ull;  // 2 s: waits that drain copies and MMAs already issued
constexpr int kThreads = 512;
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpSf0 = 4, kWarpEpi0 = 8;
constexpr int kEpiThreads = 256;

template <bool DOWN>
struct Cw {
  static constexpr int NMAT = DOWN ? 1 : 2;
  static constexpr int A_BYTES = BM * KSB;
  static constexpr int B_BYTES = NT * KSB;
  static constexpr int STAGE = NMAT * A_BYTES + B_BYTES;
  static constexpr int STG_OFF = ST * STAGE;
  // down: P tile f32 [NT][BM]; gate/up: h tile bf16 [NT][BM], then its codes [NT][BM / 2]
  static constexpr int STG_BYTES = DOWN ? NT * BM * 4 : NT * BM * 2 + NT * (BM / 2);
  static constexpr int SMEM = STG_OFF + STG_BYTES + 1024;
  static constexpr int ACC_BUFS = DOWN ? 2 : 1;
  static constexpr uint32_t ACC_COLS = NMAT * NT;
  static constexpr uint32_t SF_BASE = ACC_BUFS * ACC_COLS;
  static constexpr uint32_t SF_STAGE = (NMAT + 1) * 16;  // 4 MMAs x 4 columns per operand
  static_assert(SF_BASE + ST * SF_STAGE <= 512, "TMEM columns");
};

// Instruction descriptor of kind::mxf4nvf4: E2M1 A and B, K-major operands,
// M = 128; bit 23 selects UE8M0 scales (MXFP4) instead of UE4M3 (NVFP4).
template <bool MX>
__device__ __forceinline__ uint32_t idesc_f4(int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (MX ? (1u << 23) : 0u) | ((uint32_t)(BM >> 4) << 24);
}

// Issued from a converged warp: every lane holds the same operands, one elected
// lane issues (its commits, tc::commit_elect, track these MMAs).
template <bool MX>
__device__ __forceinline__ void mma_f4(uint32_t d, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
  if constexpr (MX) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
            "r"(d),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate));
  } else {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
            "r"(d),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate));
  }
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]));
}

__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + expf(-z)); }

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t h = e4m3_bcast_f16x2(code);
  return __low2float(*reinterpret_cast<const __half2*>(&h));
}

// Block scales of rows row0 + lane + 32 c (c < 4) for one 256-K stage, word kk
// = the scales of MMA kk -> v[4 kk + c].  NVFP4: 16 bytes per row, four per
// word; MXFP4: 8 bytes per row, two per word (low half).
template <bool MX>
__device__ __forceinline__ void load_scales(const uint8_t* base, size_t row_stride, int row0, int lane, int row_lim,
                                            int stage_off, uint32_t (&v)[16]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int r = row0 + lane + 32 * c;
    if constexpr (MX) {
      uint2 w = make_uint2(0, 0);
      if (r < row_lim) w = __ldg(reinterpret_cast<const uint2*>(base + (size_t)r * row_stride + stage_off));
      v[c] = w.x & 0xFFFFu;
      v[4 + c] = w.x >> 16;
      v[8 + c] = w.y & 0xFFFFu;
      v[12 + c] = w.y >> 16;
    } else {
      uint4 w = make_uint4(0, 0, 0, 0);
      if (r < row_lim) w = __ldg(reinterpret_cast<const uint4*>(base + (size_t)r * row_stride + stage_off));
      v[c] = w.x;
      v[4 + c] = w.y;
      v[8 + c] = w.z;
      v[12 + c] = w.w;
    }
  }
}

template <bool DOWN, bool MX>
__global__ void __launch_bounds__(kThreads, 1) pf_w4a4_kernel(PrefillArgs a, const __grid_constant__ CUtensorMap tmA0,
                                                              const __grid_constant__ CUtensorMap tmA1,
                                                              const __grid_constant__ CUtensorMap tmB) {
  using C = Cw<DOWN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[ST], sf_full[ST], empty[ST], acc_full[2], acc_empty[2], drain;
  __shared__ uint32_t tmem_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, I = a.I;
  const int K = DOWN ? I : H;
  const int N = DOWN ? H : I;
  const int RT = N / BM;
  const int nst = K / KS;
  const int P = a.T * a.k;
  const int n_items = a.rb.ctrl->n_tiles * RT;
  Ctrl* ctrl = a.rb.ctrl;

  if (tid == 0) {
    for (int i = 0; i < ST; ++i) {
      tc::bar_init(&full[i], 1);
      tc::bar_init(&sf_full[i], 128);
      tc::bar_init(&empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::bar_init(&acc_full[b], 1);
      tc::bar_init(&acc_empty[b], kEpiThreads);
    }
    tc::bar_init(&drain, 1);
    tc::bar_init_fence();
  }
  if (warp == kWarpMma) tc::tmem_alloc(&tmem_slot, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp == kWarpTma) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      uint32_t g = 0;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const int2 tile = a.tiles[it / RT];
        const int rt = it % RT, e = tile.x, pos0 = tile.y;
        const int rowA = e * N + rt * BM;
        bool ok = true;
        for (int s = 0; s < nst; ++s, ++g) {
          const int stage = g % ST;
          if (!tc::bar_wait(&empty[stage], ((g / ST) & 1) ^ 1, a.wait_ns)) {
            report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x400 | (DOWN ? 1 : 0));
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * C::STAGE;
          tc::bar_arrive_expect_tx(&full[stage], C::STAGE);
          tc::tma_load_2d(st, &tmA0, s * KSB, rowA, &full[stage]);
          if (!DOWN) tc::tma_load_2d(st + C::A_BYTES, &tmA1, s * KSB, rowA, &full[stage]);
          tc::tma_load_2d(st + C::NMAT * C::A_BYTES, &tmB, s * KSB, pos0, &full[stage]);
        }
        if (!ok) break;
      }
      // every load issued has landed before the CTA can exit (the MMA warp may have stopped early)
      tc::drain_loads(full, ST, g, kDrainLimit);
    }
    __syncwarp();
  } else if (warp >= kWarpSf0 && warp < kWarpSf0 + 4) {
    // ---------------------------------------------------- scale writers --
    const int q = warp & 3;
    const uint32_t lq = (uint32_t)(q * 32) << 16;
    const int Kb = K / (MX ? 32 : 16);  // scale bytes per row
    constexpr int kStageSf = KS / (MX ? 32 : 16);  // scale bytes per row per stage
    const uint8_t* sfb_base = DOWN ? a.hsf : a.xsfg;
    uint32_t g = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
      const int2 tile = a.tiles[it / RT];
      const int rt = it % RT, e = tile.x, pos0 = tile.y;
      bool ok = true;
      for (int s = 0; s < nst; ++s, ++g) {
        const int stage = g % ST;
        // the scales do not depend on the slot: load them before waiting for it
        uint32_t v[C::NMAT + 1][16];
#pragma unroll
        for (int m = 0; m < C::NMAT; ++m) {
          const QW& W = DOWN ? a.down : (m == 0 ? a.gate : a.up);
          load_scales<MX>(W.scales + (size_t)e * N * Kb, Kb, rt * BM, lane, N, s * kStageSf, v[m]);
        }
        load_scales<MX>(sfb_base, Kb, pos0, lane, P, s * kStageSf, v[C::NMAT]);
        if (!tc::bar_wait(&empty[stage], ((g / ST) & 1) ^ 1, a.wait_ns)) {
          report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x410 | (DOWN ? 1 : 0));
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t col = tmem + lq + C::SF_BASE + stage * C::SF_STAGE;
#pragma unroll
        for (int m = 0; m <= C::NMAT; ++m) tmem_st16(col + m * 16, v[m]);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc::fence_before_sync();
        tc::bar_arrive(&sf_full[stage]);
      }
      if (!ok) break;
    }
  } else if (warp == kWarpMma) {
    // -------------------------------------------------------------- MMA --
    // The whole warp runs this loop (values warp-uniform, branches taken by
    // all lanes); one elected lane issues each MMA and commit.
    uint32_t g = 0;
    int item = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, ++item) {
      const int2 tile = a.tiles[it / RT];
      const int n_valid = min(NT, a.rb.off[tile.x + 1] - tile.y);
      const uint32_t idesc = idesc_f4<MX>((n_valid + 15) & ~15);
      const int buf = DOWN ? (item & 1) : 0, use = DOWN ? (item >> 1) : item;
      if (!__all_sync(0xFFFFFFFFu, tc::bar_wait(&acc_empty[buf], (use & 1) ^ 1, a.wait_ns))) {
        if (lane == 0) report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x420 | (DOWN ? 1 : 0));
        break;
      }
      tc::fence_after_sync();
      const uint32_t acc = tmem + buf * C::ACC_COLS;
      for (int s = 0; s < nst; ++s, ++g) {
        const int stage = g % ST;
        const uint32_t par = (g / ST) & 1;
        const bool ready = tc::bar_wait(&full[stage], par, a.wait_ns) && tc::bar_wait(&sf_full[stage], par, a.wait_ns);
        if (!__all_sync(0xFFFFFFFFu, ready)) {
          if (lane == 0) report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x430 | (DOWN ? 1 : 0));
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t base = tc::smem_u32(smem + stage * C::STAGE);
        const uint32_t bB = base + C::NMAT * C::A_BYTES;
        const uint32_t sf = tmem + C::SF_BASE + stage * C::SF_STAGE;
#pragma unroll
        for (int kk = 0; kk < KS / 64; ++kk) {
          const uint64_t db = tc::smem_desc_sw128(bB + kk * 32);
#pragma unroll
          for (int m = 0; m < C::NMAT; ++m) {
            const uint64_t da = tc::smem_desc_sw128(base + m * C::A_BYTES + kk * 32);
            mma_f4<MX>(acc + m * NT, da, db, idesc, sf + m * 16 + kk * 4, sf + C::NMAT * 16 + kk * 4, (s | kk) != 0);
          }
        }
        tc::commit_elect(&empty[stage]);
      }
      if (!ok) break;
      tc::commit_elect(&acc_full[buf]);
    }
    tc::commit_elect(&drain);
    tc::bar_wait(&drain, 0, kDrainLimit);
    __syncwarp();
  } else if (warp >= kWarpEpi0) {
    // --------------------------------------------------------- epilogue --
    const int ew = warp - kWarpEpi0;
    const int q = warp & 3, chalf = ew >> 2;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    uint8_t* stg = smem + C::STG_OFF;
    int item = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++item) {
      const int2 tile = a.tiles[it / RT];
      const int rt = it % RT, e = tile.x, pos0 = tile.y;
      const int n_valid = min(NT, a.rb.off[e + 1] - pos0);
      const int buf = DOWN ? (item & 1) : 0, use = DOWN ? (item >> 1) : item;
      // the NVFP4 tensor scales (MXFP4 has none)
      const float ts0 = MX ? 1.f : __ldg((DOWN ? a.down.ts : a.gate.ts) + e);
      const float ts1 = (DOWN || MX) ? 1.f : __ldg(a.up.ts + e);
      const bool ready = tc::bar_wait(&acc_full[buf], use & 1, a.wait_ns);
      if (!ready) report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x440 | (DOWN ? 1 : 0));
      // all epilogue warps go on, or all stop; the barrier also frees the staging tile
      if (!tc::named_all(1, kEpiThreads, ready)) break;
      tc::fence_after_sync();
      const uint32_t acc = tq + buf * C::ACC_COLS;
      const int row = q * 32 + lane;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int c0 = chalf * 64 + i * 32;
        if (c0 >= n_valid) break;
        const int ncol = min(32, n_valid - c0);
        if (!DOWN) {
          // phase 1: h = bf16(silu(ts_g G) * (ts_u U)) into the staging tile [column][row]
          uint32_t gv[32], uv[32];
          tc::tmem_ld32(acc + c0, gv);
          tc::tmem_ld32(acc + NT + c0, uv);
          tc::tmem_ld_wait();
          uint16_t* st16 = reinterpret_cast<uint16_t*>(stg) + (size_t)c0 * BM + row;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < ncol)
              st16[j * BM] = float_to_bf16_bits(silu(__uint_as_float(gv[j]) * ts0) * (__uint_as_float(uv[j]) * ts1));
        } else {
          uint32_t dv[32];
          tc::tmem_ld32(acc + c0, dv);
          tc::tmem_ld_wait();
          // P straight from registers: per column the warp's 32 lanes write 32 consecutive rows
          float* p32 = a.P + (size_t)(pos0 + c0) * H + rt * BM + row;
          uint16_t* p16 = reinterpret_cast<uint16_t*>(a.P) + (size_t)(pos0 + c0) * H + rt * BM + row;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < ncol) {
              const float v = __uint_as_float(dv[j]) * ts0;
              if (a.p_bf16) p16[(size_t)j * H] = float_to_bf16_bits(v);
              else p32[(size_t)j * H] = v;
            }
        }
      }
      tc::fence_before_sync();
      tc::bar_arrive(&acc_empty[buf]);  // TMEM buffer free for the MMA of a later tile
      if (!DOWN && MX) {
        // phase 2: MXFP4 of h per (column, 32-row block), the MXFP4 activation rule: the
        // smallest e with 6 * 2^e >= amax, codes e2m1(h * 2^-e)
        tc::named_sync(1, kEpiThreads);
        const uint16_t* hs = reinterpret_cast<const uint16_t*>(stg);
        uint8_t* cs = stg + NT * BM * 2;
        const int et = tid - kWarpEpi0 * 32;
        for (int u = et; u < n_valid * (BM / 32); u += kEpiThreads) {
          const int c = u / (BM / 32), b = u % (BM / 32);
          const uint4* src = reinterpret_cast<const uint4*>(hs + (size_t)c * BM + b * 32);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 v = src[i];
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
          }
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_float(w[i] & 0xFFFF)), fabsf(bf16_bits_to_float(w[i] >> 16))));
          const int sc = mxfp4_act_scale_code(amax);
          const float inv = exp2i(127 - sc);
          uint32_t out[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int i = 0; i < 16; ++i)
            out[i >> 2] |= f32x2_to_e2m1x2_sat(bf16_bits_to_float(w[i] & 0xFFFF) * inv,
                                               bf16_bits_to_float(w[i] >> 16) * inv) << (8 * (i & 3));
          *reinterpret_cast<uint4*>(cs + c * (BM / 2) + b * 16) = make_uint4(out[0], out[1], out[2], out[3]);
          a.hsf[(size_t)(pos0 + c) * (I / 32) + rt * (BM / 32) + b] = (uint8_t)sc;
        }
      } else if (!DOWN) {
        // phase 2: NVFP4 of h per (column, 16-row block), the activation quantiser's
        // rule: scale e4m3(amax / 6), codes e2m1(h / scale)
        tc::named_sync(1, kEpiThreads);
        const uint16_t* hs = reinterpret_cast<const uint16_t*>(stg);
        uint8_t* cs = stg + NT * BM * 2;
        const int et = tid - kWarpEpi0 * 32;
        for (int u = et; u < n_valid * (BM / 16); u += kEpiThreads) {
          const int c = u / (BM / 16), b = u % (BM / 16);
          const uint4* src = reinterpret_cast<const uint4*>(hs + (size_t)c * BM + b * 16);
          const uint4 v0 = src[0], v1 = src[1];
          const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          float hv[16];
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            hv[2 * i] = bf16_bits_to_float(w[i] & 0xFFFF);
            hv[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
            amax = fmaxf(amax, fmaxf(fabsf(hv[2 * i]), fabsf(hv[2 * i + 1])));
          }
          const uint32_t sc = f32_to_e4m3_sat(__fdiv_rn(amax, 6.0f));
          const float sv = e4m3_value(sc);
          uint32_t out[2] = {0u, 0u};
          if (sv > 0.f) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              out[i >> 2] |= f32x2_to_e2m1x2_sat(__fdiv_rn(hv[2 * i], sv), __fdiv_rn(hv[2 * i + 1], sv)) << (8 * (i & 3));
          }
          *reinterpret_cast<uint2*>(cs + c * (BM / 2) + b * 8) = make_uint2(out[0], out[1]);
          a.hsf[(size_t)(pos0 + c) * (I / 16) + rt * (BM / 16) + b] = (uint8_t)sc;
        }
      }
      if constexpr (!DOWN) {
        // the h codes leave through the staging tile: one bulk copy per column
        tc::fence_proxy_async();  // staging writes -> bulk copy reads
        tc::named_sync(1, kEpiThreads);
        if (ew == 0) {
          for (int c = lane; c < n_valid; c += 32)
            tc::bulk_store(a.hq + (size_t)(pos0 + c) * (I / 2) + rt * (BM / 2), stg + NT * BM * 2 + c * (BM / 2),
                           BM / 2);
          tc::bulk_commit();
          tc::bulk_wait_read();
        }
      }
    }
    if (ew == 0) tc::bulk_wait();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
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

// Byte matrix [rows, cols] (row-major): boxes of 128 bytes x 128 rows,
// 128-byte swizzle, zero fill outside the matrix.
bool u8_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {(cuuint32_t)KSB, (cuuint32_t)BM};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

template <bool MX>
cudaError_t launch_w4a4(bool down, const PrefillArgs& a, int grid, cudaStream_t s) {
  alignas(64) CUtensorMap tA0, tA1, tB;
  const uint64_t P = (uint64_t)a.T * a.k;
  cudaError_t err;
  if (down) {
    if (!u8_map(&tA0, a.down.data, (uint64_t)a.I / 2, (uint64_t)a.E * a.H) ||
        !u8_map(&tB, a.hq, (uint64_t)a.I / 2, P))
      return cudaErrorInvalidValue;
    tA1 = tA0;
    err = cudaFuncSetAttribute(pf_w4a4_kernel<true, MX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cw<true>::SMEM);
    if (err != cudaSuccess) return err;
    pf_w4a4_kernel<true, MX><<<grid, kThreads, Cw<true>::SMEM, s>>>(a, tA0, tA1, tB);
  } else {
    if (!u8_map(&tA0, a.gate.data, (uint64_t)a.H / 2, (uint64_t)a.E * a.I) ||
        !u8_map(&tA1, a.up.data, (uint64_t)a.H / 2, (uint64_t)a.E * a.I) ||
        !u8_map(&tB, a.xqg, (uint64_t)a.H / 2, P))
      return cudaErrorInvalidValue;
    err = cudaFuncSetAttribute(pf_w4a4_kernel<false, MX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cw<false>::SMEM);
    if (err != cudaSuccess) return err;
    pf_w4a4_kernel<false, MX><<<grid, kThreads, Cw<false>::SMEM, s>>>(a, tA0, tA1, tB);
  }
  return cudaGetLastError();
}

cudaError_t launch_prefill_gemm_w4a4(bool down, const PrefillArgs& a, int grid, cudaStream_t s) {
  return a.act_quant == 2 ? launch_w4a4<true>(down, a, grid, s) : launch_w4a4<false>(down, a, grid, s);
}

}  // namespace qmoe
