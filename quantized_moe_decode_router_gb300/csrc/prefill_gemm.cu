// Prefill expert GEMMs on tcgen05 (exact chain; NVFP4, MXFP4 or int4 g64 weights).
//
//   gate/up: for a token tile of one expert and 128 rows of I,
//            G = Wg x^T, U = Wu x^T (two TMEM accumulators), epilogue
//            h = bf16( silu(ts_g G) * (ts_u U) ) per sorted position.
//   down:    for a token tile and 128 rows of H, D = Wd h^T, epilogue
//            P[pos] = ts_d D (FP32 partials by sorted position, DGPP README
//            "Execution and performance", engine.prefill_bf16_partials off
//            by default).
//
// The MMA is kind::f16 with f16 operands.  Weights are decoded in shared
// memory, never in HBM (DGPP README intro "no dequantized copy"): each code
// times its block scale, taken relative to a per-row factor, is folded into
// one f16 (exact for NVFP4; for MXFP4 and int4 g64 while the row's block
// scales span at most 2^23 / 2^24, see the fold below); the row factor (the
// NVFP4 tensor scale, else the row's largest block scale) multiplies the FP32
// accumulator.  Tokens enter as f16 scaled by a power of two per token (per
// sorted position for h), exact for every element above 2^-31 of the row's
// largest magnitude; the epilogue undoes the scale.  Products are exact in
// FP32 and accumulate in the tensor core's FP32 accumulator.
//
// CTA roles (persistent grid, one CTA per SM):
//   warps 0-7  decode the weight rows of each K step (cp.async ring of raw
//              codes per thread, conversion to f16) into the stage's A
//              tiles, stored in the 128-byte swizzled K-major layout (the
//              layout of the TMA-loaded B tiles; conflict-free both ways);
//   warp 8     loads the stage's token rows (B tile) with one 2-D TMA box
//              (128-byte swizzle) of the position-sorted operand rows
//              (scaled activations for gate/up, h for down); the stage's
//              mbarrier counts the bytes;
//   warp 9     allocates TMEM and issues the MMAs (the whole warp runs the
//              loop, one elected lane issues);
//              tcgen05.commit releases each stage and publishes each tile;
//   warps 10-17 the epilogue, from TMEM accumulators that are double
//              buffered so the next tile's MMAs overlap it; h is staged in
//              shared memory and written with bulk copies, P is stored from
//              registers (coalesced: a warp's lanes hold consecutive rows);
//              both by sorted position.
// Every wait on an mbarrier is bounded; a wait that gives up records
// MOE_ERR_DEVICE_TIMEOUT and the CTA winds down (draining its MMAs before
// TMEM is released).
#include <cuda.h>

#include "kernels.cuh"
#include "tc.cuh"

namespace qmoe {

namespace {

constexpr int BM = kPfRowTile;  // weight rows per tile (MMA M)
constexpr int NT = kPfTokTile;  // tokens per tile (MMA N at most)
constexpr int BK = 64;          // K per step (f16: 128 bytes per row)
constexpr int KB = BK * 2;
constexpr int kDec = 256;       // decode threads (8 warps)
constexpr uint64_t kDrainLimit = 2000000000ull;  // 2 s: waits that drain copies and MMAs already issued

// Formats whose block scale does not fold exactly into an f16 weight (an 8-bit
// code or a 4-bit code times an 11-bit FP16 scale): their codes enter the MMA
// as exact f16 integers / E4M3 values, each scale group's products accumulate
// in a TMEM block of their own, and the epilogue adds scale x block to a
// running FP32 sum (the group scale applied per group, in FP32).
template <int F>
constexpr bool promote_fmt() {
  return F == MOE_FMT_INT8_G64 || F == MOE_FMT_FP8_B128 || F == MOE_FMT_INT4_G128;
}

// LV selects a lever.  1, fold scales (promote formats): each code times its
// group scale is rounded to one BF16 weight (FP32 product, then BF16), the
// tokens enter as plain BF16, one FP32 accumulator runs across K.  2, FP8
// activations (FP8 b128): the E4M3 weight codes and per-token 1x128 E4M3
// activation codes meet on kind::f8f6f4 MMAs (K = 128 per step, one step per
// scale group), the weight and activation scales applied per group in FP32.
template <int F, bool DOWN, int LV = 0>
struct Cfg {
  static constexpr bool FS = LV == 1;
  static constexpr bool F8 = LV == 2;
  static_assert(!FS || promote_fmt<F>(), "the fold-scales lever applies to the promote formats");
  static_assert(!F8 || F == MOE_FMT_FP8_B128, "the FP8-activation lever applies to FP8 b128 weights");
  static constexpr bool PROMOTE = promote_fmt<F>() && !FS;
  static constexpr int BITS = (F == MOE_FMT_INT8_G64 || F == MOE_FMT_FP8_B128) ? 8 : 4;
  static constexpr int KSTEP = F8 ? 128 : BK;   // K per step (128 bytes of an A row either way)
  static constexpr int GS = (F8 || F == MOE_FMT_INT8_G64) ? 1 : 2;  // K steps per scale group (promote)
  static constexpr int NMAT = DOWN ? 1 : 2;
  static constexpr int SA = F8 ? 4 : 2;         // A stages (F8: copied straight in, no raw ring)
  static constexpr int SB = 4;                  // token-row (B) stages: TMA latency spans several steps
  static constexpr int TPR = kDec / (NMAT * BM);  // decode threads per weight row
  static constexpr int KT = KSTEP / TPR;          // columns per decode thread per step
  static constexpr int CODE_BYTES = KT * BITS / 8;               // per thread per step
  // fold: the codes, then the step's scale word (padded); promote and FS: the codes only
  static constexpr int RAW_BYTES = (PROMOTE || FS) ? CODE_BYTES : CODE_BYTES + 16;
  static constexpr int RAW = F8 ? 0 : (DOWN ? 6 : (BITS == 8 ? 4 : 5));  // raw-code ring stages (prefetch RAW - 1)
  static constexpr int A_BYTES = BM * KB;
  static constexpr int B_BYTES = NT * KB;
  static constexpr int A_STAGE = NMAT * A_BYTES;
  static constexpr int B_OFF = SA * A_STAGE;
  static constexpr int RAW_OFF = B_OFF + SB * B_BYTES;
  static constexpr int STG_OFF = RAW_OFF + RAW * kDec * RAW_BYTES;  // epilogue staging [NT cols][BM rows]
  static constexpr int OUT_BYTES = DOWN ? 4 : 2;                      // f32 partials / bf16 h
  static constexpr int SMEM = STG_OFF + NT * BM * OUT_BYTES + 1024;
  static constexpr uint32_t ACC_COLS = NMAT * NT;      // one accumulator set
  // fold: two accumulator sets (double buffered); promote: running sums, then the group block
  static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(CODE_BYTES % 16 == 0, "16-byte code copies");
};

// Warp roles.
constexpr int kWarpLoader = kDec / 32;       // 8
constexpr int kWarpMma = kWarpLoader + 1;    // 9
constexpr int kWarpEpi0 = kWarpMma + 1;      // 10..17: epilogue, warp w reads TMEM lanes 32 * (w % 4)
constexpr int kEpiWarps = 8;                 // two per TMEM lane quarter, each half of the columns
constexpr int kEpiThreads = kEpiWarps * 32;
static_assert(kWarpEpi0 * 32 + kEpiThreads == kPfGemmThreads, "warp roles");

// SiLU in FP32 (z / (1 + e^-z)); the quotient to within 2 ulp.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + expf(-z)); }

// ---- 4-bit formats: the weights of a row folded exactly into f16 ----------
// NVFP4: e2m1 * e4m3 (at most 6 significant bits, f16-normal), the row factor
// is the tensor scale.  MXFP4: e2m1 * 2^(c - cref), cref the row's largest
// scale code; the row factor 2^(cref - 127) goes to the epilogue.  int4 g64:
// q * M * 2^(e - eref) with the BF16 scale written M * 2^e (M an 8-bit
// integer, |q * M| <= 2040 fits f16's 11-bit significand), eref the row's
// largest exponent; row factor 2^eref.  The fold is exact while a block's
// scale lies within 2^-23 (MXFP4) / 2^-24 (int4) of the row's largest scale.
// A block exactly 2^-24 below (MXFP4) has its products rounded to f16's
// subnormal grid, and blocks further below are dropped: every weight so
// changed is below 2^-21 times the row's largest block scale (MXFP4: 6 *
// 2^-24; int4: 2040 * 2^-25 against a scale of at least 128 * 2^eref), an
// error far inside the output tolerance.

// Byte offset, within a row's scales, of the scales of K step s (BK = 64 columns).
template <int F>
__device__ __forceinline__ int step_scale_off(int s) {
  if constexpr (F == MOE_FMT_NVFP4) return s * (BK / 16);
  else return s * 2;  // MXFP4: two E8M0 codes; int4 g64: one BF16 scale
}

template <int F>
__device__ __forceinline__ size_t row_scale_bytes(int K) {
  if constexpr (F == MOE_FMT_NVFP4) return (size_t)K / 16;
  else if constexpr (F == MOE_FMT_MXFP4) return (size_t)K / 32;
  else return (size_t)K / 64 * 2;
}

// Reference exponent of a row (MXFP4: largest code; int4: largest scale exponent, -100000 if all zero).
template <int F>
__device__ __forceinline__ int row_ref(const uint8_t* srow, int K) {
  if constexpr (F == MOE_FMT_NVFP4) {
    return 0;
  } else {
    // a row's scales: K / 32 bytes (MXFP4) or K / 32 bytes of BF16 (int4 g64), a multiple of 4 bytes
    // at a 4-byte aligned address for K a multiple of 128
    const int nw = (int)(row_scale_bytes<F>(K) / 4);
    int ref = F == MOE_FMT_MXFP4 ? 0 : -100000;
#pragma unroll 4
    for (int i = 0; i < nw; ++i) {
      const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(srow) + i);
      if constexpr (F == MOE_FMT_MXFP4) {
#pragma unroll
        for (int b = 0; b < 4; ++b) ref = max(ref, (int)((w >> (8 * b)) & 0xFF));
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t sb = (w >> (16 * h)) & 0xFFFF;
          const uint32_t E8 = (sb >> 7) & 0xFF;
          if ((sb & 0x7FFF) != 0) ref = max(ref, (E8 ? (int)E8 : 1) - 134);
        }
      }
    }
    return ref;
  }
}

// The row's factor applied to its FP32 accumulator.
template <int F>
__device__ __forceinline__ float row_factor(int ref, float ts) {
  if constexpr (F == MOE_FMT_NVFP4) return ts;
  else if constexpr (F == MOE_FMT_MXFP4) return e8m0_to_float((uint32_t)ref);
  else return ref < -1000 ? 0.f : ldexpf(1.0f, ref);
}

// f16 of 2^d for d <= 0 (normal from -14, subnormal down to -24, 0 below).
__device__ __forceinline__ uint32_t f16_pow2_bits(int d) {
  return d >= -14 ? (uint32_t)(d + 15) << 10 : d >= -24 ? 1u << (d + 24) : 0u;
}

// Eight codes of one 32-bit word (k ascending) folded into four f16x2; sbits: the
// scale bits covering them (NVFP4: one E4M3 byte, MXFP4: one E8M0 byte, int4: one BF16).
template <int F>
__device__ __forceinline__ uint4 fold_word(uint32_t w, uint32_t sbits, int ref) {
  uint32_t v[4];
  uint32_t fac;
  if constexpr (F == MOE_FMT_INT4_G64) {
    uint32_t p[4];
    int4x8_to_f16x2_paired(w, p);                                    // (k0,k4) (k1,k5) (k2,k6) (k3,k7)
    v[0] = prmt(p[0], p[1], 0x5410u);                                 // (k0,k1)
    v[1] = prmt(p[2], p[3], 0x5410u);                                 // (k2,k3)
    v[2] = prmt(p[0], p[1], 0x7632u);                                 // (k4,k5)
    v[3] = prmt(p[2], p[3], 0x7632u);                                 // (k6,k7)
    const uint32_t E8 = (sbits >> 7) & 0xFF;
    const int M = (int)((sbits & 0x7F) | (E8 ? 0x80u : 0u));
    const int d = (E8 ? (int)E8 : 1) - 134 - ref;
    const float f = d >= -24 ? (float)M * ldexpf(1.0f, d) : 0.f;     // exact in f16: <= 8 bits, >= 2^-24
    const __half hf = __float2half_rn((sbits & 0x8000) ? -f : f);
    const uint32_t hb = (uint32_t)__half_as_ushort(hf);
    fac = hb | (hb << 16);
  } else {
    e2m1x8_to_f16x2(w, v);
    if constexpr (F == MOE_FMT_NVFP4) {
      fac = e4m3_bcast_f16x2(sbits);
    } else {
      const uint32_t hb = f16_pow2_bits((int)(sbits & 0xFF) - ref);
      fac = hb | (hb << 16);
    }
  }
  return make_uint4(hmul2_u32(v[0], fac), hmul2_u32(v[1], fac), hmul2_u32(v[2], fac), hmul2_u32(v[3], fac));
}

// Eight weights (k ascending) of a promote format as four f16x2 of the exact
// code values (int8 / int4 g128 integers, E4M3 values); c: the group of eight
// within the thread's code words.
template <int F>
__device__ __forceinline__ uint4 codes_to_f16(const uint32_t* cw, int c) {
  uint32_t v[4];
  if constexpr (F == MOE_FMT_INT8_G64) {
    int8x4_to_f16x2(cw[2 * c], v[0], v[1]);
    int8x4_to_f16x2(cw[2 * c + 1], v[2], v[3]);
  } else if constexpr (F == MOE_FMT_FP8_B128) {
    e4m3x4_to_f16x2(cw[2 * c], v[0], v[1]);
    e4m3x4_to_f16x2(cw[2 * c + 1], v[2], v[3]);
  } else {
    uint32_t p[4];
    int4x8_to_f16x2_paired(cw[c] ^ 0x88888888u, p);  // unsigned nibble u -> u - 8: flip the top bit
    v[0] = prmt(p[0], p[1], 0x5410u);
    v[1] = prmt(p[2], p[3], 0x5410u);
    v[2] = prmt(p[0], p[1], 0x7632u);
    v[3] = prmt(p[2], p[3], 0x7632u);
  }
  return make_uint4(v[0], v[1], v[2], v[3]);
}

// The fold-scales lever: eight weights (k ascending) of a promote format as
// four bf16x2, each bf16(fl32(code * sc)) (the FP32 product, then BF16
// nearest-even).
template <int F>
__device__ __forceinline__ uint4 fold_lever_word(const uint32_t* cw, int c, float sc) {
  const uint4 q = codes_to_f16<F>(cw, c);  // exact code values
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * sc, f.y * sc);
    o[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Scale of group g (GS K steps) for weight row `row` of expert e (FP8 b128: the
// 128 x 128 block of row tile rt).
template <int F>
__device__ __forceinline__ float group_scale(const QW& W, int e, int N, int K, int row, int rt, int g) {
  const uint8_t* sc = W.scales + (size_t)e * scale_bytes(F, N, K);
  if constexpr (F == MOE_FMT_INT8_G64) {
    return bf16_bits_to_float(__ldg(reinterpret_cast<const uint16_t*>(sc) + (size_t)row * (K / 64) + g));
  } else if constexpr (F == MOE_FMT_FP8_B128) {
    return __ldg(reinterpret_cast<const float*>(sc) + (size_t)rt * (K / 128) + g);
  } else {
    return __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(sc) + (size_t)row * (K / 128) + g)));
  }
}

// The tile list: the dispatch's (expert, first sorted position) pairs, or, for
// the shared expert (a.dense_T > 0), consecutive runs of NT tokens of one
// weight set in token order.
__device__ __forceinline__ int2 tile_at(const PrefillArgs& a, int i) {
  return a.dense_T ? make_int2(0, i * NT) : a.tiles[i];
}
__device__ __forceinline__ int tile_valid(const PrefillArgs& a, int2 t) {
  return min(NT, (a.dense_T ? a.dense_T : a.rb.off[t.x + 1]) - t.y);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
      "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

template <int F, bool DOWN, int LV>
__global__ void __launch_bounds__(kPfGemmThreads, 1) pf_gemm_kernel(PrefillArgs a,
                                                                    const __grid_constant__ CUtensorMap tmB) {
  using C = Cfg<F, DOWN, LV>;
  constexpr bool FS = C::FS, F8 = C::F8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_a[C::SA], empty_a[C::SA], full_b[C::SB], empty_b[C::SB];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], drain;
  __shared__ uint32_t tmem_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, I = a.I, k = a.k;
  const int K = DOWN ? I : H;          // reduction length
  const int N = DOWN ? H : I;          // rows of one weight matrix
  const int RT = N / BM;               // row tiles per token tile
  const int nsteps = K / C::KSTEP;
  const int n_items = (a.dense_T ? (a.dense_T + NT - 1) / NT : a.rb.ctrl->n_tiles) * RT;
  Ctrl* ctrl = a.rb.ctrl;

  if (tid == 0) {
    for (int i = 0; i < C::SA; ++i) {
      tc::bar_init(&full_a[i], kDec);
      tc::bar_init(&empty_a[i], 1);
    }
    for (int i = 0; i < C::SB; ++i) {
      tc::bar_init(&full_b[i], 1);
      tc::bar_init(&empty_b[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::bar_init(&acc_full[b], 1);
      tc::bar_init(&acc_empty[b], kEpiThreads);
    }
    tc::bar_init(&drain, 1);
    tc::bar_init_fence();
  }
  if (warp == kWarpMma) tc::tmem_alloc(&tmem_slot, C::TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp < kDec / 32) {
    // ----------------------------------------------------------- decode --
    const int d = tid;
    const int m = d / (BM * C::TPR);
    const int rr = (d % (BM * C::TPR)) / C::TPR;
    const int hh = d % C::TPR;
    const QW& W = DOWN ? a.down : (m == 0 ? a.gate : a.up);
    uint8_t* raw = smem + C::RAW_OFF + d * C::RAW_BYTES;
    uint32_t g = 0;
    bool ok = true;
    if constexpr (F8) {
      // FP8-activation lever: the E4M3 weight codes are the MMA's A operand as stored.  Each thread
      // copies its row's step (128 bytes for gate/up, 64 for down) straight into the swizzled A
      // stage and arrives two steps later, once those copies have landed.
      for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
        const int2 tile = tile_at(a, it / RT);
        const int rt = it % RT, e = tile.x;
        const int row = rt * BM + rr;
        const uint8_t* crow = W.data + (size_t)e * data_bytes(F, N, K) + (size_t)row * (size_t)K;
        const uint32_t g0 = g;
#pragma unroll 1
        for (int s = 0; s < nsteps; ++s, ++g) {
          const int stage = g % C::SA;
          if (!tc::bar_wait(&empty_a[stage], ((g / C::SA) & 1) ^ 1, a.wait_ns)) {
            report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x300 | (DOWN ? 1 : 0));
            ok = false;
            break;
          }
          uint8_t* A = smem + stage * C::A_STAGE + m * C::A_BYTES;
          const uint8_t* src = crow + (size_t)s * C::KSTEP + hh * C::KT;
#pragma unroll
          for (int j = 0; j < C::CODE_BYTES / 16; ++j)
            cp_async16(A + tc::sw128_off(rr, hh * (C::CODE_BYTES / 16) + j), src + 16 * j);
          cp_async_commit();
          if (s >= 2) {
            cp_async_wait<2>();
            tc::fence_proxy_async();
            tc::bar_arrive(&full_a[(g - 2) % C::SA]);
          }
        }
        if (!ok) break;
        // the item's last (up to two) steps
        cp_async_wait<0>();
        tc::fence_proxy_async();
        for (int s = nsteps > 2 ? nsteps - 2 : 0; s < nsteps; ++s) tc::bar_arrive(&full_a[(g0 + s) % C::SA]);
      }
    }
    if constexpr (!F8)
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const int2 tile = tile_at(a, it / RT);
      const int rt = it % RT, e = tile.x;
      const int row = rt * BM + rr;
      const uint8_t* crow = W.data + (size_t)e * data_bytes(F, N, K) + (size_t)row * ((size_t)K * C::BITS / 8);
      const uint8_t* srow = (C::PROMOTE || FS) ? nullptr
                                               : W.scales + (size_t)e * scale_bytes(F, N, K) +
                                                     (size_t)row * row_scale_bytes<F>(K);
      auto issue = [&](int s) {
        uint8_t* dst = raw + (s % C::RAW) * (kDec * C::RAW_BYTES);
        const uint8_t* src = crow + (size_t)(s * BK + hh * C::KT) * C::BITS / 8;
#pragma unroll
        for (int j = 0; j < C::CODE_BYTES / 16; ++j) cp_async16(dst + 16 * j, src + 16 * j);
        if constexpr (!C::PROMOTE && !FS) {
          // the aligned word holding the step's scales (their byte offset in it is taken at the read)
          cp_async4(dst + C::CODE_BYTES,
                    reinterpret_cast<const void*>(reinterpret_cast<uintptr_t>(srow + step_scale_off<F>(s)) & ~(uintptr_t)3));
        }
      };
#pragma unroll 1
      for (int j = 0; j < C::RAW - 1; ++j) {
        if (j < nsteps) issue(j);
        cp_async_commit();
      }
      int ref = 0;
      if constexpr (!C::PROMOTE && !FS) ref = row_ref<F>(srow, K);  // while the first steps are in flight
      // FS: the group scale of the next step, loaded one step ahead
      float sc_next = 0.f;
      if constexpr (FS) sc_next = group_scale<F>(W, e, N, K, row, rt, 0);
#pragma unroll 1
      for (int s = 0; s < nsteps; ++s, ++g) {
        if (s + C::RAW - 1 < nsteps) issue(s + C::RAW - 1);
        cp_async_commit();
        cp_async_wait<C::RAW - 1>();
        const uint8_t* src = raw + (s % C::RAW) * (kDec * C::RAW_BYTES);
        // 16-byte shared loads: conflict-free at this thread stride
        uint32_t cw[C::CODE_BYTES / 4];
#pragma unroll
        for (int c4 = 0; c4 < C::CODE_BYTES / 16; ++c4) {
          const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * c4);
          cw[4 * c4] = v.x; cw[4 * c4 + 1] = v.y; cw[4 * c4 + 2] = v.z; cw[4 * c4 + 3] = v.w;
        }
        uint4 out[C::KT / 8];
        if constexpr (FS) {
          const float sc = sc_next;
          if (s + 1 < nsteps) sc_next = group_scale<F>(W, e, N, K, row, rt, (s + 1) / C::GS);
#pragma unroll
          for (int c = 0; c < C::KT / 8; ++c) out[c] = fold_lever_word<F>(cw, c, sc);
        } else if constexpr (C::PROMOTE) {
#pragma unroll
          for (int c = 0; c < C::KT / 8; ++c) out[c] = codes_to_f16<F>(cw, c);
        } else {
          const uint32_t sw = *reinterpret_cast<const uint32_t*>(src + C::CODE_BYTES) >>
                              (8 * ((uint32_t)reinterpret_cast<uintptr_t>(srow + step_scale_off<F>(s)) & 3u));
#pragma unroll
          for (int c = 0; c < C::KT / 8; ++c) {
            const int col = hh * C::KT + c * 8;  // first column of word c within the step
            uint32_t sbits;
            if constexpr (F == MOE_FMT_NVFP4) sbits = (sw >> (8 * (col / 16))) & 0xFF;
            else if constexpr (F == MOE_FMT_MXFP4) sbits = (sw >> (8 * (col / 32))) & 0xFF;
            else sbits = sw & 0xFFFF;
            out[c] = fold_word<F>(cw[c], sbits, ref);
          }
        }
        const int stage = g % C::SA;
        if (!tc::bar_wait(&empty_a[stage], ((g / C::SA) & 1) ^ 1, a.wait_ns)) {
          report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x300 | (DOWN ? 1 : 0));
          ok = false;
          break;
        }
        uint8_t* A = smem + stage * C::A_STAGE + m * C::A_BYTES;
#pragma unroll
        for (int c = 0; c < C::KT / 8; ++c)
          *reinterpret_cast<uint4*>(A + tc::sw128_off(rr, hh * (C::KT / 8) + c)) = out[c];
        tc::fence_proxy_async();
        tc::bar_arrive(&full_a[stage]);
      }
    }
    cp_async_wait<0>();
  } else if (warp == kWarpLoader) {
    // --------------------------------------------------------- B loader --
    uint32_t g = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const int pos0 = tile_at(a, it / RT).y;
#pragma unroll 1
      for (int s = 0; s < nsteps; ++s, ++g) {
        const int stage = g % C::SB;
        if (!tc::bar_wait(&empty_b[stage], ((g / C::SB) & 1) ^ 1, a.wait_ns)) {
          report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x320 | (DOWN ? 1 : 0));
          ok = false;
          break;
        }
        uint8_t* B = smem + C::B_OFF + stage * C::B_BYTES;
        if (lane == 0) tc::bar_arrive_expect_tx(&full_b[stage], C::B_BYTES);
        __syncwarp();
        // rows past the tile's tokens (the next segment, or zero fill) only feed discarded columns
        if (lane == 0) tc::tma_load_2d(B, &tmB, s * C::KSTEP, pos0, &full_b[stage]);
      }
    }
    // every load this warp issued has landed before the CTA can exit (the MMA warp may have stopped early)
    if (lane == 0) tc::drain_loads(full_b, C::SB, g, kDrainLimit);
    __syncwarp();
  } else if (warp == kWarpMma) {
    // -------------------------------------------------------------- MMA --
    // The whole warp runs this loop (every value warp-uniform, every branch
    // taken by all lanes); one elected lane issues each MMA and commit.
    uint32_t g = 0, gg = 0;
    int item = 0;
    bool ok = true;
    // one K step's MMAs into the accumulator set at `acc` (each matrix NT columns apart)
    auto step = [&](uint32_t acc, bool accumulate, uint32_t idesc) -> bool {
      const int sa = g % C::SA, sb = g % C::SB;
      const bool ready = tc::bar_wait(&full_a[sa], (g / C::SA) & 1, a.wait_ns) &&
                         tc::bar_wait(&full_b[sb], (g / C::SB) & 1, a.wait_ns);
      if (!__all_sync(0xFFFFFFFFu, ready)) {
        if (lane == 0) report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x340 | (DOWN ? 1 : 0));
        return false;
      }
      // the decode warps fenced their generic-proxy stores before arriving; TMA writes are async-proxy
      tc::fence_after_sync();
      const uint32_t base = tc::smem_u32(smem + sa * C::A_STAGE);
      const uint32_t bB = tc::smem_u32(smem + C::B_OFF + sb * C::B_BYTES);
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        const uint64_t db = tc::smem_desc_sw128(bB + kk * 32);
#pragma unroll
        for (int mm = 0; mm < C::NMAT; ++mm) {
          const uint64_t da = tc::smem_desc_sw128(base + mm * C::A_BYTES + kk * 32);
          if constexpr (F8) tc::mma_e4m3_elect(acc + mm * NT, da, db, idesc, accumulate || kk != 0);
          else tc::mma_f16_elect(acc + mm * NT, da, db, idesc, accumulate || kk != 0);
        }
      }
      tc::commit_elect(&empty_a[sa]);
      tc::commit_elect(&empty_b[sb]);
      ++g;
      return true;
    };
    // a wait on the epilogue, taken by all lanes or failed by all
    auto acc_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      if (!__all_sync(0xFFFFFFFFu, tc::bar_wait(bar, parity, a.wait_ns))) {
        if (lane == 0) report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x330 | (DOWN ? 1 : 0));
        return false;
      }
      tc::fence_after_sync();
      return true;
    };
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, ++item) {
      const int n_valid = tile_valid(a, tile_at(a, it / RT));
      const int n_mma = (n_valid + 15) & ~15;
      // FS: bf16 operands; F8: E4M3 A and B (format code 0 of kind::f8f6f4, the bits of f16 in kind::f16)
      const uint32_t idesc = tc::idesc_f16(BM, n_mma, FS ? 1 : 0);
      if constexpr (C::PROMOTE) {
        // each scale group into the block set; the epilogue empties it before the next group
        const uint32_t blk = tmem + C::ACC_COLS;
#pragma unroll 1
        for (int s0 = 0; ok && s0 < nsteps; s0 += C::GS, ++gg) {
          if (!acc_wait(&acc_empty[0], (gg & 1) ^ 1)) {
            ok = false;
            break;
          }
#pragma unroll 1
          for (int j = 0; j < C::GS; ++j)
            if (!step(blk, j != 0, idesc)) {
              ok = false;
              break;
            }
          if (ok) tc::commit_elect(&acc_full[0]);
        }
      } else {
        const int buf = item & 1;
        if (!acc_wait(&acc_empty[buf], ((item >> 1) & 1) ^ 1)) break;
        const uint32_t acc = tmem + buf * C::ACC_COLS;
#pragma unroll 1
        for (int s = 0; s < nsteps; ++s)
          if (!step(acc, s != 0, idesc)) {
            ok = false;
            break;
          }
        if (!ok) break;
        tc::commit_elect(&acc_full[buf]);
      }
    }
    tc::commit_elect(&drain);
    tc::bar_wait(&drain, 0, kDrainLimit);
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue --
    // warp w handles TMEM lanes (= weight rows of the tile) 32 * (w % 4) ..
    // and half of the columns; the tile is staged in shared memory as
    // [column][row] and leaves with one bulk copy per column (a contiguous
    // run of the output row).
    const int ew = warp - kWarpEpi0;
    const int q = warp & 3, chalf = ew >> 2;  // columns [64 * chalf, 64 * chalf + 64)
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    uint8_t* stg = smem + C::STG_OFF;
    const int row = q * 32 + lane;
    int item = 0;
    uint32_t gg = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++item) {
      const int2 tile = tile_at(a, it / RT);
      const int rt = it % RT, e = tile.x, pos0 = tile.y;
      const int n_valid = tile_valid(a, tile);
      // per-column scale factors of this warp's columns, fetched before the wait
      float un_c[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int pos_l = pos0 + min(chalf * 64 + i * 32 + lane, n_valid - 1);
        if (FS || F8) un_c[i] = 1.f;  // plain BF16 tokens / activation scales applied per group
        else if (DOWN) un_c[i] = exp2i(-a.hsig[pos_l]);
        else un_c[i] = exp2i(-a.xsig[a.dense_T ? pos_l : a.rb.pair[pos_l] / k]);
      }
      const int erow = rt * BM + row;
      bool stop = false;
      if constexpr (C::PROMOTE) {
        // per scale group: running = scale * block (+ running), the running sums in TMEM
        // columns [0, ACC_COLS), the group's block in [ACC_COLS, 2 ACC_COLS)
        const int ngrp = nsteps / C::GS;
#pragma unroll 1
        for (int gi = 0; gi < ngrp; ++gi, ++gg) {
          float sc[C::NMAT];
#pragma unroll
          for (int mm = 0; mm < C::NMAT; ++mm)
            sc[mm] = group_scale<F>(DOWN ? a.down : (mm == 0 ? a.gate : a.up), e, N, K, erow, rt, gi);
          // F8: the group's activation scales of this warp's columns, fetched before the wait (lane j < 16
          // of chunk ch holds column chalf * 64 + ch * 16 + j)
          float asv[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (F8) {
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              const int cj = chalf * 64 + ch * 16 + (lane & 15);
              asv[ch] = cj < n_valid ? __ldg(a.asc + (size_t)(pos0 + cj) * (K / 128) + gi) : 0.f;
            }
          }
          const bool ready = tc::bar_wait(&acc_full[0], gg & 1, a.wait_ns);
          if (!ready) report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x310 | (DOWN ? 1 : 0));
          // all epilogue warps go on, or all stop; the barrier also frees the staging tile
          if (!tc::named_all(1, kEpiThreads, ready)) {
            stop = true;
            break;
          }
          tc::fence_after_sync();
          const bool last = gi == ngrp - 1;
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {
            const int c0 = chalf * 64 + ch * 16;
            if (c0 >= n_valid) break;
            float r[C::NMAT][16];
            // F8: the group's activation scale of each of the chunk's columns (lane j < 16 loads column
            // c0 + j), so the group's factor is weight scale x activation scale
            float fa[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) fa[j] = 1.f;
            if constexpr (F8) {
              const float asl = ch == 0 ? asv[0] : ch == 1 ? asv[1] : ch == 2 ? asv[2] : asv[3];
#pragma unroll
              for (int j = 0; j < 16; ++j) fa[j] = __shfl_sync(0xFFFFFFFFu, asl, j);
            }
#pragma unroll
            for (int mm = 0; mm < C::NMAT; ++mm) {
              uint32_t bv[16], rv[16];
              tc::tmem_ld16(tq + C::ACC_COLS + mm * NT + c0, bv);
              if (gi > 0) tc::tmem_ld16(tq + mm * NT + c0, rv);
              tc::tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float f = F8 ? sc[mm] * fa[j] : sc[mm];
                r[mm][j] = gi > 0 ? fmaf(f, __uint_as_float(bv[j]), __uint_as_float(rv[j]))
                                  : f * __uint_as_float(bv[j]);
              }
              if (!last) tmem_st16(tq + mm * NT + c0, r[mm]);
            }
            if (last) {
              const int ncol = min(16, n_valid - c0);
              const float un_i = un_c[(ch * 16) / 32];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float un = __shfl_sync(0xFFFFFFFFu, un_i, (ch * 16) % 32 + j);
                if (j < ncol) {
                  if (!DOWN) {
                    const float gv = r[0][j] * un, uv = r[C::NMAT - 1][j] * un;
                    reinterpret_cast<uint16_t*>(stg)[(size_t)(c0 + j) * BM + row] = float_to_bf16_bits(silu(gv) * uv);
                  } else {
                    // P row of sorted position pos0 + c0 + j: the warp's 32 lanes write 32 consecutive rows
                    const size_t o = (size_t)(pos0 + c0 + j) * H + rt * BM + row;
                    if (a.p_bf16) reinterpret_cast<uint16_t*>(a.P)[o] = float_to_bf16_bits(r[0][j] * un);
                    else a.P[o] = r[0][j] * un;
                  }
                }
              }
            }
          }
          if (!last) tmem_st_wait();
          tc::fence_before_sync();
          tc::bar_arrive(&acc_empty[0]);  // the block set is free for the next group's MMAs
        }
        if (stop) break;
      } else {
        // the factor of this thread's row (TMEM lane) in each matrix: tensor scale or 2^reference
        float rf[2];
#pragma unroll
        for (int mm = 0; mm < C::NMAT; ++mm) {
          if constexpr (FS) {
            rf[mm] = 1.f;  // the scales are in the BF16 weights
          } else {
            const QW& Wm = DOWN ? a.down : (mm == 0 ? a.gate : a.up);
            const uint8_t* sr =
                Wm.scales + (size_t)e * scale_bytes(F, N, K) + (size_t)erow * row_scale_bytes<F>(K);
            rf[mm] = row_factor<F>(row_ref<F>(sr, K), F == MOE_FMT_NVFP4 ? __ldg(Wm.ts + e) : 1.f);
          }
        }
        const float tsg = DOWN ? 0.f : rf[0], tsu = DOWN ? 0.f : rf[C::NMAT - 1];
        const int buf = item & 1;
        const bool ready = tc::bar_wait(&acc_full[buf], (item >> 1) & 1, a.wait_ns);
        if (!ready) report_error(ctrl, (uint32_t)MOE_ERR_DEVICE_TIMEOUT, 0x310 | (DOWN ? 1 : 0));
        // all epilogue warps go on, or all stop; the barrier also frees the staging tile
        // (the previous tile's copies have read it)
        if (!tc::named_all(1, kEpiThreads, ready)) break;
        tc::fence_after_sync();
        const uint32_t acc = tq + buf * C::ACC_COLS;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int c0 = chalf * 64 + i * 32;
          if (c0 >= n_valid) break;
          const int ncol = min(32, n_valid - c0);
          if (!DOWN) {
            uint32_t gv[32], uv[32];
            tc::tmem_ld32(acc + c0, gv);
            tc::tmem_ld32(acc + NT + c0, uv);
            tc::tmem_ld_wait();
            uint16_t* st16 = reinterpret_cast<uint16_t*>(stg) + (size_t)c0 * BM + row;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float un = __shfl_sync(0xFFFFFFFFu, un_c[i], j);
              if (j < ncol) {
                const float gg2 = __uint_as_float(gv[j]) * (tsg * un);
                const float uu = __uint_as_float(uv[j]) * (tsu * un);
                st16[j * BM] = float_to_bf16_bits(silu(gg2) * uu);
              }
            }
          } else {
            uint32_t dv[32];
            tc::tmem_ld32(acc + c0, dv);
            tc::tmem_ld_wait();
            // P straight from registers: for each column (sorted position) the warp's 32 lanes write
            // 32 consecutive rows of P, one coalesced 128-byte store (64 bytes under bf16 partials)
            float* p32 = a.P + (size_t)(pos0 + c0) * H + rt * BM + row;
            uint16_t* p16 = reinterpret_cast<uint16_t*>(a.P) + (size_t)(pos0 + c0) * H + rt * BM + row;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float un = __shfl_sync(0xFFFFFFFFu, un_c[i], j);
              if (j < ncol) {
                const float v = __uint_as_float(dv[j]) * (rf[0] * un);
                if (a.p_bf16) p16[(size_t)j * H] = float_to_bf16_bits(v);
                else p32[(size_t)j * H] = v;
              }
            }
          }
        }
        tc::fence_before_sync();
        tc::bar_arrive(&acc_empty[buf]);  // TMEM buffer free for the MMA of a later tile
      }
      if constexpr (!DOWN) {
        // h leaves through the staging tile: one bulk copy per column (a contiguous run of its row)
        tc::fence_proxy_async();          // staging writes -> bulk copy reads
        tc::named_sync(1, kEpiThreads);
        if (ew == 0) {
          for (int c = lane; c < n_valid; c += 32)
            tc::bulk_store(a.h + (size_t)(pos0 + c) * I + rt * BM, stg + c * BM * 2, BM * 2);
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
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
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

// f16 matrix [rows, cols] (row-major), boxes of 64 columns x box_rows rows,
// 128-byte swizzle, zero fill outside the matrix.
bool f16_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// E4M3 codes [rows, cols] (row-major bytes), boxes of 128 bytes x box_rows rows,
// 128-byte swizzle, zero fill outside the matrix (the FP8-activation lever's B).
bool u8_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {128u, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// LV: the lever (0 none, 1 fold scales: B is plain BF16 x rows and h rows; 2 FP8 activations: B is the
// E4M3 codes of x and h, their block scales in the argument block's asc).
template <int F, int LV>
cudaError_t launch_pf_gemm(bool down, const PrefillArgs& a, int grid, cudaStream_t s) {
  cudaError_t err;
  alignas(64) CUtensorMap tm;
  PrefillArgs b = a;
  const uint64_t rows = (uint64_t)a.T * a.k;
  const int K = down ? a.I : a.H;
  void* src = down ? (LV == 1 ? (void*)a.h : (void*)a.h16) : (void*)a.xg;
  if (LV == 2) {
    if (!u8_map(&tm, src, (uint64_t)K, rows, NT)) return cudaErrorInvalidValue;
    b.asc = fp8_scales_after(src, rows, K);
  } else if (!f16_map(&tm, src, (uint64_t)K, rows, NT)) {
    return cudaErrorInvalidValue;
  }
  if (down) {
    err = cudaFuncSetAttribute(pf_gemm_kernel<F, true, LV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<F, true, LV>::SMEM);
    if (err != cudaSuccess) return err;
    pf_gemm_kernel<F, true, LV><<<grid, kPfGemmThreads, Cfg<F, true, LV>::SMEM, s>>>(b, tm);
  } else {
    err = cudaFuncSetAttribute(pf_gemm_kernel<F, false, LV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<F, false, LV>::SMEM);
    if (err != cudaSuccess) return err;
    pf_gemm_kernel<F, false, LV><<<grid, kPfGemmThreads, Cfg<F, false, LV>::SMEM, s>>>(b, tm);
  }
  return cudaGetLastError();
}

cudaError_t launch_prefill_gemm(bool down, const PrefillArgs& a, int grid, cudaStream_t s) {
  switch (a.fmt) {
    case MOE_FMT_NVFP4: return launch_pf_gemm<MOE_FMT_NVFP4, 0>(down, a, grid, s);
    case MOE_FMT_MXFP4: return launch_pf_gemm<MOE_FMT_MXFP4, 0>(down, a, grid, s);
    case MOE_FMT_INT4_G64: return launch_pf_gemm<MOE_FMT_INT4_G64, 0>(down, a, grid, s);
    case MOE_FMT_INT8_G64:
      return fold_lever(a) ? launch_pf_gemm<MOE_FMT_INT8_G64, 1>(down, a, grid, s)
                           : launch_pf_gemm<MOE_FMT_INT8_G64, 0>(down, a, grid, s);
    case MOE_FMT_FP8_B128:
      return fp8_lever(a)    ? launch_pf_gemm<MOE_FMT_FP8_B128, 2>(down, a, grid, s)
             : fold_lever(a) ? launch_pf_gemm<MOE_FMT_FP8_B128, 1>(down, a, grid, s)
                             : launch_pf_gemm<MOE_FMT_FP8_B128, 0>(down, a, grid, s);
    case MOE_FMT_INT4_G128:
      return fold_lever(a) ? launch_pf_gemm<MOE_FMT_INT4_G128, 1>(down, a, grid, s)
                           : launch_pf_gemm<MOE_FMT_INT4_G128, 0>(down, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmoe
