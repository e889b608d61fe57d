// Kernel argument blocks and launch entry points shared by the host ABI and
// the kernel translation units.
#pragma once

#include "common.cuh"

namespace qmoe {

struct QW {
  const uint8_t* data;
  const uint8_t* scales;
  const float* ts;  // NVFP4 tensor scales [count], else nullptr
};

// Routing results and scratch buffers inside the caller's workspace.
struct RouteBufs {
  Ctrl* ctrl;
  float* logits;      // [T, E]
  int32_t* topk_idx;  // [T, k]
  float* topk_w;      // [T, k]
  int32_t* cnt;       // [E]
  int32_t* off;       // [E + 1]
  int32_t* pair;      // [T * k]
  int32_t* act;       // [E] active experts, ascending
};

// Optional copies of the routing results into caller buffers (moe_route).
struct RouteOut {
  int32_t* topk_idx;
  float* topk_w;
  int32_t* cnt;
  int32_t* off;
  int32_t* pair;
};

struct RouterArgs {
  int H, E, k, T;
  int wpr;            // warps per expert row of the approximate pass
  int bias_select;    // 1: the bias steers the selection only, the weights use the unbiased logits
  const uint16_t* x;  // bf16 [T, H]
  const float* w;     // [E, H]
  const float* bias;  // [E] or nullptr
  RouteBufs rb;
  RouteOut out;
  float* approx;      // [T, E] unbiased exact logits (written under bias_select)
  const float* sgate_w;  // [H] gate vector of the shared expert, or nullptr
  float* sgate;       // [T] sigmoid(x_t . sgate_w) (written when sgate_w is set)
};

// Decode-path expert kernels.
struct ExpertArgs {
  int H, I, E, k, T;
  int fmt, sfmt, Is;  // routed format; shared format (0 = none) and size
  const uint16_t* x;  // bf16 [T, H]
  QW gate, up, down, sgate, sup, sdown;
  RouteBufs rb;
  uint16_t* h;        // bf16 [T*k, I]
  uint16_t* hs;       // bf16 [T, Is]
  float* P;           // f32 [T*k, H] per-pair down partials
  float* S;           // f32 [T, H] shared expert output
  uint16_t* y;        // bf16 [T, H]
  int gu_slices, dn_slices;  // K slices per 16-row tile (1 = no split)
  int gu_slices_s;           // K slices per shared-expert tile of the gate/up kernel
  int gu_slices_t;           // K slices per routed gate/up tile beyond the first wave (>= gu_slices)
  int gu_tail_cap;           // most routed tiles the block-sum buffer holds at gu_slices_t (gu_slices == 1)
  float* gu_part;     // block sums of split tiles, [tile blocks][32 lanes][8]
  uint32_t* gu_cnt;   // [tiles] slice arrival counters
  float* dn_part;     // [tile blocks][32 lanes][4]
  uint32_t* dn_cnt;   // [tiles]
  int xs_tok_stride;  // halfs per staged token row (gate/up)
  int hs_tok_stride;  // halfs per staged hidden row (down)
  int dn_segs;        // expert segments the down kernel stages at once (1 .. kMaxDnSegs)
  const float* shared_g;  // [T] sigmoid gate of the shared expert per token, or nullptr (weight 1)
  int p_bf16;         // 1: P and S are stored as BF16 (the bf16-partials lever)
};

constexpr int kMaxDnSegs = 4;

constexpr int kExpertThreads = 256;  // 8 warps
// Gate/up: batches of at most kGuSmallT tokens run 3 CTAs per SM with 2
// cp.async ring stages per warp, larger ones 2 CTAs per SM with 3 stages.
constexpr int kGuSmallT = 4;
__host__ __device__ constexpr int gu_stages(int ctas_per_sm) { return ctas_per_sm >= 3 ? 2 : 3; }
constexpr int kStagesDN = 4;         // cp.async ring stages per warp, down (one matrix per unit)
// Bytes of one ring stage: NM matrices x 2 rows x 32 lanes x (16 B codes + 4 B scale word).
constexpr int dec_stage_bytes(int nm) { return nm * 2 * 32 * (16 + 4); }
constexpr int kRouterThreads = 256;
// Cap on stored block sums when tiles are split along K (bounds the partial buffers).
constexpr int kMaxSplitBlocks = 16384;

int router_warps_per_row(int H, int E, int sms);
// Zero the control block and every arrival counter of a workspace laid out
// for this layer and workspace size (stream-ordered memsets, no allocation);
// keep_error leaves the device-side error word and its info as they are.
int32_t clear_workspace_counters(const moe_layer* L, void* ws, size_t ws_bytes, bool keep_error, cudaStream_t s);
// Host checks of moe_decode_forward's arguments other than the workspace.
int32_t check_decode_args(const moe_layer* layer, const void* x, int32_t T, const void* y, const moe_options* opts);
// The allocation-free entry point's array on the current device, or nullptr
// in *out if no call has used it on this device yet.
int32_t noalloc_array_if_used(void** out);
cudaError_t launch_router_decode(const RouterArgs& a, cudaStream_t s);
// Caller-supplied top-k indices and weights copied into the workspace (and the shared expert's gate);
// the gate/up kernel builds the dispatch index from them.
cudaError_t launch_dispatch_ext(const RouterArgs& a, const int32_t* idx, const float* w, cudaStream_t s);
// moe_route: the dispatch index of the router's choices.
cudaError_t launch_route_dispatch(const RouterArgs& a, cudaStream_t s);
// Gate/up (down = false) or down (down = true) for a routed format;
// the shared format is selected at run time among the compiled instances.
cudaError_t launch_expert_nvfp4(int sfmt, bool down, const ExpertArgs& a, size_t smem, cudaStream_t s);
cudaError_t launch_expert_mxfp4(int sfmt, bool down, const ExpertArgs& a, size_t smem, cudaStream_t s);
cudaError_t launch_expert_int4(int sfmt, bool down, const ExpertArgs& a, size_t smem, cudaStream_t s);
cudaError_t launch_expert_int8(int sfmt, bool down, const ExpertArgs& a, size_t smem, cudaStream_t s);
cudaError_t launch_expert_fp8(int sfmt, bool down, const ExpertArgs& a, size_t smem, cudaStream_t s);
cudaError_t launch_expert_int4g128(int sfmt, bool down, const ExpertArgs& a, size_t smem, cudaStream_t s);

// ---------------------------------------------------------------- prefill --
// Any token count.  Routing: FP32 approximate logits with a rigorous error
// bound, exact (correctly rounded) logits for the experts that can still
// reach the top-k, then a chunked counting-sort dispatch.  Experts: grouped
// GEMMs on tcgen05 over token tiles of one expert each.
constexpr int kPfTokTile = 128;    // tokens per GEMM tile (MMA N)
constexpr int kPfRowTile = 128;    // weight rows per GEMM tile (MMA M)
constexpr int kPfChunk = 64;       // tokens per dispatch chunk
constexpr int kPfGemmThreads = 576;  // 8 decode warps, B loader, MMA, 8 epilogue warps

struct PrefillArgs {
  int H, I, E, k, T;
  int fmt;
  const uint16_t* x;    // bf16 [T, H]
  const float* rw;      // router [E, H]
  const float* bias;    // [E] or nullptr
  QW gate, up, down;
  RouteBufs rb;         // logits [T, E] (approximate, then exact for candidates), top-k, cnt, off, pair
  RouteOut out;
  uint16_t* xg;         // f16 [T*k, H]: row pos = x[token of pos] * 2^xsig[token] (sorted order);
                        // under the fold-scales lever the BF16 row x[token of pos] itself
  int32_t* xsig;        // [T]
  float* xnorm;         // [T] ||x_t||_2
  float* wnorm;         // [E] ||Wr_e||_2
  int32_t* hist;        // [nchunk, E]: per-chunk counts, then per-chunk bases
  int32_t* pos_of;      // [T*k] sorted position of pair p
  int2* tiles;          // [max tiles] (expert, first sorted position)
  int max_tiles;
  uint16_t* h;          // bf16 [T*k, I] in sorted order
  uint32_t* h_amax;     // unused by the prefill path (nullptr)
  uint16_t* h16;        // f16 [T*k, I]: h * 2^hsig[pos]
  int32_t* hsig;        // [T*k]
  float* P;             // f32 [T*k, H] in sorted order (row pos)
  uint16_t* y;          // bf16 [T, H]
  // approximate logits on tensor cores (bf16 split of the router matrix) instead of FP32 FMA
  int logits_tc;
  uint16_t* rw_hi;      // bf16 [E, H] = bf16(Wr)
  uint16_t* rw_lo;      // bf16 [E, H] = bf16(Wr - hi)
  int bias_select;      // 1: the bias steers the selection only (weights from the unbiased logits)
  float* unbiased;      // [T, E] unbiased exact logits of the recomputed experts (bias_select)
  uint64_t wait_ns;     // limit of every bounded device wait (nanoseconds)
  int p_bf16;           // 1: the down GEMM writes P as BF16 (the bf16-partials lever)
  int fold_scales;      // 1: the fold-scales lever (int8 g64 / FP8 b128 / int4 g128 blocks, see fold_lever)
  int fp8_act;          // 1: the FP8-activation lever (FP8 b128 blocks, see fp8_lever)
  const float* asc;     // FP8-activation lever: the B operand's per-row 1x128 scales (set per GEMM launch)
  // NVFP4 W4A4 lever (act_quant = 1)
  int act_quant;
  uint8_t* xq;          // [T, H/2] E2M1 codes of x (16-element blocks)
  uint8_t* xsf;         // [T, H/16] E4M3 block scales of x
  uint8_t* xqg;         // [T*k, H/2] codes in sorted order
  uint8_t* xsfg;        // [T*k, H/16]
  uint8_t* hq;          // [T*k, I/2] codes of h in sorted order
  uint8_t* hsf;         // [T*k, I/16]
  // the shared expert (dense over all T tokens), when the layer has one
  int sfmt, Is;         // its format (0: none) and intermediate size
  QW s_gate, s_up, s_down;
  uint16_t* xs16;       // f16 [T, H]: x[t] * 2^xsig[t] in token order (B operand of the shared gate/up)
  uint16_t* hs;         // bf16 [T, Is]
  uint16_t* hs16;       // f16 [T, Is]: hs * 2^hssig[t]
  int32_t* hssig;       // [T]
  float* S;             // [T, H] shared expert output (f32, or bf16 under p_bf16)
  const float* sgate_w; // [H] gate vector of a sigmoid-gated shared expert, or nullptr
  float* sgate;         // [T] sigmoid(x_t . sgate_w)
  int dense_T;          // > 0: this argument block is the shared expert's (tiles of NT consecutive tokens)
};

// The FP8-activation lever applies to this argument block (routed or shared):
// FP8 b128 weights meet per-token 1x128 E4M3 activations (x, then h) on
// kind::f8f6f4 MMAs, with the weight and activation block scales applied per
// 128-K group in FP32.  It takes precedence over the fold-scales lever.
__host__ __device__ inline bool fp8_lever(const PrefillArgs& a) {
  return a.fp8_act != 0 && a.fmt == MOE_FMT_FP8_B128;
}

// The fold-scales lever applies to this argument block (routed or shared):
// int8 g64, FP8 b128 and int4 g128 weights enter the GEMMs as bf16(code x
// group scale) with plain BF16 tokens and one FP32 accumulator.
__host__ __device__ inline bool fold_lever(const PrefillArgs& a) {
  return a.fold_scales != 0 && !fp8_lever(a) &&
         (a.fmt == MOE_FMT_INT8_G64 || a.fmt == MOE_FMT_FP8_B128 || a.fmt == MOE_FMT_INT4_G128);
}

// FP8-activation lever: the E4M3 codes of a B operand occupy the first rows x K
// bytes of its f16 buffer (xg / h16), the FP32 block scales [rows, K/128]
// follow them (K is a multiple of 128, so they stay 16-byte aligned).
__host__ __device__ inline float* fp8_scales_after(void* codes, size_t rows, int K) {
  return reinterpret_cast<float*>(static_cast<uint8_t*>(codes) + rows * (size_t)K);
}

// Optional host callback between launches (event records of the timed entry
// point): mark(ctx, i) after stage i.
struct Marks {
  void (*fn)(void*, int);
  void* ctx;
  void operator()(int i) const {
    if (fn) fn(ctx, i);
  }
};
// Router + dispatch (+ the sorted token copy when a.xg is set); marks 1
// (logits), 2 (top-k), 3 (dispatch).
cudaError_t launch_prefill_route(const PrefillArgs& a, cudaStream_t s, Marks mk = Marks{nullptr, nullptr});
// Expert GEMMs + combine (after launch_prefill_route); marks 4 (gate/up),
// 5 (h conversion), 6 (down), 7 (combine).
cudaError_t launch_prefill_experts(const PrefillArgs& a, int sms, cudaStream_t s, Marks mk = Marks{nullptr, nullptr});
cudaError_t launch_prefill_topk(const PrefillArgs& a, cudaStream_t s);
bool prefill_logits_tc_ok(const PrefillArgs& a);
cudaError_t launch_prefill_logits_tc(const PrefillArgs& a, cudaStream_t s);
// The exact-chain grouped GEMMs for a.fmt (any of the six weight formats); a.dense_T > 0 runs them
// densely over tokens 0 .. dense_T - 1 of one weight set (the shared expert).
cudaError_t launch_prefill_gemm(bool down, const PrefillArgs& a, int grid, cudaStream_t s);
cudaError_t launch_prefill_gemm_w4a4(bool down, const PrefillArgs& a, int grid, cudaStream_t s);

// Decode combine y = bf16(sum_j w_j P_j (+ g S)), launched after the down
// kernel as a programmatic dependent of it.
cudaError_t launch_combine_decode(const ExpertArgs& a, cudaStream_t s);


// moe_dequantize / moe_quantize_act_nvfp4
cudaError_t launch_dequantize(int fmt, QW w, int N, int K, int expert, int row0, int nrows, float* out,
                              cudaStream_t s);
cudaError_t launch_quantize_act_nvfp4(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales,
                                      cudaStream_t s);
cudaError_t launch_quantize_act_mxfp4(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales,
                                      cudaStream_t s);

// Bytes of one matrix's codes / scales in a format.
__host__ __device__ inline size_t data_bytes(int fmt, int N, int K) {
  switch (fmt) {
    case MOE_FMT_NVFP4: case MOE_FMT_MXFP4: case MOE_FMT_INT4_G64: case MOE_FMT_INT4_G128: return (size_t)N * K / 2;
    case MOE_FMT_INT8_G64: case MOE_FMT_FP8_B128: return (size_t)N * K;
    default: return 0;
  }
}

__host__ __device__ inline size_t scale_bytes(int fmt, int N, int K) {
  switch (fmt) {
    case MOE_FMT_NVFP4: return (size_t)N * (K / 16);
    case MOE_FMT_MXFP4: return (size_t)N * (K / 32);
    case MOE_FMT_INT4_G64: case MOE_FMT_INT8_G64: return (size_t)N * (K / 64) * 2;
    case MOE_FMT_FP8_B128: return (size_t)(N / 128) * (K / 128) * 4;
    case MOE_FMT_INT4_G128: return (size_t)N * (K / 128) * 2;
    default: return 0;
  }
}

// Columns of one decode work unit (four lanes' chunks) in a format; a warp's
// share of K must be a multiple of it.
__host__ __device__ inline int decode_unit_k(int fmt) {
  switch (fmt) {
    case MOE_FMT_NVFP4: case MOE_FMT_MXFP4: case MOE_FMT_INT4_G64: case MOE_FMT_INT4_G128:
      return 128;  // 16 bytes per lane
    case MOE_FMT_INT8_G64: case MOE_FMT_FP8_B128: return 64;
    default: return 0;
  }
}

// The decode kernels sum K as blocks of units (pairs of units when a row has
// an even number of them): the block layout depends only on (format, K).
// Both are 0 for a format code that is not a weight format (0 = no shared expert).
__host__ __device__ inline int dec_block_units(int fmt, int K) {
  const int uk = decode_unit_k(fmt);
  return (uk == 0 || (K / uk) % 2 == 0) ? 2 : 1;
}
__host__ __device__ inline int dec_blocks(int fmt, int K) {
  const int uk = decode_unit_k(fmt);
  return uk == 0 ? 0 : K / uk / dec_block_units(fmt, K);
}

}  // namespace qmoe
