/*
 * moe.h - C ABI of the quantized mixture-of-experts layer for GB300 (sm_103a).
 *
 * One MoE layer computed directly on block-quantized checkpoint weights, with
 * no dequantized copy: router softmax + top-k, expert dispatch, gate/up
 * projection with SwiGLU, down projection and the weighted combine, BF16
 * activations and FP32 accumulation.
 *
 * Sources (the DGPP pages):
 *  - DGPP README (GitHub mirror), intro bullets "Serves checkpoints as
 *    published" (formats read by kernels written for each, no dequantized
 *    copy) and "Exact" (the default chain computes what the checkpoint
 *    specifies; reduced-precision levers are explicit and off by default).
 *  - DGPP README, "Execution and performance" table: engine.prefill_bf16_partials
 *    (per-expert partials summed in fp32 by default), engine.prefill_fold_scales
 *    (per-group scale fma by default), engine.prefill_fp8_gemm (per-token 1x128
 *    e4m3 activations for FP8 weights, off by default), engine.expert_tile_list (expert GEMM over
 *    a compact list of routed segments' tiles), engine.expert_gemm_pair (gate
 *    and up in one launch).
 *  - "DGPP: a GB10-optimized C/CUDA inference engine" (NVIDIA Developer Forums),
 *    post 1, quantisation table (NVFP4 / MXFP4 routed experts, int4 g64 routed
 *    with int8 g64 shared experts, FP8 shared experts; activations stay BF16);
 *    post 15 "Lossless bf12" (decode streams weights at the memory line rate;
 *    weights rebuilt in registers).
 *  - same thread, weekly update on page 5: NVFP4 W4A4 prefill is opt-in.
 *
 * Conventions
 *  - Every pointer marked "device" is a CUDA device pointer owned by the
 *    caller; descriptors (moe_layer, moe_options) live in host memory and are
 *    read only during the call.  The library allocates nothing and keeps no
 *    global state, with one exception: the fixed device array of
 *    moe_decode_forward_noalloc (below).  It is safe to call concurrently on
 *    different streams with different workspaces.
 *  - All calls are asynchronous on `stream` and make no host reads of device
 *    data, so they can be captured in a CUDA graph.  Arguments are validated
 *    on the host before any launch; a failed validation launches nothing.
 *  - Device pointers must be 16-byte aligned (MOE_ERR_MISALIGNED otherwise).
 *  - Weight matrices W[N, K] are row-major with the reduction dimension K
 *    innermost; experts are stacked contiguously: W_e = base + e * stride.
 *    Gate and up are [I, H] per expert, down is [H, I].
 *  - Activations x and outputs y are BF16 [T, H] row-major.
 *  - Results are deterministic: no floating-point atomics; per-expert
 *    partials are summed in FP32 in a fixed order.
 */
#ifndef QMOE_MOE_H
#define QMOE_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's cudaStream_t; NULL selects the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,      /* null pointer, bad size, T out of range, unknown enum   */
  MOE_ERR_UNSUPPORTED = -2,      /* valid but not implemented (shape or format combination) */
  MOE_ERR_MISALIGNED = -3,       /* a device pointer is not 16-byte aligned                 */
  MOE_ERR_WORKSPACE = -4,        /* workspace null or smaller than moe_workspace_size()     */
  MOE_ERR_CUDA = -5,             /* a CUDA runtime call or launch failed                    */
  MOE_ERR_DEVICE_TIMEOUT = -6,   /* a bounded device-side wait gave up (see moe_check)      */
  MOE_ERR_DEVICE_BAD_INDEX = -7  /* a device-side index check failed (see moe_check)        */
} moe_status;

/* Weight formats (DGPP forum post 1, quantisation table). */
typedef enum {
  MOE_FMT_NONE = 0,
  /* E2M1 codes, two per byte (low nibble = even k); E4M3 scale per 16
   * elements, scales [N, K/16] u8; FP32 tensor scale per expert.
   * W = e2m1 * e4m3 * tensor_scale. */
  MOE_FMT_NVFP4 = 1,
  /* E2M1 codes as NVFP4; E8M0 scale per 32 elements, scales [N, K/32] u8.
   * W = e2m1 * 2^(scale - 127). */
  MOE_FMT_MXFP4 = 2,
  /* Symmetric int4, two's-complement nibbles (low nibble = even k), BF16 scale
   * per 64 elements, scales [N, K/64] bf16.  W = q * s. */
  MOE_FMT_INT4_G64 = 3,
  /* Symmetric int8 [N, K], BF16 scale per 64 elements, scales [N, K/64] bf16. */
  MOE_FMT_INT8_G64 = 4,
  /* E4M3 codes [N, K], FP32 scale per 128x128 block, scales [N/128, K/128] f32. */
  MOE_FMT_FP8_B128 = 5,
  /* The AutoRound / GPTQ int4 group-128 layout (DGPP README "Highlights":
   * int4 group-128 experts served in their packed form): unsigned nibbles u
   * (low nibble = even k) with zero point 8, FP16 scale per 128 elements,
   * scales [N, K/128] f16.  W = (u - 8) * s. */
  MOE_FMT_INT4_G128 = 6
} moe_format;

/* A stack of matrices W_e[N, K] (e = 0 .. count-1) in one format. */
typedef struct {
  const void* data;          /* device; codes of expert e at data + e * data_bytes(N, K)      */
  const void* scales;        /* device; scales of expert e at scales + e * scale_bytes(N, K)  */
  const float* tensor_scale; /* device [count] f32; NVFP4 only (ignored for other formats)    */
} moe_qweight;

/* One MoE layer.  Routed experts: E of them, top_k chosen per token. */
typedef struct {
  int32_t hidden;            /* H */
  int32_t inter;             /* I, routed expert intermediate size */
  int32_t n_experts;         /* E, 1 .. 1024 */
  int32_t top_k;             /* k, 1 .. min(E, 16) */
  int32_t fmt;               /* moe_format of the routed experts */
  const float* router_w;     /* device [E, H] f32 */
  const float* router_bias;  /* device [E] f32, added to the FP32 logits, or NULL */
  moe_qweight gate;          /* [E] x [I, H] */
  moe_qweight up;            /* [E] x [I, H] */
  moe_qweight down;          /* [E] x [H, I] */
  int32_t shared_fmt;        /* moe_format of the shared expert, MOE_FMT_NONE if absent */
  int32_t shared_inter;      /* Is */
  moe_qweight shared_gate;   /* [1] x [Is, H] */
  moe_qweight shared_up;     /* [1] x [Is, H] */
  moe_qweight shared_down;   /* [1] x [H, Is] */
  /* device [H] f32 or NULL.  When set, the shared expert's output is scaled
   * per token by sigmoid(g_t), g_t the correctly rounded FP32 dot product of
   * x_t with this vector (a gated shared expert); NULL: weight 1. */
  const float* shared_expert_gate;
  /* 0: router_bias shifts the logits that decide both the selection and the
   * weights.  1: the bias steers the selection only and the weights come
   * from the unbiased logits of the selected experts (a load-balancing
   * correction that leaves the mixture weights as the router computes them). */
  int32_t bias_select;
} moe_layer;

typedef struct {
  /* 0 (default): BF16 activations, the exact chain.  1: the NVFP4 W4A4
   * lever (prefill only, NVFP4 routed experts): activations and SwiGLU
   * outputs re-quantised to NVFP4 16-element blocks before the projections
   * (DGPP forum, page 5 weekly update: W4A4 prefill is opt-in).  2: the same
   * lever for MXFP4 routed experts, with MXFP4 activations (32-element
   * blocks, E8M0 scales; the rule of moe_quantize_act_mxfp4). */
  int32_t act_quant;
  /* 0 (default): FP32 per-expert partials.  1: the down projection's
   * partials are rounded to BF16 before the weighted sum (DGPP README
   * "Execution and performance", engine.prefill_bf16_partials, a lever that
   * halves the partials' bytes and is not bitwise the default chain). */
  int32_t bf16_partials;
  /* 0 (default: 2 s): every bounded device-side wait of the prefill
   * kernels gives up after this many microseconds and reports
   * MOE_ERR_DEVICE_TIMEOUT through moe_check. */
  int32_t wait_limit_us;
  /* 0 (default): the exact chain.  1: the fold-scales lever (prefill only;
   * DGPP README "Execution and performance", engine.prefill_fold_scales):
   * int8 g64, FP8 b128 and int4 g128 weights, routed or shared, enter the
   * grouped GEMMs as BF16 values bf16(fl32(code * group scale)) against
   * plain BF16 activations, with one FP32 accumulator across K instead of
   * one per scale group.  Not bitwise the default chain.  NVFP4, MXFP4 and
   * int4 g64 weights already reach the MMA with their scales folded exactly
   * and are unchanged by it.  The decode entry points return
   * MOE_ERR_UNSUPPORTED when it is set. */
  int32_t fold_scales;
  /* 0 (default): the exact chain.  1: the FP8-activation lever (prefill
   * only; DGPP README "Execution and performance", engine.prefill_fp8_gemm):
   * FP8 b128 experts, routed or shared, meet per-token 1x128 E4M3
   * activations on FP8 tensor cores: x, and h after its BF16 rounding, are
   * quantised per 128-element block with scale fl32(amax / 448) and codes
   * e4m3_rne_sat(fl32(v / scale)), and each 128-K group's products are scaled
   * by weight scale x activation scale in FP32.  Not bitwise the default
   * chain.  For FP8 b128 experts it takes precedence over fold_scales; other
   * formats are unchanged by it.  The decode entry points return
   * MOE_ERR_UNSUPPORTED when it is set. */
  int32_t fp8_act;
  int32_t reserved[3];       /* must be zero */
} moe_options;

/* Largest token count moe_decode_forward accepts. */
#define MOE_DECODE_MAX_TOKENS 8

/* Human-readable name of a status code (static string, never NULL).
 * Interface convenience, no passage: the pages define no error reporting. */
const char* moe_status_string(int32_t status);

/*
 * Bytes of device workspace needed by moe_route / moe_decode_forward /
 * moe_prefill_forward for up to max_tokens tokens (0 if the layer or options
 * are invalid).  The workspace must be 256-byte aligned and initialised once
 * with moe_workspace_init before its first use; the library leaves it
 * re-usable after every call.  It holds the routing results, the per-expert
 * activations h and the FP32 partials (DGPP README "Execution and
 * performance", engine.prefill_bf16_partials: partials summed in FP32 by
 * default), so that the caller owns every device buffer.
 */
size_t moe_workspace_size(const moe_layer* layer, int32_t max_tokens, const moe_options* opts);

/* Zero the workspace control block (stream-ordered).  Call once per workspace.
 * Interface convenience, no passage. */
int32_t moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Router and dispatch only (DGPP README "Execution and performance",
 * engine.expert_tile_list: routed segments per expert).
 *   logits     l[t, e] = fl32( sum_h x[t, h] * router_w[e, h] ), the correctly
 *              rounded FP32 dot product, then fl32(l + router_bias[e]) if a bias
 *              is given.  Selection and weights use these exact logits.  For
 *              T <= MOE_DECODE_MAX_TOKENS every expert's logit is computed
 *              exactly and the workspace's logits array (moe_workspace_layout)
 *              holds all of them; for larger T the router finds them with an
 *              FP32 pass and a rigorous error bound, then recomputes exactly
 *              every expert that can still reach the top-k, so those experts
 *              hold l[t, e] and the others -inf.
 *   topk_idx   [T, k] i32: experts by logit descending, ties to the lower id.
 *   topk_w     [T, k] f32: exp(l_j - l_0) / sum_i exp(l_i - l_0) over the selected.
 *   expert_cnt [E] i32 pairs per expert; expert_off [E+1] i32 exclusive scan.
 *   pair_list  [T*k] i32: pair ids p = t*k + j grouped by expert, ascending p
 *              within an expert (a stable counting sort).
 * Any of the output pointers may be NULL (that output is not written).
 * T: 1 .. max_tokens of the workspace.
 */
int32_t moe_route(const moe_layer* layer, const void* x /* device bf16 [T, H] */, int32_t T,
                  int32_t* topk_idx, float* topk_w, int32_t* expert_cnt, int32_t* expert_off,
                  int32_t* pair_list, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Whole layer for decode-sized batches, T = 1 .. MOE_DECODE_MAX_TOKENS:
 *   y[t] = bf16( sum_j topk_w[t, j] * down_e( h_tj ) + shared(x_t) ),
 *   h_tj = bf16( silu(gate_e x_t) * (up_e x_t) ),  e = topk_idx[t, j],
 * with the shared expert (weight 1, no gate) added when present.  Weights are
 * read in their checkpoint formats and decoded in registers (DGPP README
 * intro bullet "Serves checkpoints as published": no dequantized copy; forum
 * post 15 "Lossless bf12": decode streams the weights at the memory line
 * rate); activations BF16, accumulation and partials FP32, h and y rounded
 * to BF16 once (forum post 1, quantisation table: activations stay BF16;
 * README "Execution and performance", engine.prefill_bf16_partials and
 * engine.prefill_fold_scales off by default).  Routing outputs are left in
 * the workspace (see moe_workspace_layout; logits as for moe_route).  opts may be NULL (defaults);
 * act_quant must be 0 here (MOE_ERR_UNSUPPORTED otherwise).
 */
int32_t moe_decode_forward(const moe_layer* layer, const void* x /* device bf16 [T, H] */, int32_t T,
                           void* y /* device bf16 [T, H] */, const moe_options* opts, void* ws, size_t ws_bytes,
                           moe_stream_t stream);

/*
 * The expert half of moe_decode_forward on routing the caller computed: for
 * T = 1 .. MOE_DECODE_MAX_TOKENS tokens and the caller's top-k choice
 * (topk_idx device i32 [T, k], expert ids; topk_w device f32 [T, k], mixture
 * weights), y[t] = bf16( sum_j topk_w[t, j] * down_e( h_tj ) + shared(x_t) )
 * with the same expert kernels, dispatch (a stable counting sort of the pairs
 * by expert; DGPP README "Execution and performance", engine.expert_tile_list)
 * and rounding points.  This serves layers whose router is not the softmax
 * top-k of moe_route (a sigmoid or group-limited router, or routing decided
 * elsewhere); router_w and router_bias are not read.  An id outside
 * [0, n_experts) is reported as MOE_ERR_DEVICE_BAD_INDEX through moe_check and
 * its pair is left out (y is then undefined).  Other arguments, checks and
 * results are those of moe_decode_forward.
 */
int32_t moe_experts_forward(const moe_layer* layer, const void* x /* device bf16 [T, H] */, int32_t T,
                            const int32_t* topk_idx, const float* topk_w, void* y /* device bf16 [T, H] */,
                            const moe_options* opts, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Whole layer for any T >= 1 (prefill), same result definition as
 * moe_decode_forward; expert projections run as grouped GEMMs over a compact
 * tile list of the routed segments (DGPP README "Execution and performance":
 * engine.expert_tile_list, engine.expert_gemm_pair), with FP32 partials and
 * a combine pass.  Supported: every routed and shared format, hidden, inter
 * and shared inter multiples of 128 (other shapes return MOE_ERR_UNSUPPORTED
 * before any launch); a shared expert runs as a dense GEMM over all T tokens.
 * MXFP4 and int4 g64 weights are folded into f16 relative to their row's
 * largest block scale: exact while a row's block scales span at most 2^23
 * (MXFP4) / 2^24 (int4); blocks further below are rounded to f16's subnormal
 * grid or dropped (weights under 2^-21 times the row's largest block scale).
 * int8 g64, FP8 b128 and int4 g128 weights enter the MMA unscaled and each
 * scale group is applied in FP32.  opts->act_quant selects the W4A4 lever
 * (DGPP forum, page 5 weekly update: W4A4 prefill is opt-in): 1 for NVFP4
 * routed experts (x and h quantised to NVFP4 16-element blocks, the rule of
 * moe_quantize_act_nvfp4), 2 for MXFP4 routed experts (MXFP4 32-element
 * blocks, the rule of moe_quantize_act_mxfp4); the projections then run as
 * block-scaled FP4 GEMMs.  It needs no shared expert, hidden and inter
 * multiples of 256 and 16-byte aligned scale arrays.  opts->fold_scales and
 * opts->fp8_act select the other two prefill levers (see moe_options); each
 * changes only the experts of its formats and needs no other condition.
 * Routing outputs are left in the workspace; in its logits array only the
 * experts the router recomputed exactly (every selected one among them) hold
 * their FP32 logit, the others hold -inf.
 */
int32_t moe_prefill_forward(const moe_layer* layer, const void* x /* device bf16 [T, H] */, int32_t T,
                            void* y /* device bf16 [T, H] */, const moe_options* opts, void* ws, size_t ws_bytes,
                            moe_stream_t stream);

/*
 * Interface convenience for measurement, no passage:
 * moe_prefill_forward that also records up to eight CUDA events on `stream`
 * (events[i] a cudaEvent_t or NULL): [0] before the first kernel, [1] after
 * the approximate router logits, [2] after top-k, [3] after the dispatch
 * index, [4] after the gate/up GEMM, [5] after the h conversion, [6] after
 * the down GEMM, [7] after the combine.  Inside a stream capture the records
 * become event-record nodes.  For per-kernel timing only.
 */
int32_t moe_prefill_forward_timed(const moe_layer* layer, const void* x, int32_t T, void* y,
                                  const moe_options* opts, void* ws, size_t ws_bytes, moe_stream_t stream,
                                  void* const* events);

/*
 * Interface convenience for measurement, no passage:
 * moe_decode_forward that also records four CUDA events on `stream`: before
 * the router kernel, after it, after the gate/up kernel and after the down +
 * combine kernel (events[i] is a cudaEvent_t; any entry may be NULL).  For
 * per-kernel timing; the event records between launches stop the kernels
 * from overlapping their prologues, so whole-layer timing should use
 * moe_decode_forward.
 */
int32_t moe_decode_forward_timed(const moe_layer* layer, const void* x, int32_t T, void* y,
                                 const moe_options* opts, void* ws, size_t ws_bytes, moe_stream_t stream,
                                 void* const* events);

/*
 * moe_decode_forward without a caller-supplied workspace, for callers that
 * cannot allocate device memory: code running inside a host framework that
 * owns every device buffer and gives plugins no allocator, or a serving loop
 * that forbids allocations once it has started.  (The DGPP pages have no
 * counterpart; this is an interface convenience of this library.)
 *  - The workspace is a fixed 32 MiB array in the library's device memory;
 *    every GPU that loads the library holds it until the process exits.  A
 *    layer and T whose moe_workspace_size exceeds 32 MiB are rejected with
 *    MOE_ERR_WORKSPACE.  Every argument check of moe_decode_forward runs
 *    first: a rejected call touches neither the array nor the device.
 *  - Every call clears, on `stream`, the counters of the array that must
 *    start at zero.  The first call on a device also clears the array's
 *    device-side error word; make that first call before any stream capture.
 *  - Every call shares the one array, so calls that overlap on the GPU, from
 *    any stream or thread, race: serialise them.
 *  - A device-side error (see moe_check) stays in the array's error word
 *    until moe_check(NULL, 0, stream) reads and clears it.
 *  - The routing results stay in the array; they are not exposed.
 *  - After a device reset the array is looked up again and the next call
 *    counts as the first on that device.
 * Other arguments, checks and results are those of moe_decode_forward.
 */
int32_t moe_decode_forward_noalloc(const moe_layer* layer, const void* x /* device bf16 [T, H] */, int32_t T,
                                   void* y /* device bf16 [T, H] */, const moe_options* opts, moe_stream_t stream);

/*
 * Launch plan of a decode call (moe_decode_forward) for a layer, T tokens and
 * `num_sms` streaming multiprocessors: how each kernel splits the reduction
 * dimension K of a 16-row weight tile between warps, and the shared memory
 * it stages.  Host only: no device access, no launch; the layer's pointers
 * are checked like moe_decode_forward's but never dereferenced.
 *
 * A K split changes no result: every tile is summed in fixed blocks added in
 * block order whatever the split (DGPP README "Accuracy and correctness":
 * deterministic, batch-invariant output).  Errors: MOE_ERR_INVALID_ARG (null
 * out, T outside 1 .. MOE_DECODE_MAX_TOKENS, num_sms < 1, invalid layer),
 * MOE_ERR_UNSUPPORTED (the layer's staging does not fit in shared memory).
 */
typedef struct {
  int32_t gu_slices;        /* K slices of a routed gate/up tile in the first wave of tasks */
  int32_t gu_slices_shared; /* K slices of a shared-expert gate/up tile */
  int32_t gu_slices_tail;   /* K slices of a routed gate/up tile beyond the first wave */
  int32_t gu_tail_cap;      /* most routed tiles split that way */
  int32_t dn_slices;        /* K slices of a down tile */
  int32_t dn_segs;          /* expert segments the down kernel stages at once */
  int32_t gu_ctas_per_sm;   /* gate/up CTAs (of 8 warps) per SM */
  int32_t reserved;
  size_t gu_smem;           /* dynamic shared memory per gate/up CTA, bytes */
  size_t dn_smem;           /* dynamic shared memory per down CTA, bytes */
  size_t gu_split_blocks;   /* most K-block sums the gate/up kernel may store */
  size_t dn_split_blocks;   /* most K-block sums the down kernel may store */
  size_t split_block_capacity; /* K-block sums the workspace holds per kernel */
} moe_decode_plan_info;

int32_t moe_decode_plan(const moe_layer* layer, int32_t T, int32_t num_sms, moe_decode_plan_info* out);

/*
 * Read and clear the device-side error flag of a workspace.  Synchronises
 * `stream` (this is the one call that blocks).  Returns MOE_OK,
 * MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_DEVICE_BAD_INDEX (the first device-side
 * error since the last read), MOE_ERR_WORKSPACE for a null or short ws,
 * MOE_ERR_CUDA if the synchronisation or the copy fails.  ws = NULL with
 * ws_bytes = 0 reads the fixed array of moe_decode_forward_noalloc on the
 * current device (MOE_OK if no such call has run there).  Interface
 * convenience, no passage: the pages define no error reporting; kernels
 * never trap, so errors surface here.
 */
int32_t moe_check(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Byte offsets, within the workspace, of the routing results a forward call leaves there
 * (interface convenience for inspection and testing, no passage). */
typedef struct {
  size_t logits;      /* f32 [T, E] */
  size_t topk_idx;    /* i32 [T, k] */
  size_t topk_w;      /* f32 [T, k] */
  size_t expert_cnt;  /* i32 [E] */
  size_t expert_off;  /* i32 [E + 1] */
  size_t pair_list;   /* i32 [T * k] */
  size_t total;       /* workspace bytes for this max_tokens */
  /* moe_prefill_forward with act_quant = 1 (2): the NVFP4 (MXFP4) codes and E4M3 (E8M0) block
   * scales of each pair's SwiGLU output h, by sorted position (position pos holds pair
   * pair_list[pos]) */
  size_t h_codes;     /* u8 [T * k, I / 2], low nibble = even column */
  size_t h_scales;    /* u8 [T * k, I / 16] (act_quant 1) or [T * k, I / 32] (act_quant 2) */
} moe_ws_layout;

int32_t moe_workspace_layout(const moe_layer* layer, int32_t max_tokens, const moe_options* opts,
                             moe_ws_layout* out);

/*
 * Decode rows [row0, row0 + nrows) of expert `expert` of a weight stack to
 * FP32 (format decode, the step every projection kernel performs in
 * registers; exposed for bit-exact checking).  out[r, k] = fl32(exact value):
 * e2m1 * e4m3 * ts (NVFP4), e2m1 * 2^(c-127) (MXFP4), q * s (int4/int8 g64),
 * e4m3 * s (FP8 b128).  out: device f32 [nrows, K].
 */
int32_t moe_dequantize(int32_t fmt, const moe_qweight* w, int32_t N, int32_t K, int32_t expert, int32_t row0,
                       int32_t nrows, float* out, moe_stream_t stream);

/*
 * NVFP4 activation quantizer of the W4A4 lever, per 16-element block of each
 * row: s = e4m3_rne_sat( fl32(amax / 6) ), code = e2m1_rne_sat( fl32(a / s) ),
 * tensor scale 1; a block whose scale rounds to zero gets zero codes.
 *   x: device bf16 [rows, K]; codes: device u8 [rows, K/2] (low nibble = even k);
 *   scales: device u8 [rows, K/16] (E4M3).  K a multiple of 16.
 */
int32_t moe_quantize_act_nvfp4(const void* x, int32_t rows, int32_t K, uint8_t* codes, uint8_t* scales,
                               moe_stream_t stream);

/*
 * MXFP4 activation quantizer of the W4A4 lever (act_quant = 2), per
 * 32-element block of each row: the block exponent e is the smallest integer
 * with 6 * 2^e >= amax (e = 0 for an all-zero block), its E8M0 scale code
 * e + 127 clamped to [0, 254]; code = e2m1_rne_sat( a / 2^e ) (the rule of
 * the MXFP4 checkpoints' scales, DGPP forum post 1 quantisation table and the
 * MXFP4 config's scale = 2^ceil(log2(amax / 6))).
 *   x: device bf16 [rows, K]; codes: device u8 [rows, K/2] (low nibble = even k);
 *   scales: device u8 [rows, K/32] (E8M0).  K a multiple of 32.
 */
int32_t moe_quantize_act_mxfp4(const void* x, int32_t rows, int32_t K, uint8_t* codes, uint8_t* scales,
                               moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QMOE_MOE_H */
