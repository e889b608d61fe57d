// Host side of the C ABI (include/moe.h): argument validation, workspace
// layout, tiling choices and kernel launches.  Nothing here allocates device
// memory; every buffer belongs to the caller.
#include <cstddef>
#include <cstring>

#include "kernels.cuh"

using namespace qmoe;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool valid_fmt(int f) { return f >= MOE_FMT_NVFP4 && f <= MOE_FMT_INT4_G128; }

// Shape rules of the formats and of the kernels (16-byte units along K,
// 128-row FP8 scale blocks).
bool shape_ok(int fmt, int N, int K) {
  if (N <= 0 || K <= 0 || N % 16 || K % 128) return false;
  if (fmt == MOE_FMT_FP8_B128 && (N % 128 || K % 128)) return false;
  return true;
}

struct Layout {
  size_t ctrl, logits, topk_idx, topk_w, cnt, off, pair, act, h, hs, P, S, approx, sgate, gu_part, gu_cnt,
      dn_part, dn_cnt;
  // prefill path
  size_t xg, xsig, xnorm, wnorm, hist, pos_of, tiles, h16, hsig, xq, xsf, xqg, xsfg, hq, hsf, rw_hi, rw_lo;
  size_t xs16, hs16, hssig;  // the shared expert's operands in prefill
  int max_tiles;
  size_t total;
};

Layout make_layout(const moe_layer* L, int maxT) {
  Layout o;
  size_t at = 0;
  auto take = [&](size_t bytes) {
    size_t p = at;
    at = align_up(at + bytes);
    return p;
  };
  const size_t T = (size_t)maxT, E = (size_t)L->n_experts, k = (size_t)L->top_k, H = (size_t)L->hidden,
               I = (size_t)L->inter, Is = (size_t)(L->shared_fmt ? L->shared_inter : 0);
  o.ctrl = take(sizeof(Ctrl));
  o.logits = take(T * E * 4);
  o.topk_idx = take(T * k * 4);
  o.topk_w = take(T * k * 4);
  o.cnt = take(E * 4);
  o.off = take((E + 1) * 4);
  o.pair = take(T * k * 4);
  o.act = take(E * 4);
  o.h = take(T * k * I * 2);
  o.hs = take(T * Is * 2 + 16);
  o.P = take(T * k * H * 4);
  o.S = take(T * H * 4 + 16);
  o.approx = take(T * E * 4);
  o.sgate = take(T * 4);
  // block sums of tiles split along K (at most kMaxSplitBlocks entries)
  const size_t act_max = T * k < E ? T * k : E;
  const size_t gu_tiles = act_max * (I / 16) + Is / 16, dn_tiles = (act_max + 1) * (H / 16);
  o.gu_part = take((size_t)kMaxSplitBlocks * 32 * 8 * 4);
  o.gu_cnt = take(gu_tiles * 4);
  o.dn_part = take((size_t)kMaxSplitBlocks * 32 * 4 * 4);
  o.dn_cnt = take(dn_tiles * 4);
  const size_t nchunk = (T + kPfChunk - 1) / kPfChunk;
  o.max_tiles = (int)(T * k / kPfTokTile + E + 1);
  o.xg = take(T * k * H * 2);
  o.xsig = take(T * 4);
  o.xnorm = take(T * 4);
  o.wnorm = take(E * 4);
  o.hist = take(nchunk * E * 4);
  o.pos_of = take(T * k * 4);
  o.tiles = take((size_t)o.max_tiles * 8);
  o.h16 = take(T * k * I * 2);
  o.hsig = take(T * k * 4);
  o.xq = take(T * H / 2);
  o.xsf = take(T * H / 16);
  o.xqg = take(T * k * H / 2);
  o.xsfg = take(T * k * H / 16);
  o.hq = take(T * k * I / 2);
  o.hsf = take(T * k * I / 16);
  o.rw_hi = take(E * H * 2);
  o.rw_lo = take(E * H * 2);
  o.xs16 = take(Is ? T * H * 2 : 0);
  o.hs16 = take(T * Is * 2);
  o.hssig = take(Is ? T * 4 : 0);
  o.total = at;
  return o;
}

int32_t check_qweight(const moe_qweight& w, int fmt, int N, int K) {
  if (!w.data || !w.scales) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w.data) || !aligned4(w.scales)) return MOE_ERR_MISALIGNED;
  if (fmt == MOE_FMT_NVFP4) {
    if (!w.tensor_scale) return MOE_ERR_INVALID_ARG;
    if (!aligned4(w.tensor_scale)) return MOE_ERR_MISALIGNED;
  }
  if (!shape_ok(fmt, N, K)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int32_t check_layer(const moe_layer* L) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (L->hidden <= 0 || L->inter <= 0 || L->n_experts <= 0 || L->top_k <= 0) return MOE_ERR_INVALID_ARG;
  if (L->n_experts > 1024 || L->top_k > 16 || L->top_k > L->n_experts) return MOE_ERR_UNSUPPORTED;
  if (!valid_fmt(L->fmt)) return MOE_ERR_INVALID_ARG;
  if (!L->router_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(L->router_w)) return MOE_ERR_MISALIGNED;
  if (L->router_bias && !aligned4(L->router_bias)) return MOE_ERR_MISALIGNED;
  const int H = L->hidden, I = L->inter;
  int32_t st;
  if ((st = check_qweight(L->gate, L->fmt, I, H)) != MOE_OK) return st;
  if ((st = check_qweight(L->up, L->fmt, I, H)) != MOE_OK) return st;
  if ((st = check_qweight(L->down, L->fmt, H, I)) != MOE_OK) return st;
  if (L->shared_fmt != MOE_FMT_NONE) {
    if (!valid_fmt(L->shared_fmt)) return MOE_ERR_INVALID_ARG;
    const int Is = L->shared_inter;
    if (Is <= 0) return MOE_ERR_INVALID_ARG;
    if ((st = check_qweight(L->shared_gate, L->shared_fmt, Is, H)) != MOE_OK) return st;
    if ((st = check_qweight(L->shared_up, L->shared_fmt, Is, H)) != MOE_OK) return st;
    if ((st = check_qweight(L->shared_down, L->shared_fmt, H, Is)) != MOE_OK) return st;
  }
  if (L->shared_expert_gate) {
    if (L->shared_fmt == MOE_FMT_NONE) return MOE_ERR_INVALID_ARG;  // a gate needs a shared expert
    if (!aligned16(L->shared_expert_gate)) return MOE_ERR_MISALIGNED;
  }
  if (L->bias_select != 0 && L->bias_select != 1) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int32_t check_options(const moe_options* o) {
  if (!o) return MOE_OK;
  if (o->act_quant < 0 || o->act_quant > 2) return MOE_ERR_INVALID_ARG;
  if (o->bf16_partials != 0 && o->bf16_partials != 1) return MOE_ERR_INVALID_ARG;
  if (o->wait_limit_us < 0) return MOE_ERR_INVALID_ARG;
  if (o->fold_scales != 0 && o->fold_scales != 1) return MOE_ERR_INVALID_ARG;
  if (o->fp8_act != 0 && o->fp8_act != 1) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i)
    if (o->reserved[i] != 0) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Device-wait limit of the prefill kernels in nanoseconds (2 s unless the options set one).
uint64_t wait_limit_ns(const moe_options* o) {
  return (o && o->wait_limit_us > 0) ? (uint64_t)o->wait_limit_us * 1000ull : 2000000000ull;
}

int32_t check_ws(const moe_layer* L, int maxT, void* ws, size_t ws_bytes) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_MISALIGNED;
  if (ws_bytes < make_layout(L, maxT).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

QW qw(const moe_qweight& w, int fmt) {
  QW q;
  q.data = static_cast<const uint8_t*>(w.data);
  q.scales = static_cast<const uint8_t*>(w.scales);
  q.ts = fmt == MOE_FMT_NVFP4 ? w.tensor_scale : nullptr;
  return q;
}

RouteBufs route_bufs(const Layout& lo, void* ws) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  RouteBufs r;
  r.ctrl = reinterpret_cast<Ctrl*>(b + lo.ctrl);
  r.logits = reinterpret_cast<float*>(b + lo.logits);
  r.topk_idx = reinterpret_cast<int32_t*>(b + lo.topk_idx);
  r.topk_w = reinterpret_cast<float*>(b + lo.topk_w);
  r.cnt = reinterpret_cast<int32_t*>(b + lo.cnt);
  r.off = reinterpret_cast<int32_t*>(b + lo.off);
  r.pair = reinterpret_cast<int32_t*>(b + lo.pair);
  r.act = reinterpret_cast<int32_t*>(b + lo.act);
  return r;
}

// The largest token count a workspace of ws_bytes supports for this layer.
int ws_max_tokens(const moe_layer* L, size_t ws_bytes) {
  int lo = 0, hi = 1;
  while (hi < (1 << 24) && make_layout(L, hi).total <= ws_bytes) { lo = hi; hi *= 2; }
  while (hi - lo > 1) {
    int mid = lo + (hi - lo) / 2;
    if (make_layout(L, mid).total <= ws_bytes) lo = mid; else hi = mid;
  }
  return lo;
}

int32_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// K slices per 16-row tile: split while the tasks stay below ~2 per resident
// warp, the slices divide the accumulation blocks of both formats and the
// stored block sums fit the partial buffer.  The result of a tile does not
// depend on the split (blocks are always added in block order).
int choose_slices(int K_r, int fmt_r, long tiles_r, int K_s, int fmt_s, long tiles_s, int warps) {
  const int Br = dec_blocks(fmt_r, K_r), Bs = fmt_s ? dec_blocks(fmt_s, K_s) : Br;
  if (tiles_r * Br + tiles_s * Bs > kMaxSplitBlocks) return 1;
  int S = 1;
  while (Br % (2 * S) == 0 && Bs % (2 * S) == 0 && (tiles_r + tiles_s) * 2 * S * 4 <= 5L * warps) S *= 2;
  return S;
}

cudaError_t launch_expert(int fmt, int sfmt, bool down, const ExpertArgs& a, size_t smem, cudaStream_t s) {
  switch (fmt) {
    case MOE_FMT_NVFP4: return launch_expert_nvfp4(sfmt, down, a, smem, s);
    case MOE_FMT_MXFP4: return launch_expert_mxfp4(sfmt, down, a, smem, s);
    case MOE_FMT_INT4_G64: return launch_expert_int4(sfmt, down, a, smem, s);
    case MOE_FMT_INT8_G64: return launch_expert_int8(sfmt, down, a, smem, s);
    case MOE_FMT_FP8_B128: return launch_expert_fp8(sfmt, down, a, smem, s);
    case MOE_FMT_INT4_G128: return launch_expert_int4g128(sfmt, down, a, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

RouterArgs router_args(const moe_layer* L, const Layout& lo, void* ws, const void* x, int T) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  RouterArgs ra;
  std::memset(&ra, 0, sizeof(ra));
  ra.H = L->hidden; ra.E = L->n_experts; ra.k = L->top_k; ra.T = T;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  ra.wpr = router_warps_per_row(L->hidden, L->n_experts, sms);
  ra.x = static_cast<const uint16_t*>(x);
  ra.w = L->router_w;
  ra.bias = L->router_bias;
  ra.rb = route_bufs(lo, ws);
  ra.approx = reinterpret_cast<float*>(b + lo.approx);
  ra.bias_select = L->bias_select;
  ra.sgate_w = L->shared_fmt ? L->shared_expert_gate : nullptr;
  ra.sgate = reinterpret_cast<float*>(b + lo.sgate);
  return ra;
}


// Launch plan of a decode call: K splits, staging strides and shared-memory
// sizes, from the layer's shapes and formats and the SM count (host only).
struct DecodePlan {
  int gu_slices, gu_slices_s, gu_slices_t, gu_tail_cap, dn_slices, dn_segs;
  int xs_tok_stride, hs_tok_stride;
  size_t smem_gu, smem_dn;
  long gu_blocks, dn_blocks;  // most K-block sums each kernel may store
};

int32_t plan_decode(const moe_layer* L, int T, int sms, DecodePlan* p) {
  const int H = L->hidden, I = L->inter, Is = L->shared_fmt ? L->shared_inter : 0;
  const int warps = sms * 16;  // resident warps the expert kernels aim for
  const long act = (long)T * L->top_k < L->n_experts ? (long)T * L->top_k : L->n_experts;
  const int Br = dec_blocks(L->fmt, H);
  p->gu_slices = choose_slices(H, L->fmt, act * (I / 16), H, L->shared_fmt, Is / 16, warps);
  p->dn_slices = choose_slices(I, L->fmt, act * (H / 16), Is, L->shared_fmt, Is ? H / 16 : 0, warps);
  // shared-expert tiles of gate/up: split K until a task carries no more bytes
  // than a routed one (both formats' blocks permitting), so no task outlasts the rest
  const int Sr = p->gu_slices;
  p->gu_slices_s = Sr;
  long shared_blocks = 0;
  if (L->shared_fmt) {
    const double br = (double)(data_bytes(L->fmt, I, H) + scale_bytes(L->fmt, I, H)) / I / Sr;
    const double bs = (double)(data_bytes(L->shared_fmt, Is, H) + scale_bytes(L->shared_fmt, Is, H)) / Is;
    const int Bs = dec_blocks(L->shared_fmt, H);
    int Ss = 1;
    while (bs / Ss > 1.15 * br && Bs % (2 * Ss) == 0) Ss *= 2;
    const long blocks = (Sr > 1 ? act * (I / 16) * (long)Br : 0) + (long)(Is / 16) * Bs;
    p->gu_slices_s = blocks <= kMaxSplitBlocks ? Ss : 1;
    if (p->gu_slices_s > 1) shared_blocks = (long)(Is / 16) * Bs;
  }
  // routed tiles beyond the first wave of tasks: up to 8 slices (the kernel
  // decides how many tiles from the active-expert count); with unsplit head
  // tiles only the tail's block sums are stored, after which come the shared ones
  int St = Sr;
  while (St < 8 && Br % (2 * St) == 0) St *= 2;
  p->gu_slices_t = St;
  const long cap = Sr > 1 ? act * (I / 16) : (kMaxSplitBlocks - shared_blocks) / Br;
  p->gu_tail_cap = (int)(cap < 0 ? 0 : cap);
  p->gu_blocks = (Sr > 1 ? act * (I / 16) : (St > Sr ? p->gu_tail_cap : 0)) * (long)Br + shared_blocks;
  p->dn_blocks = p->dn_slices > 1 ? act * (H / 16) * (long)dec_blocks(L->fmt, I) +
                                        (L->shared_fmt ? (long)(H / 16) * dec_blocks(L->shared_fmt, Is) : 0)
                                  : 0;
  // token rows staged with a stride of 16 banks: the MMA operand loads of two
  // rows in one quarter warp fall on disjoint banks
  p->xs_tok_stride = H + 32;
  const int Kmax = Is > I ? Is : I;
  p->hs_tok_stride = Kmax + 32;

  const size_t warps_cta = kExpertThreads / 32;
  const int gu_st = gu_stages(T <= kGuSmallT ? 3 : 2);
  p->smem_gu = (size_t)T * p->xs_tok_stride * 2 + warps_cta * gu_st * dec_stage_bytes(2);
  // the down kernel stages up to kMaxDnSegs expert segments of h at once, as
  // many as keep two CTAs per SM
  const size_t seg_bytes = (size_t)(MOE_DECODE_MAX_TOKENS + 1) * p->hs_tok_stride * 2;
  const size_t rings_dn = warps_cta * kStagesDN * dec_stage_bytes(1);
  const size_t half_sm = 113 * 1024;
  const int segs = half_sm > rings_dn ? (int)((half_sm - rings_dn) / seg_bytes) : 1;
  p->dn_segs = segs < 1 ? 1 : (segs > kMaxDnSegs ? kMaxDnSegs : segs);
  p->smem_dn = (size_t)p->dn_segs * seg_bytes + rings_dn;
  if (p->smem_gu > 227 * 1024 || p->smem_dn > 227 * 1024) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int32_t decode_forward_impl(const moe_layer* L, const void* x, int32_t T, void* y, const moe_options* opts, void* ws,
                            size_t ws_bytes, cudaStream_t stream, void* const* events,
                            const int32_t* ext_idx = nullptr, const float* ext_w = nullptr) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (events) cudaStreamIsCapturing(stream, &cap);
  auto mark = [&](int i) {
    if (!events || !events[i]) return;
    cudaEvent_t ev = static_cast<cudaEvent_t>(events[i]);
    // inside a stream capture an external record becomes an event-record node
    if (cap == cudaStreamCaptureStatusActive) cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal);
    else cudaEventRecord(ev, stream);
  };
  const int maxT = ws_max_tokens(L, ws_bytes);
  const Layout lo = make_layout(L, maxT);
  uint8_t* b = static_cast<uint8_t*>(ws);
  const int H = L->hidden, I = L->inter, Is = L->shared_fmt ? L->shared_inter : 0;
  const RouterArgs ra = router_args(L, lo, ws, x, T);

  ExpertArgs ea;
  std::memset(&ea, 0, sizeof(ea));
  ea.H = H; ea.I = I; ea.E = L->n_experts; ea.k = L->top_k; ea.T = T;
  ea.fmt = L->fmt; ea.sfmt = L->shared_fmt; ea.Is = Is;
  ea.x = ra.x;
  ea.gate = qw(L->gate, L->fmt); ea.up = qw(L->up, L->fmt); ea.down = qw(L->down, L->fmt);
  if (L->shared_fmt) {
    ea.sgate = qw(L->shared_gate, L->shared_fmt);
    ea.sup = qw(L->shared_up, L->shared_fmt);
    ea.sdown = qw(L->shared_down, L->shared_fmt);
  }
  ea.rb = ra.rb;
  ea.h = reinterpret_cast<uint16_t*>(b + lo.h);
  ea.hs = reinterpret_cast<uint16_t*>(b + lo.hs);
  ea.P = reinterpret_cast<float*>(b + lo.P);
  ea.S = reinterpret_cast<float*>(b + lo.S);
  ea.gu_part = reinterpret_cast<float*>(b + lo.gu_part);
  ea.gu_cnt = reinterpret_cast<uint32_t*>(b + lo.gu_cnt);
  ea.dn_part = reinterpret_cast<float*>(b + lo.dn_part);
  ea.dn_cnt = reinterpret_cast<uint32_t*>(b + lo.dn_cnt);
  ea.y = static_cast<uint16_t*>(y);
  ea.shared_g = ra.sgate_w ? ra.sgate : nullptr;
  ea.p_bf16 = (opts && opts->bf16_partials) ? 1 : 0;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
  DecodePlan pl;
  const int32_t pst = plan_decode(L, T, sms, &pl);
  if (pst != MOE_OK) return pst;
  ea.gu_slices = pl.gu_slices;
  ea.gu_slices_s = pl.gu_slices_s;
  ea.gu_slices_t = pl.gu_slices_t;
  ea.gu_tail_cap = pl.gu_tail_cap;
  ea.dn_slices = pl.dn_slices;
  ea.dn_segs = pl.dn_segs;
  ea.xs_tok_stride = pl.xs_tok_stride;
  ea.hs_tok_stride = pl.hs_tok_stride;
  const size_t smem_gu = pl.smem_gu, smem_dn = pl.smem_dn;

  mark(0);
  cudaError_t err = ext_idx ? launch_dispatch_ext(ra, ext_idx, ext_w, stream) : launch_router_decode(ra, stream);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  mark(1);
  err = launch_expert(L->fmt, L->shared_fmt, false, ea, smem_gu, stream);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  mark(2);
  err = launch_expert(L->fmt, L->shared_fmt, true, ea, smem_dn, stream);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  err = launch_combine_decode(ea, stream);
  mark(3);
  return cuda_status(err);
}

PrefillArgs prefill_args(const moe_layer* L, const Layout& lo, void* ws, const void* x, int T, void* y) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  PrefillArgs a;
  std::memset(&a, 0, sizeof(a));
  a.H = L->hidden; a.I = L->inter; a.E = L->n_experts; a.k = L->top_k; a.T = T;
  a.fmt = L->fmt;
  a.x = static_cast<const uint16_t*>(x);
  a.rw = L->router_w;
  a.bias = L->router_bias;
  a.gate = qw(L->gate, L->fmt); a.up = qw(L->up, L->fmt); a.down = qw(L->down, L->fmt);
  a.rb = route_bufs(lo, ws);
  a.xg = reinterpret_cast<uint16_t*>(b + lo.xg);
  a.xsig = reinterpret_cast<int32_t*>(b + lo.xsig);
  a.xnorm = reinterpret_cast<float*>(b + lo.xnorm);
  a.wnorm = reinterpret_cast<float*>(b + lo.wnorm);
  a.hist = reinterpret_cast<int32_t*>(b + lo.hist);
  a.pos_of = reinterpret_cast<int32_t*>(b + lo.pos_of);
  a.tiles = reinterpret_cast<int2*>(b + lo.tiles);
  a.max_tiles = lo.max_tiles;
  a.h = reinterpret_cast<uint16_t*>(b + lo.h);
  a.h_amax = nullptr;  // the h conversion finds each row's maximum itself
  a.h16 = reinterpret_cast<uint16_t*>(b + lo.h16);
  a.hsig = reinterpret_cast<int32_t*>(b + lo.hsig);
  a.P = reinterpret_cast<float*>(b + lo.P);
  a.y = static_cast<uint16_t*>(y);
  a.xq = b + lo.xq;
  a.xsf = b + lo.xsf;
  a.xqg = b + lo.xqg;
  a.xsfg = b + lo.xsfg;
  a.hq = b + lo.hq;
  a.hsf = b + lo.hsf;
  a.rw_hi = reinterpret_cast<uint16_t*>(b + lo.rw_hi);
  a.rw_lo = reinterpret_cast<uint16_t*>(b + lo.rw_lo);
  a.logits_tc = prefill_logits_tc_ok(a) ? 1 : 0;
  a.bias_select = L->bias_select;
  a.unbiased = reinterpret_cast<float*>(b + lo.approx);
  a.wait_ns = 2000000000ull;
  if (L->shared_fmt) {
    a.sfmt = L->shared_fmt;
    a.Is = L->shared_inter;
    a.s_gate = qw(L->shared_gate, L->shared_fmt);
    a.s_up = qw(L->shared_up, L->shared_fmt);
    a.s_down = qw(L->shared_down, L->shared_fmt);
    a.xs16 = reinterpret_cast<uint16_t*>(b + lo.xs16);
    a.hs = reinterpret_cast<uint16_t*>(b + lo.hs);
    a.hs16 = reinterpret_cast<uint16_t*>(b + lo.hs16);
    a.hssig = reinterpret_cast<int32_t*>(b + lo.hssig);
    a.S = reinterpret_cast<float*>(b + lo.S);
    a.sgate_w = L->shared_expert_gate;
    a.sgate = reinterpret_cast<float*>(b + lo.sgate);
  }
  return a;
}

int sm_count(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

// Layers the prefill expert GEMMs implement: the exact chain for every routed
// and shared format with hidden, inter and shared inter multiples of 128; the
// W4A4 lever for NVFP4 routed experts without a shared expert, with whole
// 256-column stages and 16-byte aligned scale rows.
bool prefill_supported(const moe_layer* L, int act_quant) {
  if (L->hidden % 128 != 0 || L->inter % 128 != 0) return false;
  if (L->shared_fmt != MOE_FMT_NONE && L->shared_inter % 128 != 0) return false;
  if (!act_quant) return true;
  // the W4A4 lever: NVFP4 activations on NVFP4 weights, MXFP4 activations on MXFP4 weights
  if (L->fmt != (act_quant == 2 ? MOE_FMT_MXFP4 : MOE_FMT_NVFP4) || L->shared_fmt != MOE_FMT_NONE) return false;
  const auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  return L->hidden % 256 == 0 && L->inter % 256 == 0 && a16(L->gate.scales) && a16(L->up.scales) &&
         a16(L->down.scales);
}

}  // namespace

int32_t qmoe::clear_workspace_counters(const moe_layer* L, void* ws, size_t ws_bytes, bool keep_error,
                                       cudaStream_t s) {
  const Layout lo = make_layout(L, ws_max_tokens(L, ws_bytes));
  uint8_t* b = static_cast<uint8_t*>(ws);
  // the error word and its info come first in the control block
  const size_t skip = keep_error ? offsetof(Ctrl, router_arrive) : 0;
  const size_t sections[3][2] = {{lo.ctrl + skip, sizeof(Ctrl) - skip},
                                 {lo.gu_cnt, lo.dn_part - lo.gu_cnt},
                                 {lo.dn_cnt, lo.xg - lo.dn_cnt}};
  for (const auto& sec : sections)
    if (cudaMemsetAsync(b + sec[0], 0, sec[1], s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" {

const char* moe_status_string(int32_t status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape or format combination not supported";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED: device pointer not aligned";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing or too small";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a bounded device-side wait gave up";
    case MOE_ERR_DEVICE_BAD_INDEX: return "MOE_ERR_DEVICE_BAD_INDEX: device-side index check failed";
    default: return "unknown moe_status";
  }
}

size_t moe_workspace_size(const moe_layer* layer, int32_t max_tokens, const moe_options* opts) {
  if (check_layer(layer) != MOE_OK || check_options(opts) != MOE_OK || max_tokens < 1) return 0;
  return make_layout(layer, max_tokens).total;
}

int32_t moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!ws || ws_bytes < sizeof(Ctrl)) return MOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_MISALIGNED;
  // control block plus every counter section: zero the whole workspace once
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

int32_t moe_workspace_layout(const moe_layer* layer, int32_t max_tokens, const moe_options* opts,
                             moe_ws_layout* out) {
  int32_t st = check_layer(layer);
  if (st != MOE_OK) return st;
  if ((st = check_options(opts)) != MOE_OK) return st;
  if (!out || max_tokens < 1) return MOE_ERR_INVALID_ARG;
  const Layout lo = make_layout(layer, max_tokens);
  out->logits = lo.logits;
  out->topk_idx = lo.topk_idx;
  out->topk_w = lo.topk_w;
  out->expert_cnt = lo.cnt;
  out->expert_off = lo.off;
  out->pair_list = lo.pair;
  out->total = lo.total;
  out->h_codes = lo.hq;
  out->h_scales = lo.hsf;
  return MOE_OK;
}

int32_t moe_route(const moe_layer* layer, const void* x, int32_t T, int32_t* topk_idx, float* topk_w,
                  int32_t* expert_cnt, int32_t* expert_off, int32_t* pair_list, void* ws, size_t ws_bytes,
                  moe_stream_t stream) {
  int32_t st = check_layer(layer);
  if (st != MOE_OK) return st;
  if (!x) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x)) return MOE_ERR_MISALIGNED;
  if (T < 1) return MOE_ERR_INVALID_ARG;
  const void* outs[5] = {topk_idx, topk_w, expert_cnt, expert_off, pair_list};
  for (const void* p : outs)
    if (p && !aligned4(p)) return MOE_ERR_MISALIGNED;
  if ((st = check_ws(layer, T, ws, ws_bytes)) != MOE_OK) return st;
  const int maxT = ws_max_tokens(layer, ws_bytes);
  const Layout lo = make_layout(layer, maxT);
  if (T > MOE_DECODE_MAX_TOKENS) {
    PrefillArgs pa = prefill_args(layer, lo, ws, x, T, nullptr);
    pa.out.topk_idx = topk_idx; pa.out.topk_w = topk_w; pa.out.cnt = expert_cnt; pa.out.off = expert_off;
    pa.out.pair = pair_list;
    pa.xg = nullptr;
    return cuda_status(launch_prefill_route(pa, reinterpret_cast<cudaStream_t>(stream)));
  }
  RouterArgs ra = router_args(layer, lo, ws, x, T);
  ra.out.topk_idx = topk_idx; ra.out.topk_w = topk_w; ra.out.cnt = expert_cnt; ra.out.off = expert_off;
  ra.out.pair = pair_list;
  if ((size_t)T * layer->hidden * 2 > 200 * 1024) return MOE_ERR_UNSUPPORTED;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t err = launch_router_decode(ra, s);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_route_dispatch(ra, s));
}

}  // extern "C"

// Host checks of a decode call's arguments other than the workspace (no device access).
int32_t qmoe::check_decode_args(const moe_layer* layer, const void* x, int32_t T, const void* y,
                                const moe_options* opts) {
  int32_t st = check_layer(layer);
  if (st != MOE_OK) return st;
  if ((st = check_options(opts)) != MOE_OK) return st;
  if (opts && (opts->act_quant || opts->fold_scales || opts->fp8_act)) return MOE_ERR_UNSUPPORTED;  // prefill levers
  if (!x || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return MOE_ERR_MISALIGNED;
  if (T < 1) return MOE_ERR_INVALID_ARG;
  if (T > MOE_DECODE_MAX_TOKENS) return MOE_ERR_UNSUPPORTED;
  if ((size_t)T * layer->hidden * 2 > 200 * 1024) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

extern "C" {

static int32_t decode_forward_checked(const moe_layer* layer, const void* x, int32_t T, void* y,
                                      const moe_options* opts, void* ws, size_t ws_bytes, moe_stream_t stream,
                                      void* const* events) {
  int32_t st = qmoe::check_decode_args(layer, x, T, y, opts);
  if (st != MOE_OK) return st;
  if ((st = check_ws(layer, T, ws, ws_bytes)) != MOE_OK) return st;
  return decode_forward_impl(layer, x, T, y, opts, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), events);
}

int32_t moe_decode_forward(const moe_layer* layer, const void* x, int32_t T, void* y, const moe_options* opts,
                           void* ws, size_t ws_bytes, moe_stream_t stream) {
  return decode_forward_checked(layer, x, T, y, opts, ws, ws_bytes, stream, nullptr);
}

int32_t moe_experts_forward(const moe_layer* layer, const void* x, int32_t T, const int32_t* topk_idx,
                            const float* topk_w, void* y, const moe_options* opts, void* ws, size_t ws_bytes,
                            moe_stream_t stream) {
  int32_t st = qmoe::check_decode_args(layer, x, T, y, opts);
  if (st != MOE_OK) return st;
  if (!topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned4(topk_idx) || !aligned4(topk_w)) return MOE_ERR_MISALIGNED;
  if ((st = check_ws(layer, T, ws, ws_bytes)) != MOE_OK) return st;
  return decode_forward_impl(layer, x, T, y, opts, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr,
                             topk_idx, topk_w);
}

int32_t moe_decode_plan(const moe_layer* layer, int32_t T, int32_t num_sms, moe_decode_plan_info* out) {
  if (!out || T < 1 || T > MOE_DECODE_MAX_TOKENS || num_sms < 1) return MOE_ERR_INVALID_ARG;
  const int32_t st = check_layer(layer);
  if (st != MOE_OK) return st;
  DecodePlan pl;
  const int32_t pst = plan_decode(layer, T, num_sms, &pl);
  if (pst != MOE_OK) return pst;
  std::memset(out, 0, sizeof(*out));
  out->gu_slices = pl.gu_slices;
  out->gu_slices_shared = pl.gu_slices_s;
  out->gu_slices_tail = pl.gu_slices_t;
  out->gu_tail_cap = pl.gu_tail_cap;
  out->dn_slices = pl.dn_slices;
  out->dn_segs = pl.dn_segs;
  out->gu_ctas_per_sm = T <= kGuSmallT ? 3 : 2;
  out->gu_smem = pl.smem_gu;
  out->dn_smem = pl.smem_dn;
  out->gu_split_blocks = (size_t)pl.gu_blocks;
  out->dn_split_blocks = (size_t)pl.dn_blocks;
  out->split_block_capacity = kMaxSplitBlocks;
  return MOE_OK;
}

int32_t moe_decode_forward_timed(const moe_layer* layer, const void* x, int32_t T, void* y,
                                 const moe_options* opts, void* ws, size_t ws_bytes, moe_stream_t stream,
                                 void* const* events) {
  return decode_forward_checked(layer, x, T, y, opts, ws, ws_bytes, stream, events);
}

struct MarkCtx {
  void* const* events;
  cudaStream_t stream;
  bool capturing;
};

static void record_mark(void* ctx, int i) {
  const MarkCtx* m = static_cast<const MarkCtx*>(ctx);
  if (!m->events || !m->events[i]) return;
  cudaEvent_t ev = static_cast<cudaEvent_t>(m->events[i]);
  if (m->capturing) cudaEventRecordWithFlags(ev, m->stream, cudaEventRecordExternal);
  else cudaEventRecord(ev, m->stream);
}

static int32_t prefill_forward_checked(const moe_layer* layer, const void* x, int32_t T, void* y,
                                       const moe_options* opts, void* ws, size_t ws_bytes, moe_stream_t stream,
                                       void* const* events) {
  int32_t st = check_layer(layer);
  if (st != MOE_OK) return st;
  if ((st = check_options(opts)) != MOE_OK) return st;
  if (!x || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return MOE_ERR_MISALIGNED;
  if (T < 1) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(layer, T, ws, ws_bytes)) != MOE_OK) return st;
  const int aq = opts ? opts->act_quant : 0;
  if (!prefill_supported(layer, aq)) return MOE_ERR_UNSUPPORTED;
  int sms = 0;
  if ((st = sm_count(&sms)) != MOE_OK) return st;
  const Layout lo = make_layout(layer, ws_max_tokens(layer, ws_bytes));
  PrefillArgs pa = prefill_args(layer, lo, ws, x, T, y);
  pa.act_quant = aq;
  pa.wait_ns = wait_limit_ns(opts);
  pa.p_bf16 = (opts && opts->bf16_partials) ? 1 : 0;
  pa.fold_scales = (opts && opts->fold_scales) ? 1 : 0;
  pa.fp8_act = (opts && opts->fp8_act) ? 1 : 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MarkCtx mc{events, s, false};
  if (events) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &cap);
    mc.capturing = cap == cudaStreamCaptureStatusActive;
  }
  const Marks mk{events ? record_mark : nullptr, &mc};
  mk(0);
  cudaError_t err = launch_prefill_route(pa, s, mk);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_prefill_experts(pa, sms, s, mk));
}

int32_t moe_prefill_forward(const moe_layer* layer, const void* x, int32_t T, void* y, const moe_options* opts,
                            void* ws, size_t ws_bytes, moe_stream_t stream) {
  return prefill_forward_checked(layer, x, T, y, opts, ws, ws_bytes, stream, nullptr);
}

int32_t moe_prefill_forward_timed(const moe_layer* layer, const void* x, int32_t T, void* y,
                                  const moe_options* opts, void* ws, size_t ws_bytes, moe_stream_t stream,
                                  void* const* events) {
  return prefill_forward_checked(layer, x, T, y, opts, ws, ws_bytes, stream, events);
}

int32_t moe_check(void* ws, size_t ws_bytes, moe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!ws && ws_bytes == 0) {
    // the allocation-free entry point's array on the current device
    void* p = nullptr;
    const int32_t st = qmoe::noalloc_array_if_used(&p);
    if (st != MOE_OK || !p) return st;
    ws = p;
    ws_bytes = sizeof(Ctrl);
  }
  if (!ws || ws_bytes < sizeof(Ctrl)) return MOE_ERR_WORKSPACE;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  Ctrl c;
  if (cudaMemcpy(&c, ws, sizeof(Ctrl), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (c.error == 0) return MOE_OK;
  const uint32_t zero[2] = {0, 0};
  if (cudaMemcpy(ws, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
  return (int32_t)c.error;
}

int32_t moe_dequantize(int32_t fmt, const moe_qweight* w, int32_t N, int32_t K, int32_t expert, int32_t row0,
                       int32_t nrows, float* out, moe_stream_t stream) {
  if (!w || !out || !valid_fmt(fmt)) return MOE_ERR_INVALID_ARG;
  int32_t st = check_qweight(*w, fmt, N, K);
  if (st != MOE_OK) return st;
  if (!aligned16(out)) return MOE_ERR_MISALIGNED;
  if (expert < 0 || row0 < 0 || nrows < 1 || row0 + nrows > N) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_dequantize(fmt, qw(*w, fmt), N, K, expert, row0, nrows, out,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

int32_t moe_quantize_act_nvfp4(const void* x, int32_t rows, int32_t K, uint8_t* codes, uint8_t* scales,
                               moe_stream_t stream) {
  if (!x || !codes || !scales || rows < 1 || K < 16 || K % 16) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(codes) & 7)) return MOE_ERR_MISALIGNED;
  return cuda_status(launch_quantize_act_nvfp4(static_cast<const uint16_t*>(x), rows, K, codes, scales,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

int32_t moe_quantize_act_mxfp4(const void* x, int32_t rows, int32_t K, uint8_t* codes, uint8_t* scales,
                               moe_stream_t stream) {
  if (!x || !codes || !scales || rows < 1 || K < 32 || K % 32) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(codes)) return MOE_ERR_MISALIGNED;
  return cuda_status(launch_quantize_act_mxfp4(static_cast<const uint16_t*>(x), rows, K, codes, scales,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
