"""The MoE layer in plain FP64 (oracle; test infrastructure).

Steps and rounding points (DGPP pages: page 1 README "Exact" bullet and
"exactness / levers" paragraph; page 3 README "Execution and performance"
table, rows engine.prefill_bf16_partials and engine.prefill_fold_scales;
page 4 forum post 1 quantisation table, "Activations stay BF16"):

  x            BF16 activations [T, H]
  logits       l[t, e] = fl32( sum_h x[t, h] * Wr[e, h] )   correctly rounded FP32
               (+ fl32 addition of an optional per-expert bias)
  top-k        experts ordered by (l descending, e ascending), first k kept
  weights      w_j = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k selected,
               in FP64, stored as FP32 (equal to a full softmax renormalised
               over the top-k; the shared denominator cancels)
  dispatch     pairs p = t*k + j grouped by expert, ascending p within an expert
  per pair     g = W_gate x, u = W_up x (FP64), h = bf16( silu(g) * u ),
               P = W_down h (FP64)
  combine      y_t = bf16( sum_j w_tj * P_tj  +  S_t ), S_t the shared expert
               (weight 1, no gate) computed the same way

Weights are decoded exactly (``formats.decode``); the only roundings are the
FP32 logits and weights and the two BF16 roundings of h and y, which is the
"FP32 accumulation, BF16 activations" chain evaluated without accumulation
error.
"""
from __future__ import annotations

import math
from fractions import Fraction
from typing import Optional

import numpy as np

from . import formats as F

_U64 = 2.0 ** -53


# ---------------------------------------------------------------- router ----

def _fl32_exact(products: list) -> np.float32:
    """Correctly rounded FP32 of the exact sum of FP64-exact products."""
    d = math.fsum(products)                  # correctly rounded FP64 of the exact sum
    f = np.float32(d)
    fd = float(f)
    if fd == d:
        return f
    other = np.nextafter(f, np.float32(np.inf) if d > fd else np.float32(-np.inf))
    mid = (fd + float(other)) / 2.0          # exact in FP64
    if d != mid:
        return f                             # d strictly inside f's rounding interval
    # d sits exactly on an FP32 midpoint: decide with the exact rational sum.
    s = sum(Fraction(p) for p in products)
    m = Fraction(mid)
    if s > m:
        return np.float32(max(fd, float(other)))
    if s < m:
        return np.float32(min(fd, float(other)))
    return f if (f.view(np.uint32) & 1) == 0 else other   # exact tie: even


def router_logits(x_bits: np.ndarray, Wr: np.ndarray, bias: Optional[np.ndarray] = None):
    """Correctly rounded FP32 router logits.

    Returns (logits f32 [T, E], near_midpoint bool [T, E]).  Each BF16 x FP32
    product is exact in FP64.  The FP64 BLAS dot carries at most
    gamma_n * sum|x_h Wr_eh| error; every logit whose FP64 result lies within
    that bound (plus 2^-40 relative) of an FP32 rounding midpoint is
    recomputed from an exactly rounded sum (math.fsum, then exact rationals
    at a midpoint), which settles both its rounding and its distance to the
    midpoint.  ``near_midpoint`` then marks the logits whose exact value lies
    within 2^-40 (relative) of an FP32 rounding midpoint: a compensated FP32
    dot may round those differently, so callers report them.
    """
    X = F.bf16_to_f64(x_bits)
    W = np.asarray(Wr, dtype=np.float32).astype(np.float64)
    T, H = X.shape
    d = X @ W.T
    n = H
    gamma = n * _U64 / (1.0 - n * _U64)
    bound = gamma * (np.abs(X) @ np.abs(W).T) * (1.0 + 1e-9) + 1e-300
    l32 = d.astype(np.float32)
    # entries the FP64 result cannot settle: its rounding, or its distance to the nearer midpoint
    uncertain = midpoint_distance(d, l32) <= 2.0 ** -40 * np.maximum(np.abs(d), 1e-300) + bound
    d_exact = d.copy()
    for t, e in zip(*np.nonzero(uncertain)):
        prods = [float(a) * float(b) for a, b in zip(X[t], W[e])]
        d_exact[t, e] = math.fsum(prods)        # within 2^-53 relative of the exact sum
        l32[t, e] = _fl32_exact(prods)
    near = near_midpoint(d_exact, l32)
    if bias is not None:
        l32 = (l32 + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)
    return l32, near


def midpoint_distance(d: np.ndarray, l32: np.ndarray) -> np.ndarray:
    """Distance from d to the nearer of the two FP32 rounding midpoints around l32 (exact in FP64)."""
    f = l32.astype(np.float64)
    up = np.nextafter(l32, np.float32(np.inf)).astype(np.float64)
    dn = np.nextafter(l32, np.float32(-np.inf)).astype(np.float64)
    return np.minimum(np.abs(d - (f + up) / 2.0), np.abs(d - (f + dn) / 2.0))


def near_midpoint(d_exact: np.ndarray, l32: np.ndarray) -> np.ndarray:
    """Logits whose exact dot product lies within 2^-40 (relative) of an FP32 midpoint.

    d_exact holds the dot products to within 2^-53 relative (the FP64 result
    wherever it is provably farther from a midpoint) and l32 the correctly
    rounded FP32 logits.  A compensated FP32 dot product (float-float, whose
    error before its last rounding is of order 2^-44 relative) may round the
    flagged ones the other way.
    """
    return midpoint_distance(d_exact, l32) <= 2.0 ** -40 * np.maximum(np.abs(d_exact), 1e-300)


def topk(l32: np.ndarray, k: int) -> np.ndarray:
    """Top-k expert ids per token, ordered by (logit desc, expert id asc)."""
    T, E = l32.shape
    ids = np.arange(E)
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        order = np.lexsort((ids, -l32[t].astype(np.float64)))
        out[t] = order[:k]
    return out


def topk_weights(l32: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Renormalised softmax weights over the selected experts, FP64 -> FP32."""
    sel = np.take_along_axis(l32.astype(np.float64), idx.astype(np.int64), axis=1)
    z = np.exp(sel - sel[:, :1])
    return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)


def topk_weights_full_softmax(l32: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Same weights via a softmax over all experts followed by renormalisation (FP64)."""
    L = l32.astype(np.float64)
    p = np.exp(L - L.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def route(x_bits, Wr, bias, k, bias_select: bool = False):
    """Logits, top-k and weights.  The bias (if any) is added to the FP32 logits.
    Default: the biased logits decide both the selection and the weights.  With
    bias_select the bias steers the selection only and the weights come from the
    unbiased logits of the selected experts (the variant where a per-expert
    correction balances the load without changing the mixture weights).  Returns
    (selection logits f32, near-midpoint flags, indices, weights)."""
    l32, near = router_logits(x_bits, Wr, None)
    lsel = l32 if bias is None else (l32 + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)
    idx = topk(lsel, k)
    w = topk_weights(l32 if bias_select else lsel, idx)
    return lsel, near, idx, w


def shared_gate(x_bits, w_gate) -> np.ndarray:
    """Sigmoid gate of the shared expert per token: sigma(g_t), g_t the correctly
    rounded FP32 dot product of the token with the gate vector [H] (the router's
    logit rule), sigma(z) = 1 / (1 + e^-z) in FP64."""
    g, _ = router_logits(x_bits, np.asarray(w_gate, dtype=np.float32)[None, :])
    return 1.0 / (1.0 + np.exp(-g[:, 0].astype(np.float64)))


# -------------------------------------------------------------- dispatch ----

def dispatch(idx: np.ndarray, E: int):
    """Stable counting sort of pairs p = t*k + j by expert.

    Returns (cnt [E] i32, off [E+1] i32, pair [T*k] i32): the pairs routed to
    expert e are pair[off[e]:off[e+1]], in ascending p.
    """
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    cnt = np.bincount(flat, minlength=E).astype(np.int32)
    off = np.zeros(E + 1, dtype=np.int32)
    np.cumsum(cnt, out=off[1:])
    pair = np.argsort(flat, kind="stable").astype(np.int32)
    return cnt, off, pair


# ---------------------------------------------------------------- experts ----

def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


# activation quantisers of the levers: the W4A4 lever's NVFP4 (1) and MXFP4 (2) blocks, and the
# FP8-activation lever's per-token 1x128 E4M3 blocks (3, applied to FP8 b128 experts only)
ACT_FP8 = 3


def act_fake_quant(a: np.ndarray, act_quant: int) -> np.ndarray:
    """The levers' activation quantiser: act_quant 1 (or True) = NVFP4
    16-element blocks, 2 = MXFP4 32-element blocks, 3 = E4M3 128-element
    blocks (``fp8_quantize_act``); 0 = none."""
    if not act_quant:
        return a
    if int(act_quant) == ACT_FP8:
        return fp8_fake_quant(a)
    return mxfp4_fake_quant(a) if int(act_quant) == 2 else nvfp4_fake_quant(a)


def swiglu_mlp(Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray, X: np.ndarray,
               act_quant: int = 0) -> tuple:
    """One SwiGLU expert on token rows X [n, H] (FP64 values).

    Returns (h, P): h = bf16(silu(X Wg^T) * (X Wu^T)) [n, I] as FP64 values,
    P = h Wd^T [n, H] in FP64.  With act_quant the token rows and h are
    replaced by their quantised values (NVFP4 for 1, MXFP4 for 2, E4M3 1x128
    blocks for 3) before each projection.
    """
    X = act_fake_quant(X, act_quant)
    g = X @ Wg.T
    u = X @ Wu.T
    h = F.round_bf16(silu(g) * u)
    hq = act_fake_quant(h, act_quant)
    P = hq @ Wd.T
    return h, P


# ------------------------------------------------ W4A4 activation quantizer ----

def nvfp4_quantize_act(a: np.ndarray):
    """NVFP4 quantisation of activation rows in 16-element blocks, tensor scale 1.

    Per block: s = e4m3_rne_sat( fl32(amax / 6) ); code = e2m1_rne_sat( fl32(a / s) ),
    with FP32 division emulated as an FP64 divide rounded to FP32 (correct
    because 53 >= 2*24 + 2).  A block whose scale rounds to zero gets all-zero
    codes.  Returns (codes [.., K] u8 0..15, scale codes [.., K/16] u8).
    """
    a = np.asarray(a, dtype=np.float64)
    *lead, K = a.shape
    blk = a.reshape(*lead, K // 16, 16)
    amax = np.abs(blk).max(axis=-1)
    s_code = F.e4m3_encode_rne_sat(np.float32(amax / 6.0).astype(np.float64))
    s = F.E4M3_TABLE[s_code]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.float32(blk / s[..., None]).astype(np.float64)
    q = np.where((s > 0)[..., None], q, 0.0)
    codes = F.e2m1_encode_rne(q)
    codes = np.where((s > 0)[..., None], codes, 0).astype(np.uint8)
    return codes.reshape(*lead, K), s_code.astype(np.uint8)


def nvfp4_dequantize_act(codes: np.ndarray, s_code: np.ndarray) -> np.ndarray:
    *lead, K = codes.shape
    v = F.E2M1_TABLE[codes].reshape(*lead, K // 16, 16) * F.E4M3_TABLE[s_code][..., None]
    return v.reshape(*lead, K)


def nvfp4_fake_quant(a: np.ndarray) -> np.ndarray:
    return nvfp4_dequantize_act(*nvfp4_quantize_act(a))


def mxfp4_quantize_act(a: np.ndarray):
    """MXFP4 quantisation of activation rows in 32-element blocks (the MXFP4
    checkpoint rule, reading Q3): the block exponent e is the smallest integer
    with 6 * 2^e >= amax (amax = 0 -> e = 0), its E8M0 code e + 127 clamped to
    [0, 254]; code = e2m1_rne_sat( a / 2^e ) (the division by a power of two is
    exact).  Returns (codes [.., K] u8 0..15, scale codes [.., K/32] u8).
    """
    a = np.asarray(a, dtype=np.float64)
    *lead, K = a.shape
    blk = a.reshape(*lead, K // 32, 32)
    amax = np.abs(blk).max(axis=-1)
    # log2(amax / 6) lies in [p - 3.585, p - 2.585) for amax = f 2^p, f in [0.5, 1): e is p - 3 or p - 2
    _, p = np.frexp(np.where(amax > 0, amax, 1.0))
    e = np.where(6.0 * np.ldexp(1.0, p - 3) >= amax, p - 3, p - 2)
    e = np.where(amax > 0, e, 0)
    s_code = np.clip(e + 127, 0, 254)
    s = np.ldexp(1.0, s_code - 127)
    codes = F.e2m1_encode_rne(blk / s[..., None])
    return codes.reshape(*lead, K).astype(np.uint8), s_code.astype(np.uint8)


def mxfp4_dequantize_act(codes: np.ndarray, s_code: np.ndarray) -> np.ndarray:
    *lead, K = codes.shape
    v = F.E2M1_TABLE[codes].reshape(*lead, K // 32, 32) * np.ldexp(1.0, s_code.astype(np.int64) - 127)[..., None]
    return v.reshape(*lead, K)


def mxfp4_fake_quant(a: np.ndarray) -> np.ndarray:
    return mxfp4_dequantize_act(*mxfp4_quantize_act(a))


# ---------------------------------------------- FP8 activation lever ----

E4M3_MAX = 448.0


def fp8_quantize_act(a: np.ndarray):
    """Per-token 1x128 E4M3 quantisation of activation rows.

    DGPP README "Execution and performance" table, row engine.prefill_fp8_gemm:
    FP8 projections run on the fp8 tensor cores from per-token 1x128 e4m3
    activations against the checkpoint's 128x128 weight scales.  Reading: per
    128-element block of a row, the FP32 scale s = fl32(amax / 448) (448 the
    largest finite E4M3 value; amax = 0 gives s = 0 and zero codes) and
    code = e4m3_rne_sat( fl32(a / s) ), both quotients IEEE FP32 divisions as
    a kernel computes them.  Returns (codes [.., K] u8, scales [.., K/128] f32).
    """
    a = np.asarray(a, dtype=np.float64)
    *lead, K = a.shape
    blk = a.reshape(*lead, K // 128, 128)
    amax = np.abs(blk).max(axis=-1)
    s = (amax.astype(np.float32) / np.float32(E4M3_MAX)).astype(np.float32)   # amax: BF16 values, exact in FP32
    pos = s > 0
    q = (blk.astype(np.float32) / np.where(pos, s, np.float32(1.0))[..., None]).astype(np.float64)
    codes = np.where(pos[..., None], F.e4m3_encode_rne_sat(q), 0)   # a zero block: +0 codes
    return codes.reshape(*lead, K).astype(np.uint8), s


def fp8_dequantize_act(codes: np.ndarray, s: np.ndarray) -> np.ndarray:
    *lead, K = codes.shape
    v = F.E4M3_TABLE[codes].reshape(*lead, K // 128, 128) * np.asarray(s, dtype=np.float64)[..., None]
    return v.reshape(*lead, K)


def fp8_fake_quant(a: np.ndarray) -> np.ndarray:
    return fp8_dequantize_act(*fp8_quantize_act(a))


# ------------------------------------------------------------------ layer ----

def _decoded(qm, e, fold_scales: bool = False):
    return F.decode_qmat_fold(qm, e) if fold_scales else F.decode_qmat(qm, e)


def layer_forward(layer, x_bits: np.ndarray, act_quant: int = 0, tokens=None, expert_cache=None,
                  bias_select: bool = False, bf16_partials: bool = False, routing=None,
                  fold_scales: bool = False, fp8_act: bool = False):
    """Full MoE layer on host-resident checkpoint data (a synth.HostLayer).

    tokens: optional subset of token rows whose outputs are wanted (routing is
    still computed for every token, so the dispatch index is complete).
    expert_cache: optional callable e -> (Wg, Wu, Wd) FP64, to regenerate
    experts lazily instead of reading them from ``layer``.
    bias_select: the router bias steers the selection only (see ``route``).
    bf16_partials: every expert's down-projection output (the routed partials
    and the shared expert's) is rounded to BF16 before the weighted sum (page
    3 README "Execution and performance", engine.prefill_bf16_partials, a
    lever off by default).
    A gate vector in ``layer.extra["shared_gate_w"]`` ([H] f32) scales the
    shared expert by its sigmoid gate (``shared_gate``); without one the shared
    expert enters with weight 1.
    routing: optional (idx [T, k] i32, w [T, k] f32) chosen by the caller; the
    router is then skipped and these pairs and weights are used as given.
    act_quant: the W4A4 lever's activation quantisation (1 or True: NVFP4, 2:
    MXFP4), applied to the token rows and to h before each projection.
    fold_scales: the fold-scales lever (``formats.fold_scales_weights``):
    int8 g64, FP8 b128 and int4 g128 weights, routed and shared, enter as
    bf16(fl32(code * scale)); the rest of the chain is unchanged.  An
    ``expert_cache`` must then supply the folded weights itself.
    fp8_act: the FP8-activation lever (``fp8_quantize_act``): FP8 b128 experts,
    routed or shared, see their token rows and h (after its BF16 rounding) as
    per-token 1x128 E4M3 blocks; their weights stay exact (the lever takes
    precedence over fold_scales for them).  Other experts are unchanged.
    Returns a dict of every intermediate the CUDA path exposes.
    """
    cfg = layer.cfg
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    T = x_bits.shape[0]
    if routing is None:
        l32, near, idx, w = route(x_bits, layer.router_w, layer.router_b, cfg.k, bias_select)
    else:
        idx = np.asarray(routing[0], dtype=np.int32)
        w = np.asarray(routing[1], dtype=np.float32)
        l32, near = None, np.zeros((T, cfg.E), dtype=bool)
    cnt, off, pair = dispatch(idx, cfg.E)
    fp8_r = bool(fp8_act) and cfg.fmt == F.FMT_FP8_B128
    fp8_s = bool(fp8_act) and cfg.shared_fmt == F.FMT_FP8_B128
    aq_r = ACT_FP8 if fp8_r else act_quant
    aq_s = ACT_FP8 if fp8_s else act_quant
    want = np.arange(T) if tokens is None else np.asarray(sorted(set(int(t) for t in tokens)))
    X = F.bf16_to_f64(x_bits)
    acc = {int(t): np.zeros(cfg.H) for t in want}
    h_out = {}
    want_set = set(int(t) for t in want)
    for e in range(cfg.E):
        ps = [int(p) for p in pair[off[e]:off[e + 1]] if int(p) // cfg.k in want_set]
        if not ps:
            continue
        if expert_cache is not None:
            Wg, Wu, Wd = expert_cache(e)
        else:
            fr = fold_scales and not fp8_r
            Wg, Wu, Wd = _decoded(layer.gate, e, fr), _decoded(layer.up, e, fr), _decoded(layer.down, e, fr)
        rows = np.array([p // cfg.k for p in ps])
        h, P = swiglu_mlp(Wg, Wu, Wd, X[rows], aq_r)
        if bf16_partials:
            P = F.round_bf16(P)
        for i, p in enumerate(ps):
            t, j = divmod(p, cfg.k)
            acc[t] += float(w[t, j]) * P[i]
            h_out[p] = h[i]
    S = None
    if layer.shared_gate is not None:
        fs = fold_scales and not fp8_s
        Wg, Wu, Wd = (_decoded(layer.shared_gate, 0, fs), _decoded(layer.shared_up, 0, fs),
                      _decoded(layer.shared_down, 0, fs))
        _, S = swiglu_mlp(Wg, Wu, Wd, X[want], aq_s)
        if bf16_partials:
            S = F.round_bf16(S)
        gw = getattr(layer, "extra", {}).get("shared_gate_w")
        if gw is not None:
            S = S * shared_gate(x_bits[want], gw)[:, None]
    y = np.zeros((len(want), cfg.H))
    for i, t in enumerate(want):
        y[i] = acc[int(t)] + (S[i] if S is not None else 0.0)
    return {
        "logits": l32, "near_midpoint": near, "topk_idx": idx, "topk_w": w,
        "expert_cnt": cnt, "expert_off": off, "pair_list": pair,
        "tokens": want, "y_f64": y, "y_bits": F.f64_to_bf16_bits(y), "h": h_out, "shared": S,
    }


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of BF16 values at |v| (the unit in the last place)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    ulp = np.ldexp(1.0, np.maximum(e - 8, -133))
    return np.where(a > 0, ulp, 2.0 ** -133)


def within_tolerance(y_test: np.ndarray, y_ref: np.ndarray, ulps: float = 2.0, abs_tol: float = 1e-3):
    """Elementwise |y_test - y_ref| <= max(ulps * ulp_bf16(y_ref), abs_tol)."""
    y_test = np.asarray(y_test, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    tol = np.maximum(ulps * bf16_ulp(y_ref), abs_tol)
    return np.abs(y_test - y_ref) <= tol
