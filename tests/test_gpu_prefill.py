"""GPU parity of the prefill path (any token count) against the FP64 oracle,
through the C ABI.

Routing: the approximate-then-exact router must give bit-exact top-k indices,
expert counts, offsets and pair lists, FP32 weights within a few ulp, and the
exact (correctly rounded) logit for every expert it recomputed.  Layer output
y within max(2 BF16 ulp, 1e-3) of the oracle, on small ragged shapes (several
token tiles of one expert, a ragged tail, experts with no tokens) and on the
prefill workload at full size (sampled tokens).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import formats as F
from oracle import moe as M
from quantized_moe_decode_router_gb300 import _binding as B
from quantized_moe_decode_router_gb300.device import to_device
from synth.configs import (FMT_FP8_B128, FMT_INT4_G64, FMT_INT4_G128, FMT_INT8_G64, FMT_MXFP4, FMT_NVFP4,
                           LayerConfig)
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    G.lib()


def assert_prefill_routing(got: dict, ref: dict, near: np.ndarray):
    """Indices and dispatch bit-exact; every logit the router recomputed is the
    correctly rounded value (the others are -inf in the workspace)."""
    lg, lr = got["logits"], ref["logits"]
    recomputed = ~np.isneginf(lg)
    diff = (lg.view(np.uint32) != lr.view(np.uint32)) & recomputed
    assert not np.any(diff & ~near), f"{int(np.sum(diff & ~near))} recomputed logits differ"
    T, k = ref["topk_idx"].shape
    assert np.all(recomputed[np.arange(T)[:, None], ref["topk_idx"]]), "a selected expert was not recomputed"
    np.testing.assert_array_equal(got["topk_idx"], ref["topk_idx"])
    np.testing.assert_array_equal(got["expert_cnt"], ref["expert_cnt"])
    np.testing.assert_array_equal(got["expert_off"], ref["expert_off"])
    np.testing.assert_array_equal(got["pair_list"], ref["pair_list"])
    np.testing.assert_allclose(got["topk_w"], ref["topk_w"], rtol=8 * 2.0 ** -24, atol=2.0 ** -30)


def _check_y(y_bits, ref_bits, tokens=None):
    y = F.bf16_to_f64(y_bits if tokens is None else y_bits[tokens])
    r = F.bf16_to_f64(ref_bits)
    ok = M.within_tolerance(y, r)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        raise AssertionError(f"{int((~ok).sum())} of {ok.size} outputs outside tolerance; e.g. "
                             + ", ".join(f"{tuple(b)}: {y[tuple(b)]} vs {r[tuple(b)]}" for b in bad))


# ------------------------------------------------------------------ routing ----

ROUTE_CASES = [("tiny_nvfp4", 9), ("tiny_nvfp4", 300), ("decode_nvfp4", 64), ("decode_mxfp4", 33),
               ("prefill_nvfp4", 700), ("prefill_nvfp4", 4096)]


@pytest.mark.parametrize("name,T", ROUTE_CASES)
def test_prefill_route_matches_oracle(name, T):
    hl = G.host_layer(name)
    dl = G.device_layer(name)
    x = synth.make_tokens(hl.cfg, T, seed=0, batch=T)
    got = G.route(dl, x)
    l32, near, idx, w = M.route(x, hl.router_w, hl.router_b, hl.cfg.k)
    cnt, off, pair = M.dispatch(idx, hl.cfg.E)
    ref = {"logits": l32, "topk_idx": idx, "topk_w": w, "expert_cnt": cnt, "expert_off": off, "pair_list": pair}
    assert_prefill_routing(got, ref, near)


def test_prefill_route_ties_break_to_lower_id():
    cfg = LayerConfig("ties", FMT_NVFP4, H=256, E=16, k=4, I=128)
    hl = synth.make_layer(cfg, seed=3)
    for r in (5, 9, 12):
        hl.router_w[r] = hl.router_w[2]
    dl = to_device(hl)
    x = synth.make_tokens(cfg, 40, seed=3)
    got = G.route(dl, x)
    l32, near, idx, w = M.route(x, hl.router_w, None, cfg.k)
    cnt, off, pair = M.dispatch(idx, cfg.E)
    assert_prefill_routing(got, {"logits": l32, "topk_idx": idx, "topk_w": w, "expert_cnt": cnt,
                                 "expert_off": off, "pair_list": pair}, near)


# -------------------------------------------------------------------- layer ----

SMALL = [
    LayerConfig("p_tiny", FMT_NVFP4, H=256, E=6, k=2, I=256),
    LayerConfig("p_rows3", FMT_NVFP4, H=384, E=5, k=3, I=384),
    LayerConfig("p_skew", FMT_NVFP4, H=512, E=24, k=4, I=128, zipf_s=1.1),
    LayerConfig("p_mxfp4", FMT_MXFP4, H=640, E=7, k=2, I=256),
    LayerConfig("p_int4", FMT_INT4_G64, H=384, E=9, k=3, I=384, zipf_s=1.1),
    # shared experts of every format (dense over all tokens), and the formats whose scale is applied
    # per group in FP32 (int8 g64, FP8 b128, int4 g128) as routed experts
    LayerConfig("p_nvfp4_fp8", FMT_NVFP4, H=512, E=8, k=2, I=256, shared_fmt=FMT_FP8_B128, shared_I=384),
    LayerConfig("p_int4_int8", FMT_INT4_G64, H=384, E=6, k=3, I=256, shared_fmt=FMT_INT8_G64, shared_I=256),
    LayerConfig("p_int8_nvfp4", FMT_INT8_G64, H=256, E=5, k=2, I=128, shared_fmt=FMT_NVFP4, shared_I=256),
    LayerConfig("p_fp8_mxfp4", FMT_FP8_B128, H=384, E=6, k=2, I=256, shared_fmt=FMT_MXFP4, shared_I=128),
    LayerConfig("p_g128", FMT_INT4_G128, H=512, E=7, k=3, I=256, shared_fmt=FMT_INT4_G128, shared_I=256),
    LayerConfig("p_mx_int4", FMT_MXFP4, H=256, E=4, k=2, I=128, shared_fmt=FMT_INT4_G64, shared_I=128),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c.name for c in SMALL])
@pytest.mark.parametrize("T", [1, 17, 300])
def test_prefill_small_shapes(cfg, T):
    hl = synth.make_layer(cfg, seed=7)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, T, seed=7, batch=T)
    y, routing = G.decode(dl, x, prefill=True)
    ref = M.layer_forward(hl, x)
    _check_y(y, ref["y_bits"])
    assert_prefill_routing(routing, ref, ref["near_midpoint"])


# the fold-scales lever: layers with int8 g64 / FP8 b128 / int4 g128 experts, routed or shared
FOLD = [c for c in SMALL if {c.fmt, c.shared_fmt} & {FMT_INT8_G64, FMT_FP8_B128, FMT_INT4_G128}]


@pytest.mark.parametrize("cfg", FOLD, ids=[c.name for c in FOLD])
@pytest.mark.parametrize("T", [1, 17, 300])
def test_prefill_fold_scales_matches_oracle(cfg, T):
    hl = synth.make_layer(cfg, seed=9)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, T, seed=9, batch=T)
    y, routing = G.decode(dl, x, prefill=True, fold_scales=1)
    ref = M.layer_forward(hl, x, fold_scales=True)
    _check_y(y, ref["y_bits"])
    assert_prefill_routing(routing, ref, ref["near_midpoint"])


def test_prefill_fold_scales_is_a_lever():
    # on int8 routed experts the lever changes the output (not bitwise the exact chain) ...
    cfg = next(c for c in SMALL if c.name == "p_int8_nvfp4")
    hl = synth.make_layer(cfg, seed=10)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, 300, seed=10, batch=3)
    y_fold, _ = G.decode(dl, x, prefill=True, fold_scales=1)
    y_exact, _ = G.decode(dl, x, prefill=True)
    assert not np.array_equal(y_fold, y_exact)
    _check_y(y_exact, M.layer_forward(hl, x)["y_bits"])
    # ... and leaves a layer of exactly folded formats (NVFP4 routed, no shared expert) bit for bit
    cfg2 = SMALL[2]
    hl2 = synth.make_layer(cfg2, seed=10)
    dl2 = to_device(hl2)
    x2 = synth.make_tokens(cfg2, 300, seed=10, batch=4)
    assert np.array_equal(G.decode(dl2, x2, prefill=True, fold_scales=1)[0], G.decode(dl2, x2, prefill=True)[0])


@pytest.mark.parametrize("name,T,tokens", [("decode_int4", 384, [0, 200, 383]),
                                           ("decode_nvfp4", 1024, [0, 511, 1023])])
def test_prefill_fold_scales_full_size_sampled(name, T, tokens):
    """The lever on the int4 g64 layer's int8 g64 shared expert and the NVFP4 layer's FP8 b128 shared
    expert at full size, sampled tokens."""
    hl = G.host_layer(name)
    dl = G.device_layer(name)
    x = synth.make_tokens(hl.cfg, T, seed=1, batch=T)
    y, routing = G.decode(dl, x, prefill=True, fold_scales=1)
    ref = M.layer_forward(hl, x, tokens=tokens, fold_scales=True)
    _check_y(y, ref["y_bits"], tokens)
    assert_prefill_routing(routing, ref, ref["near_midpoint"])


# the FP8-activation lever: layers with an FP8 b128 expert, routed or shared
FP8A = [c for c in SMALL if FMT_FP8_B128 in (c.fmt, c.shared_fmt)]


@pytest.mark.parametrize("cfg", FP8A, ids=[c.name for c in FP8A])
@pytest.mark.parametrize("T", [1, 17, 300])
def test_prefill_fp8_act_matches_oracle(cfg, T):
    hl = synth.make_layer(cfg, seed=11)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, T, seed=11, batch=T)
    y, routing = G.decode(dl, x, prefill=True, fp8_act=1)
    ref = M.layer_forward(hl, x, fp8_act=True)
    _check_y(y, ref["y_bits"])
    assert_prefill_routing(routing, ref, ref["near_midpoint"])


def test_prefill_fp8_act_is_a_lever_and_composes_with_fold_scales():
    cfg = next(c for c in SMALL if c.name == "p_fp8_mxfp4")
    hl = synth.make_layer(cfg, seed=12)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, 300, seed=12, batch=5)
    y_f8, _ = G.decode(dl, x, prefill=True, fp8_act=1)
    y_exact, _ = G.decode(dl, x, prefill=True)
    assert not np.array_equal(y_f8, y_exact)
    # both levers: the FP8 b128 routed experts take the FP8-activation path (precedence), so the output
    # equals the FP8-activation lever alone
    y_both, _ = G.decode(dl, x, prefill=True, fp8_act=1, fold_scales=1)
    assert np.array_equal(y_both, y_f8)
    _check_y(y_both, M.layer_forward(hl, x, fp8_act=True, fold_scales=True)["y_bits"])
    # an NVFP4 layer without an FP8 expert is left bit for bit
    cfg2 = SMALL[2]
    hl2 = synth.make_layer(cfg2, seed=12)
    dl2 = to_device(hl2)
    x2 = synth.make_tokens(cfg2, 300, seed=12, batch=6)
    assert np.array_equal(G.decode(dl2, x2, prefill=True, fp8_act=1)[0], G.decode(dl2, x2, prefill=True)[0])


def test_prefill_fp8_act_full_size_sampled():
    """The lever on the NVFP4 decode layer's FP8 b128 shared expert at full size, sampled tokens."""
    hl = G.host_layer("decode_nvfp4")
    dl = G.device_layer("decode_nvfp4")
    T, tokens = 1024, [0, 511, 1023]
    x = synth.make_tokens(hl.cfg, T, seed=2, batch=T)
    y, routing = G.decode(dl, x, prefill=True, fp8_act=1)
    ref = M.layer_forward(hl, x, tokens=tokens, fp8_act=True)
    _check_y(y, ref["y_bits"], tokens)
    assert_prefill_routing(routing, ref, ref["near_midpoint"])


@pytest.mark.parametrize("T,tokens", [(256, [0, 37, 255]), (4096, [0, 1, 2047, 4095])])
def test_prefill_workload_matches_oracle(T, tokens):
    hl = G.host_layer("prefill_nvfp4")
    dl = G.device_layer("prefill_nvfp4")
    x = synth.make_tokens(hl.cfg, T, seed=0, batch=T)
    y, routing = G.decode(dl, x, prefill=True)
    ref = M.layer_forward(hl, x, tokens=tokens)
    _check_y(y, ref["y_bits"], tokens)
    assert_prefill_routing(routing, ref, ref["near_midpoint"])
    assert np.isfinite(F.bf16_to_f64(y)).all()


def test_prefill_deterministic_and_batch_invariant():
    cfg = SMALL[2]
    hl = synth.make_layer(cfg, seed=8)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, 300, seed=8, batch=1)
    y1, _ = G.decode(dl, x, prefill=True)
    y2, _ = G.decode(dl, x, prefill=True)
    assert np.array_equal(y1, y2)
    y_part, _ = G.decode(dl, x[100:160], prefill=True)
    assert np.array_equal(y_part, y1[100:160])


@pytest.mark.parametrize("name,T,tokens", [("decode_mxfp4", 512, [0, 255, 511]),
                                           ("decode_int4", 384, [0, 200, 383]),
                                           ("decode_nvfp4", 1024, [0, 511, 1023])])
def test_prefill_decode_layers_at_full_size_sampled(name, T, tokens):
    """Prefill of the MXFP4, int4 g64 (+ int8 g64 shared) and NVFP4 (+ FP8 b128
    shared) decode layers at full size, sampled tokens."""
    hl = G.host_layer(name)
    dl = G.device_layer(name)
    cfg = hl.cfg
    x = synth.make_tokens(cfg, T, seed=0, batch=T)
    y, routing = G.decode(dl, x, prefill=True)
    ref = M.layer_forward(hl, x, tokens=tokens)
    _check_y(y, ref["y_bits"], tokens)
    assert_prefill_routing(routing, ref, ref["near_midpoint"])


def _spread_rows(qm, fmt, drops):
    """Lower one scale block of every third row by each of `drops` powers of two
    (MXFP4: E8M0 code; int4 g64: the BF16 scale's exponent)."""
    qm = synth.QMat(qm.fmt, qm.N, qm.K, qm.data.copy(), qm.scales.copy(), qm.ts.copy())
    rows = np.arange(0, qm.N, 3)
    nblk = qm.scales.shape[2]
    for j, drop in enumerate(drops):
        blk = np.arange(j, nblk, 2 * len(drops))
        sub = qm.scales[:, rows[:, None], blk[None, :]].astype(np.int32)
        if fmt == FMT_MXFP4:
            new = np.maximum(sub - drop, 1)
        else:
            ex = (sub >> 7) & 0xFF
            new = (sub & 0x807F) | (np.maximum(ex - drop, 1) << 7)
        qm.scales[:, rows[:, None], blk[None, :]] = new.astype(qm.scales.dtype)
    return qm


@pytest.mark.parametrize("fmt", [FMT_MXFP4, FMT_INT4_G64])
def test_prefill_wide_scale_spreads(fmt):
    """Blocks 2^-22, 2^-24 and 2^-30 below their row's largest scale: the first
    fold exactly, the second exactly (int4) or rounded to f16's subnormal grid
    (MXFP4), the third drop out; all stay inside the output tolerance."""
    cfg = LayerConfig(f"p_spread_{fmt}", fmt, H=512, E=6, k=2, I=256)
    hl = synth.make_layer(cfg, seed=4)
    for attr in ("gate", "up", "down"):
        setattr(hl, attr, _spread_rows(getattr(hl, attr), fmt, (22, 24, 30)))
    dl = to_device(hl)
    x = synth.make_tokens(cfg, 200, seed=4, batch=200)
    y, routing = G.decode(dl, x, prefill=True)
    ref = M.layer_forward(hl, x)
    _check_y(y, ref["y_bits"])


@pytest.mark.parametrize("case", ["w4a4_shared", "w4a4_mxfp4", "w4a4_int8"])
def test_prefill_unsupported_is_reported(case):
    """The W4A4 lever is implemented for NVFP4 (act_quant 1) and MXFP4 (act_quant 2)
    routed experts without a shared expert, each on its own format: other
    layers report MOE_ERR_UNSUPPORTED before any launch."""
    if case == "w4a4_shared":
        cfg = LayerConfig("p_u1", FMT_NVFP4, H=256, E=4, k=2, I=256, shared_fmt=FMT_FP8_B128, shared_I=128)
    elif case == "w4a4_mxfp4":
        cfg = LayerConfig("p_u2", FMT_MXFP4, H=256, E=4, k=2, I=256)
    else:
        cfg = LayerConfig("p_u3", FMT_INT8_G64, H=256, E=4, k=2, I=256)
    dl = to_device(synth.make_layer(cfg, seed=1))
    x = G.x_device(synth.make_tokens(cfg, 20, seed=1))
    y = torch.zeros((20, cfg.H), dtype=torch.int16, device="cuda")
    ws = G.new_ws(dl, 20, 1)
    st = B.moe_prefill_forward(dl, x, 20, y, ws, raise_on_error=False, act_quant=1)
    assert st == B.MOE_ERR_UNSUPPORTED
    if cfg.fmt == FMT_MXFP4:   # MXFP4 activations on MXFP4 weights is supported; not on the others
        return
    st = B.moe_prefill_forward(dl, x, 20, y, ws, raise_on_error=False, act_quant=2)
    assert st == B.MOE_ERR_UNSUPPORTED


# ------------------------------------------------------------ W4A4 lever ----

W4A4 = [
    LayerConfig("w4_small", FMT_NVFP4, H=512, E=6, k=2, I=256),
    LayerConfig("w4_skew", FMT_NVFP4, H=768, E=20, k=4, I=512, zipf_s=1.1),
    # MXFP4 weights with MXFP4 activations (act_quant 2)
    LayerConfig("w4_mx_small", FMT_MXFP4, H=512, E=6, k=2, I=256),
    LayerConfig("w4_mx_skew", FMT_MXFP4, H=768, E=20, k=4, I=512, zipf_s=1.1),
]


def _aq(cfg):
    """The W4A4 lever's activation format for a layer: 2 (MXFP4) for MXFP4 weights, else 1 (NVFP4)."""
    return 2 if cfg.fmt == FMT_MXFP4 else 1


# Measured share of W4A4 outputs outside max(2 BF16 ulp, 1e-3) of the oracle's W4A4 mode (which
# quantises the FP64 h): a few per mille, from the blocks the staged check below explains.
W4A4_OUTLIER_CAP = 0.01


def _bf16_neighbours(v):
    """The BF16 values just below and just above each FP64 value (equal when v is a BF16 value)."""
    b = F.f64_to_bf16_bits(v).astype(np.int64)
    r = F.bf16_to_f64(b.astype(np.uint16))
    lo = np.where(r <= v, r, F.bf16_to_f64(np.where(b & 0x8000, b + 1, b - 1).astype(np.uint16)))
    hi = np.where(r >= v, r, F.bf16_to_f64(np.where(b & 0x8000, b - 1, b + 1).astype(np.uint16)))
    return lo, hi


def _check_w4a4(hl, x_bits, y_bits, routing, tokens=None, aq=1):
    """W4A4 parity in two exact stages (aq 1: NVFP4 activations in 16-element blocks; aq 2: MXFP4
    activations in 32-element blocks).
    (1) Down projection and combine: y equals, within max(2 BF16 ulp, 1e-3) everywhere, the oracle's
        down projection and weighted combine applied to the GPU's own FP4 h (codes and scales read
        from the workspace).
    (2) Gate/up and the h quantiser: the GPU's h codes and scales equal the oracle's (the activation
        rule applied to bf16(silu(g) * u) of the quantised token, in FP64) on every block,
        except blocks where some element's unrounded h lies within 2^-12 (relative) of a BF16
        rounding midpoint and one choice of BF16 neighbours for those elements reproduces the GPU's
        block exactly: the GPU reaches h with FP32 accumulation, so it may round such an h the
        other way.  Any other difference fails.
    Returns the share of outputs outside the 2-ulp bar of the oracle's own W4A4 result."""
    cfg = hl.cfg
    k, I, H = cfg.k, cfg.I, cfg.H
    T = x_bits.shape[0]
    want = np.arange(T) if tokens is None else np.asarray(sorted(tokens))
    want_set = set(int(t) for t in want)
    pair, off, w = routing["pair_list"], routing["expert_off"], routing["topk_w"]
    codes = np.empty((T * k, I), dtype=np.uint8)
    codes[:, 0::2] = routing["h_codes"] & 0xF
    codes[:, 1::2] = routing["h_codes"] >> 4
    sc = routing["h_scales"]
    quantize = M.mxfp4_quantize_act if aq == 2 else M.nvfp4_quantize_act
    dequantize = M.mxfp4_dequantize_act if aq == 2 else M.nvfp4_dequantize_act
    nb = 32 if aq == 2 else 16
    hq_gpu = dequantize(codes, sc)
    Xq = M.act_fake_quant(F.bf16_to_f64(x_bits), aq)
    acc = {int(t): np.zeros(H) for t in want}
    unexplained, mismatched, blocks = [], 0, 0
    for e in range(cfg.E):
        pos = [q for q in range(off[e], off[e + 1]) if int(pair[q]) // k in want_set]
        if not pos:
            continue
        Wg, Wu, Wd = (F.decode_qmat(hl.gate, e), F.decode_qmat(hl.up, e), F.decode_qmat(hl.down, e))
        rows = np.array([int(pair[q]) // k for q in pos])
        h_pre = M.silu(Xq[rows] @ Wg.T) * (Xq[rows] @ Wu.T)
        q_or, s_or = quantize(F.round_bf16(h_pre))
        P = hq_gpu[pos] @ Wd.T
        for i, q in enumerate(pos):
            t, j = divmod(int(pair[q]), k)
            acc[t] += float(w[t, j]) * P[i]
            for b in range(I // nb):
                blocks += 1
                sl = slice(nb * b, nb * b + nb)
                if s_or[i, b] == sc[q, b] and np.array_equal(q_or[i, sl], codes[q, sl]):
                    continue
                mismatched += 1
                hp = h_pre[i, sl]
                lo, hi = _bf16_neighbours(hp)
                near = np.abs(hp - (lo + hi) / 2) <= 2.0 ** -12 * np.abs(hp)
                idx = np.flatnonzero(near & (lo != hi))
                ok = False
                if len(idx) <= 10:
                    base = F.round_bf16(hp)
                    for mask in range(1 << len(idx)):
                        v = base.copy()
                        for n, ii in enumerate(idx):
                            v[ii] = hi[ii] if (mask >> n) & 1 else lo[ii]
                        cq, cs = quantize(v[None, :])
                        if cs[0, 0] == sc[q, b] and np.array_equal(cq[0], codes[q, sl]):
                            ok = True
                            break
                if not ok:
                    unexplained.append((q, b))
    assert not unexplained, f"{len(unexplained)} of {blocks} h blocks differ beyond a BF16 rounding flip: {unexplained[:5]}"
    assert mismatched <= 0.02 * blocks + 2, f"{mismatched} of {blocks} h blocks differ"
    y = F.bf16_to_f64(y_bits if tokens is None else y_bits[want])
    y_stage = np.stack([acc[int(t)] for t in want])
    ok = M.within_tolerance(y, F.bf16_to_f64(F.f64_to_bf16_bits(y_stage)))
    assert ok.all(), f"{int((~ok).sum())} of {ok.size} outputs differ from the down + combine of the GPU's h"
    assert np.isfinite(y).all()
    ref = M.layer_forward(hl, x_bits, act_quant=aq, tokens=tokens)
    frac = float((~M.within_tolerance(y, F.bf16_to_f64(ref["y_bits"]))).mean())
    print(f"W4A4 (act_quant {aq}): {mismatched} of {blocks} h blocks flipped by BF16 rounding; "
          f"{frac:.2e} of outputs outside 2 ulp of the oracle's W4A4 result")
    assert frac <= W4A4_OUTLIER_CAP, frac
    return frac


@pytest.mark.parametrize("cfg", W4A4, ids=[c.name for c in W4A4])
@pytest.mark.parametrize("T", [1, 37, 300])
def test_prefill_w4a4_matches_oracle(cfg, T):
    hl = synth.make_layer(cfg, seed=9)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, T, seed=9, batch=T)
    y, routing = G.decode(dl, x, prefill=True, act_quant=_aq(cfg))
    _check_w4a4(hl, x, y, routing, aq=_aq(cfg))
    ref = M.layer_forward(hl, x, act_quant=_aq(cfg))
    assert_prefill_routing(routing, ref, ref["near_midpoint"])


def test_prefill_w4a4_mxfp4_workload_sampled():
    # the MXFP4 layer's shapes (H=4096, I=2048) with fewer experts, so that the layer stays small
    cfg = G.host_layer("decode_mxfp4").cfg.with_(name="w4_mx_wide", E=32)
    hl = synth.make_layer(cfg, seed=3)
    dl = to_device(hl)
    T = 512
    tokens = [0, 1, 255, 511]
    x = synth.make_tokens(cfg, T, seed=3, batch=T)
    y, routing = G.decode(dl, x, prefill=True, act_quant=2)
    _check_w4a4(hl, x, y, routing, tokens, aq=2)


def test_prefill_w4a4_workload_sampled():
    hl = G.host_layer("prefill_nvfp4")
    dl = G.device_layer("prefill_nvfp4")
    T = 4096
    tokens = sorted(set([0, 1, 2047, 4095] + list(np.random.default_rng(1).choice(T, 60, replace=False))))
    x = synth.make_tokens(hl.cfg, T, seed=0, batch=T)
    y, routing = G.decode(dl, x, prefill=True, act_quant=1)
    _check_w4a4(hl, x, y, routing, tokens)


def test_prefill_w4a4_differs_from_exact_chain():
    # the lever is a different computation: it must not silently run the exact chain
    cfg = W4A4[0]
    hl = synth.make_layer(cfg, seed=4)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, 64, seed=4)
    y_exact, _ = G.decode(dl, x, prefill=True)
    y_w4, _ = G.decode(dl, x, prefill=True, act_quant=1)
    assert not np.array_equal(y_exact, y_w4)
    _check_y(y_exact, M.layer_forward(hl, x)["y_bits"])
