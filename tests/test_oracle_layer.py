"""Pins for the oracle's MoE layer.

* one expert, top-1, weight 1.0 reduces to a plain SwiGLU MLP, computed here
  with torch CPU float64 ops on weights decoded independently through torch's
  float8 casts;
* the shared expert adds exactly a plain SwiGLU MLP (same independent path);
* duplicated experts: a top-2 layer whose two experts are identical equals
  the top-1 layer (the weights sum to one);
* permuting expert ids permutes the routing and leaves y unchanged;
* batch invariance: a token's output does not depend on the other tokens;
* the W4A4 activation quantizer round-trips on-grid blocks and matches
  brute force, and an independent torch quantiser (float8_e4m3fn cast of
  the block scale, round-half-even on the binade's quantum for E2M1);
* the W4A4 mode of the layer: one expert, top-1, weight 1 equals the SwiGLU
  MLP with x quantised, h rounded to BF16 and then quantised, in that order;
* planted mistakes in the oracle are caught by these pins.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import formats as F
from oracle import moe as M
from synth.configs import FMT_FP8_B128, FMT_INT4_G64, FMT_INT4_G128, FMT_INT8_G64, FMT_MXFP4, FMT_NVFP4, LayerConfig


def _torch_e2m1(codes: np.ndarray) -> torch.Tensor:
    """E2M1 codes -> float64 through torch's float8_e4m3fn decoder (bit-field re-encoding)."""
    c = torch.from_numpy(codes.astype(np.int32))
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    body = torch.where(e == 0, torch.where(m == 0, 0, 6 << 3), ((e + 6) << 3) | (m << 2))
    return ((s << 7) | body).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)


def _torch_decode(qm, e=0) -> torch.Tensor:
    """Independent decoder (torch casts + explicit layout handling), float64 [N, K]."""
    N, K, d = qm.N, qm.K, qm.data[e]
    if qm.fmt in (FMT_NVFP4, FMT_MXFP4, FMT_INT4_G64, FMT_INT4_G128):
        lo, hi = d & 0xF, d >> 4
        codes = np.stack([lo, hi], axis=-1).reshape(N, K)
    if qm.fmt == FMT_NVFP4:
        v = _torch_e2m1(codes)
        s = torch.from_numpy(qm.scales[e]).view(torch.float8_e4m3fn).to(torch.float64)
        return v * s.repeat_interleave(16, dim=1) * float(qm.ts[e])
    if qm.fmt == FMT_MXFP4:
        v = _torch_e2m1(codes)
        s = torch.from_numpy(qm.scales[e]).view(torch.float8_e8m0fnu).to(torch.float64)
        return v * s.repeat_interleave(32, dim=1)
    if qm.fmt == FMT_INT4_G64:
        q = torch.from_numpy(codes.astype(np.int8))
        q = torch.where(q >= 8, q - 16, q).to(torch.float64)
        s = torch.from_numpy(qm.scales[e].view(np.int16)).view(torch.bfloat16).to(torch.float64)
        return q * s.repeat_interleave(64, dim=1)
    if qm.fmt == FMT_INT8_G64:
        q = torch.from_numpy(d.view(np.int8)).to(torch.float64)
        s = torch.from_numpy(qm.scales[e].view(np.int16)).view(torch.bfloat16).to(torch.float64)
        return q * s.repeat_interleave(64, dim=1)
    if qm.fmt == FMT_INT4_G128:
        q = torch.from_numpy(codes.astype(np.int16)).to(torch.float64) - 8.0
        s = torch.from_numpy(qm.scales[e].view(np.int16)).view(torch.float16).to(torch.float64)
        return q * s.repeat_interleave(128, dim=1)
    if qm.fmt == FMT_FP8_B128:
        q = torch.from_numpy(d).view(torch.float8_e4m3fn).to(torch.float64)
        s = torch.from_numpy(qm.scales[e]).to(torch.float64)
        return q * s.repeat_interleave(128, 0).repeat_interleave(128, 1)
    raise ValueError


def _torch_mlp(Wg, Wu, Wd, X):
    g = X @ Wg.T
    u = X @ Wu.T
    h = torch.nn.functional.silu(g) * u
    h = h.to(torch.float32).to(torch.bfloat16).to(torch.float64)   # bf16 activation (via fp32)
    return h @ Wd.T


def _small(fmt, shared_fmt=0, E=1, k=1, H=128, I=64):
    return LayerConfig(f"small_{fmt}", fmt, H=H, E=E, k=k, I=I, shared_fmt=shared_fmt,
                       shared_I=128 if shared_fmt == FMT_FP8_B128 else (I if shared_fmt else 0))


@pytest.mark.parametrize("fmt,H,I", [(FMT_NVFP4, 128, 64), (FMT_MXFP4, 128, 64), (FMT_INT4_G64, 128, 128),
                                     (FMT_INT8_G64, 128, 128), (FMT_INT4_G128, 256, 128)])
def test_single_expert_equals_plain_swiglu_mlp(fmt, H, I):
    cfg = _small(fmt, H=H, I=I)
    lay = synth.make_layer(cfg, seed=3)
    x = synth.make_tokens(cfg, 5, seed=3)
    out = M.layer_forward(lay, x)
    assert np.all(out["topk_idx"] == 0) and np.all(out["topk_w"] == 1.0)
    X = torch.from_numpy(F.bf16_to_f64(x))
    y_ref = _torch_mlp(_torch_decode(lay.gate), _torch_decode(lay.up), _torch_decode(lay.down), X).numpy()
    ok = M.within_tolerance(F.bf16_to_f64(out["y_bits"]), y_ref, ulps=1.0, abs_tol=1e-6)
    assert ok.all(), np.abs(F.bf16_to_f64(out["y_bits"]) - y_ref).max()


@pytest.mark.parametrize("shared_fmt", [FMT_FP8_B128, FMT_INT8_G64])
def test_shared_expert_adds_plain_mlp(shared_fmt):
    cfg = _small(FMT_NVFP4, shared_fmt, E=4, k=2, H=128, I=64)
    lay = synth.make_layer(cfg, seed=4)
    x = synth.make_tokens(cfg, 3, seed=4)
    with_shared = M.layer_forward(lay, x)
    lay_ns = synth.HostLayer(cfg.with_(shared_fmt=0, shared_I=0), lay.seed, lay.router_w, lay.router_b,
                             lay.gate, lay.up, lay.down)
    without = M.layer_forward(lay_ns, x)
    X = torch.from_numpy(F.bf16_to_f64(x))
    S = _torch_mlp(_torch_decode(lay.shared_gate), _torch_decode(lay.shared_up), _torch_decode(lay.shared_down),
                   X).numpy()
    assert np.allclose(with_shared["y_f64"] - without["y_f64"], S, rtol=1e-12, atol=1e-12)


def test_sigmoid_gated_shared_expert():
    # with a gate vector the shared expert enters scaled by sigmoid(x . w_gate), computed here with torch
    # float64 (the dot of BF16 x FP32 values is exact in FP64, so its FP32 rounding is unambiguous)
    cfg = _small(FMT_NVFP4, FMT_INT8_G64, E=4, k=2, H=128, I=128)
    lay = synth.make_layer(cfg, seed=10)
    x = synth.make_tokens(cfg, 5, seed=10)
    base = M.layer_forward(lay, x)
    gw = (np.random.default_rng(10).standard_normal(cfg.H) * 0.1).astype(np.float32)
    lay_g = synth.HostLayer(cfg, lay.seed, lay.router_w, lay.router_b, lay.gate, lay.up, lay.down,
                            lay.shared_gate, lay.shared_up, lay.shared_down, extra={"shared_gate_w": gw})
    gated = M.layer_forward(lay_g, x)
    X = torch.from_numpy(F.bf16_to_f64(x))
    g = (X @ torch.from_numpy(gw.astype(np.float64))).to(torch.float32).to(torch.float64)
    sig = torch.sigmoid(g).numpy()
    S = _torch_mlp(_torch_decode(lay.shared_gate), _torch_decode(lay.shared_up), _torch_decode(lay.shared_down),
                   X).numpy()
    assert np.allclose(gated["y_f64"] - base["y_f64"], (sig[:, None] - 1.0) * S, rtol=1e-10, atol=1e-12)
    assert np.array_equal(gated["topk_idx"], base["topk_idx"])


def test_bf16_partials_round_each_expert_output():
    # the lever: y = bf16( sum_j w_j bf16(P_j) + bf16(S) ), each P_j from an independent torch float64 MLP
    cfg = _small(FMT_NVFP4, FMT_FP8_B128, E=5, k=3, H=128, I=128)
    lay = synth.make_layer(cfg, seed=12)
    x = synth.make_tokens(cfg, 6, seed=12)
    out = M.layer_forward(lay, x, bf16_partials=True)
    X = torch.from_numpy(F.bf16_to_f64(x))
    S = _torch_mlp(_torch_decode(lay.shared_gate), _torch_decode(lay.shared_up), _torch_decode(lay.shared_down),
                   X).numpy()
    y = F.round_bf16(S)
    for t in range(x.shape[0]):
        for j in range(cfg.k):
            e = int(out["topk_idx"][t, j])
            P = _torch_mlp(_torch_decode(lay.gate, e), _torch_decode(lay.up, e), _torch_decode(lay.down, e),
                           X[t:t + 1]).numpy()[0]
            y[t] += float(out["topk_w"][t, j]) * F.round_bf16(P)
    assert np.allclose(out["y_f64"], y, rtol=1e-12, atol=1e-14)
    assert not np.array_equal(out["y_f64"], M.layer_forward(lay, x)["y_f64"])


@pytest.mark.parametrize("fmt,shared_fmt,H,I", [(FMT_INT8_G64, FMT_FP8_B128, 128, 128),
                                                (FMT_INT4_G128, FMT_INT8_G64, 256, 128)])
def test_fold_scales_lever_equals_mlp_on_bf16_weights(fmt, shared_fmt, H, I):
    # the lever: every int8 g64 / FP8 b128 / int4 g128 weight enters as bf16(fp32(code x scale)); here
    # the folded weights come from torch's fp64 -> fp32 -> bf16 casts of an independent torch decode
    cfg = _small(fmt, shared_fmt, E=1, k=1, H=H, I=I)
    lay = synth.make_layer(cfg, seed=14)
    x = synth.make_tokens(cfg, 5, seed=14)
    out = M.layer_forward(lay, x, fold_scales=True)
    fold = lambda W: W.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    X = torch.from_numpy(F.bf16_to_f64(x))
    y_ref = (_torch_mlp(fold(_torch_decode(lay.gate)), fold(_torch_decode(lay.up)), fold(_torch_decode(lay.down)), X)
             + _torch_mlp(fold(_torch_decode(lay.shared_gate)), fold(_torch_decode(lay.shared_up)),
                          fold(_torch_decode(lay.shared_down)), X)).numpy()
    ok = M.within_tolerance(F.bf16_to_f64(out["y_bits"]), y_ref, ulps=1.0, abs_tol=1e-6)
    assert ok.all(), np.abs(F.bf16_to_f64(out["y_bits"]) - y_ref).max()
    assert not np.array_equal(out["y_f64"], M.layer_forward(lay, x)["y_f64"])   # not the exact chain


def test_fold_scales_lever_leaves_exactly_folded_formats():
    # NVFP4 routed experts: the lever changes nothing (their scales already fold exactly)
    cfg = _small(FMT_NVFP4, E=4, k=2, H=128, I=64)
    lay = synth.make_layer(cfg, seed=15)
    x = synth.make_tokens(cfg, 4, seed=15)
    assert np.array_equal(M.layer_forward(lay, x, fold_scales=True)["y_f64"], M.layer_forward(lay, x)["y_f64"])


def test_identical_experts_top2_equals_top1():
    cfg1 = _small(FMT_NVFP4, E=1, k=1)
    lay1 = synth.make_layer(cfg1, seed=5)
    cfg2 = cfg1.with_(E=2, k=2)
    dup = lambda q: synth.QMat(q.fmt, q.N, q.K, np.concatenate([q.data, q.data]),
                               np.concatenate([q.scales, q.scales]), np.concatenate([q.ts, q.ts]))
    rw = np.concatenate([lay1.router_w, lay1.router_w * np.float32(0.5)])
    lay2 = synth.HostLayer(cfg2, 5, rw, None, dup(lay1.gate), dup(lay1.up), dup(lay1.down))
    x = synth.make_tokens(cfg1, 4, seed=5)
    y1 = M.layer_forward(lay1, x)["y_f64"]
    o2 = M.layer_forward(lay2, x)
    assert np.allclose(o2["topk_w"].astype(np.float64).sum(1), 1.0, atol=2 ** -23)
    scale = o2["topk_w"].astype(np.float64).sum(1, keepdims=True)
    assert np.allclose(o2["y_f64"], y1 * scale, rtol=1e-12, atol=1e-15)


def test_permuting_expert_ids_permutes_routing_only():
    cfg = _small(FMT_NVFP4, E=6, k=3)
    lay = synth.make_layer(cfg, seed=6)
    x = synth.make_tokens(cfg, 7, seed=6)
    base = M.layer_forward(lay, x)
    perm = np.array([3, 5, 0, 1, 4, 2])                # new id i holds old expert perm[i]
    inv = np.argsort(perm)
    sub = lambda q: synth.QMat(q.fmt, q.N, q.K, q.data[perm], q.scales[perm], q.ts[perm])
    lp = synth.HostLayer(cfg, 6, lay.router_w[perm], None, sub(lay.gate), sub(lay.up), sub(lay.down))
    out = M.layer_forward(lp, x)
    # same experts chosen, renamed (ordering among equal logits may differ only on exact ties)
    assert np.array_equal(perm[out["topk_idx"]], base["topk_idx"]) or np.array_equal(
        np.sort(perm[out["topk_idx"]], 1), np.sort(base["topk_idx"], 1))
    assert np.array_equal(out["y_bits"], base["y_bits"])
    assert np.array_equal(inv[base["topk_idx"]], out["topk_idx"])


def test_batch_invariance():
    cfg = _small(FMT_MXFP4, E=5, k=2)
    lay = synth.make_layer(cfg, seed=7)
    x = synth.make_tokens(cfg, 6, seed=7)
    full = M.layer_forward(lay, x)
    for t in (0, 3, 5):
        one = M.layer_forward(lay, x[t:t + 1])
        assert np.array_equal(one["y_bits"][0], full["y_bits"][t])
        assert np.array_equal(one["topk_idx"][0], full["topk_idx"][t])
    sub = M.layer_forward(lay, x, tokens=[5, 1])
    assert np.array_equal(sub["y_bits"], full["y_bits"][[1, 5]])


def test_nvfp4_act_quantizer_pins():
    # on-grid block: values e2m1 * s with amax = 6 s -> exact round trip
    s = 0.75                                          # e4m3 0.75 (exact), amax/6 = 0.75
    codes = np.array([7, 1, 2, 3, 4, 5, 6, 0, 9, 10, 11, 12, 13, 14, 15, 8])
    a = F.E2M1_TABLE[codes] * s
    q, sc = M.nvfp4_quantize_act(a[None, :])
    assert F.E4M3_TABLE[sc[0, 0]] == s
    assert np.array_equal(M.nvfp4_dequantize_act(q, sc)[0], a)
    # zero block -> zero scale, zero codes
    q0, s0 = M.nvfp4_quantize_act(np.zeros((1, 16)))
    assert s0[0, 0] == 0 and np.all(q0 == 0)
    # brute force on random blocks: each value is the nearest E2M1 multiple of the block scale
    rng = np.random.default_rng(9)
    A = F.round_bf16(rng.standard_normal((64, 32)))
    q, sc = M.nvfp4_quantize_act(A)
    D = M.nvfp4_dequantize_act(q, sc)
    for r in range(64):
        for b in range(2):
            blk = A[r, b * 16:(b + 1) * 16]
            sv = F.E4M3_TABLE[sc[r, b]]
            amax6 = float(np.float32(np.abs(blk).max() / 6.0))
            assert sv == F.E4M3_TABLE[F.e4m3_encode_rne_sat(np.array([amax6]))[0]]
            for i in range(16):
                y = float(np.float32(blk[i] / sv))
                cand = np.abs(min(abs(y), 6.0) - F.E2M1_GRID)
                nearest = np.flatnonzero(cand == cand.min())       # one code, or two on a tie
                pick = nearest[0] if len(nearest) == 1 else nearest[nearest % 2 == 0][0]   # tie: even code
                assert abs(D[r, b * 16 + i]) / sv == F.E2M1_GRID[pick]


def test_mxfp4_act_quantizer_pins():
    # on-grid block: values e2m1 * 2^e with amax = 6 * 2^e -> exact round trip, scale code e + 127
    codes = np.array([7, 1, 2, 3, 4, 5, 6, 0, 9, 10, 11, 12, 13, 14, 15, 8] * 2)
    for e in (-9, -1, 0, 3):
        a = F.E2M1_TABLE[codes] * 2.0 ** e
        q, sc = M.mxfp4_quantize_act(a[None, :])
        assert sc[0, 0] == e + 127
        assert np.array_equal(M.mxfp4_dequantize_act(q, sc)[0], a)
    # zero block -> scale code 127 (2^0), zero codes
    q0, s0 = M.mxfp4_quantize_act(np.zeros((1, 32)))
    assert s0[0, 0] == 127 and np.all(q0 == 0)
    # brute force: e is the smallest integer with 6 * 2^e >= amax (boundaries included), each value the
    # nearest E2M1 multiple of 2^e (ties to the even code)
    rng = np.random.default_rng(21)
    A = F.round_bf16(rng.standard_normal((48, 64)) * np.exp(rng.uniform(-12, 12, (48, 1))))
    A[0, :32] = F.round_bf16(np.linspace(-6.0, 6.0, 32) * 2.0 ** -4)     # amax exactly 6 * 2^-4
    A[1, :32] = A[0, :32] * (1 + 2.0 ** -7)                               # just above: the next exponent
    q, sc = M.mxfp4_quantize_act(A)
    D = M.mxfp4_dequantize_act(q, sc)
    for r in range(48):
        for b in range(2):
            blk = A[r, b * 32:(b + 1) * 32]
            amax = np.abs(blk).max()
            e = next(e for e in range(-140, 140) if 6.0 * 2.0 ** e >= amax) if amax > 0 else 0
            assert sc[r, b] == e + 127
            for i in range(32):
                y = blk[i] / 2.0 ** e
                cand = np.abs(min(abs(y), 6.0) - F.E2M1_GRID)
                nearest = np.flatnonzero(cand == cand.min())
                pick = nearest[0] if len(nearest) == 1 else nearest[nearest % 2 == 0][0]
                assert abs(D[r, b * 32 + i]) / 2.0 ** e == F.E2M1_GRID[pick]
    assert sc[0, 0] == 123 and sc[1, 0] == 124
    # the synthetic checkpoints' MXFP4 encoder (plain C, the same rule for weights) agrees on every
    # code and scale of the same rows
    data, scales, _ = synth.quantize(FMT_MXFP4, A.astype(np.float32))
    codes_c = F.unpack_nibbles(data)
    assert np.array_equal(scales, sc)
    assert np.array_equal(codes_c & 7, q & 7)                               # magnitudes
    nz = (codes_c & 7) != 0
    assert np.array_equal((codes_c & 8)[nz], (q & 8)[nz])                  # signs of the non-zero codes


def _torch_fp8_quant(A: torch.Tensor):
    """Per-token 1x128 E4M3 codes and FP32 scales, written with torch float32 arithmetic and torch's own
    float -> float8_e4m3fn cast (an independent E4M3 encoder): s = amax / 448, code = e4m3(a / s)."""
    *lead, K = A.shape
    a32 = A.to(torch.float32).reshape(*lead, K // 128, 128)
    s = a32.abs().amax(dim=-1) / 448.0
    q = a32 / torch.where(s > 0, s, torch.ones_like(s))[..., None]
    codes = q.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    codes = torch.where((s > 0)[..., None], codes, torch.zeros_like(codes))
    return codes.reshape(*lead, K), s


def _fp8_pin_failures(quant=None) -> int:
    """Mismatches of the oracle's FP8 activation quantiser against the torch version, over random BF16
    rows at many magnitudes and hand-made blocks (zeros, one non-zero, values on the E4M3 grid, tiny
    values that land on E4M3 subnormal codes)."""
    quant = quant or M.fp8_quantize_act
    rng = np.random.default_rng(33)
    A = F.round_bf16(rng.standard_normal((40, 384)) * np.exp(rng.uniform(-20, 20, (40, 1))))
    A[0, :128] = 0.0
    A[1, :128] = 0.0
    A[1, 77] = -3.5
    A[2, :128] = F.round_bf16(F.E4M3_TABLE[np.arange(128) % 126] * 2.0 ** -3)   # every magnitude on the grid
    A[3, :128] = F.round_bf16(rng.standard_normal(128) * 1e-3)
    A[3, 5] = 40.0                                                                # small codes, subnormals
    codes, s = quant(A)
    tc, ts = _torch_fp8_quant(torch.from_numpy(A))
    bad = int(np.sum(codes != tc.numpy())) + int(np.sum(s.view(np.uint32) != ts.numpy().view(np.uint32)))
    return bad


def test_fp8_act_quantizer_pins():
    assert _fp8_pin_failures() == 0
    rng = np.random.default_rng(34)
    A = F.round_bf16(rng.standard_normal((16, 256)) * np.exp(rng.uniform(-8, 8, (16, 1))))
    codes, s = M.fp8_quantize_act(A)
    D = M.fp8_dequantize_act(codes, s)
    blk = lambda v: v.reshape(16, 2, 128)
    # each block's largest magnitude takes the largest code (+-448), so it comes back to 448 s
    assert np.array_equal(np.abs(blk(D)).max(axis=-1), 448.0 * s.astype(np.float64))
    # every value within half an E4M3 step: 2^-4 relative, or 2^-10 s on the subnormal grid
    assert np.all(np.abs(D - A) <= np.maximum(2.0 ** -4 * np.abs(A), np.repeat(s, 128, axis=1) * 2.0 ** -10))
    # zero block: zero scale and codes
    c0, s0 = M.fp8_quantize_act(np.zeros((1, 128)))
    assert s0[0, 0] == 0 and np.all(c0 == 0)


def _fp8_scale_240(a):
    # wrong: the E4M3 "fnuz" maximum 240 instead of 448
    return _fp8_scaled(a, 240.0)


def _fp8_scaled(a, top):
    a = np.asarray(a, dtype=np.float64)
    *lead, K = a.shape
    blk = a.reshape(*lead, K // 128, 128)
    s = (np.abs(blk).max(axis=-1).astype(np.float32) / np.float32(top)).astype(np.float32)
    q = (blk.astype(np.float32) / np.where(s > 0, s, 1)[..., None]).astype(np.float64)
    return np.where((s > 0)[..., None], F.e4m3_encode_rne_sat(q), 0).reshape(*lead, K).astype(np.uint8), s


def _fp8_truncating(a):
    _, s = _ORIG["fp8"](a)
    a = np.asarray(a, dtype=np.float64)
    *lead, K = a.shape
    q = (a.reshape(*lead, K // 128, 128).astype(np.float32) / np.where(s > 0, s, 1)[..., None]).astype(np.float64)
    # wrong: round toward zero on the E4M3 grid
    mag = np.abs(q).reshape(-1)
    grid = F.E4M3_TABLE[:127]
    idx = np.clip(np.searchsorted(grid, mag, side="right") - 1, 0, 126)
    tc = np.where(q.reshape(-1) < 0, idx | 0x80, idx).astype(np.uint8)
    tc = np.where(idx == 0, 0, tc)
    return np.where((s > 0)[..., None], tc.reshape(q.shape), 0).reshape(*lead, K).astype(np.uint8), s


def _torch_fp8_fake(A: torch.Tensor) -> torch.Tensor:
    codes, s = _torch_fp8_quant(A)
    v = codes.view(torch.float8_e4m3fn).to(torch.float64).reshape(*A.shape[:-1], A.shape[-1] // 128, 128)
    return (v * s.to(torch.float64)[..., None]).reshape(A.shape)


@pytest.mark.parametrize("shared", [False, True])
def test_fp8_act_lever_equals_quantised_mlp(shared):
    # an FP8 b128 expert (routed, or the shared expert beside an NVFP4 routed one) under the lever: x and
    # h (after its BF16 rounding) quantised by the torch E4M3 version, exact weights
    fmt, sfmt = (FMT_NVFP4, FMT_FP8_B128) if shared else (FMT_FP8_B128, 0)
    cfg = _small(fmt, sfmt, E=1, k=1, H=256, I=128)
    lay = synth.make_layer(cfg, seed=16)
    x = synth.make_tokens(cfg, 5, seed=16)
    out = M.layer_forward(lay, x, fp8_act=True)
    X = torch.from_numpy(F.bf16_to_f64(x))

    def mlp_fp8(Wg, Wu, Wd):
        Xq = _torch_fp8_fake(X)
        h = (torch.nn.functional.silu(Xq @ Wg.T) * (Xq @ Wu.T)).to(torch.float32).to(torch.bfloat16)
        return _torch_fp8_fake(h.to(torch.float64)) @ Wd.T

    if shared:
        y_ref = (_torch_mlp(_torch_decode(lay.gate), _torch_decode(lay.up), _torch_decode(lay.down), X)
                 + mlp_fp8(_torch_decode(lay.shared_gate), _torch_decode(lay.shared_up), _torch_decode(lay.shared_down)))
    else:
        y_ref = mlp_fp8(_torch_decode(lay.gate), _torch_decode(lay.up), _torch_decode(lay.down))
    ok = M.within_tolerance(F.bf16_to_f64(out["y_bits"]), y_ref.numpy(), ulps=1.0, abs_tol=1e-6)
    assert ok.all(), np.abs(F.bf16_to_f64(out["y_bits"]) - y_ref.numpy()).max()
    assert not np.array_equal(out["y_f64"], M.layer_forward(lay, x)["y_f64"])
    # NVFP4 experts are untouched by the lever
    if shared:
        lay_ns = synth.HostLayer(cfg.with_(shared_fmt=0, shared_I=0), lay.seed, lay.router_w, lay.router_b,
                                 lay.gate, lay.up, lay.down)
        assert np.array_equal(M.layer_forward(lay_ns, x, fp8_act=True)["y_f64"], M.layer_forward(lay_ns, x)["y_f64"])


def _torch_mxfp4_fake_quant(A: torch.Tensor) -> torch.Tensor:
    """MXFP4 quantise-dequantise of BF16-valued rows in 32-element blocks, written independently of
    the oracle: the exponent as ceil(log2(amax / 6)) in float64 (exact at the powers of two), the
    E2M1 code by round-half-even on the binade's quantum, saturating at 6."""
    n, K = A.shape
    B = A.reshape(n, K // 32, 32).to(torch.float64)
    amax = B.abs().amax(dim=-1)
    e = torch.where(amax > 0, torch.ceil(torch.log2(amax / 6.0)), torch.zeros_like(amax))
    s = torch.pow(2.0, e)
    y = B / s[..., None]
    ay = y.abs()
    quantum = torch.where(ay < 2, 0.5, torch.where(ay < 4, 1.0, 2.0))
    v = torch.clamp(torch.round(ay / quantum) * quantum, max=6.0) * torch.sign(y)
    return (v * s[..., None]).reshape(n, K)


def _torch_nvfp4_fake_quant(A: torch.Tensor) -> torch.Tensor:
    """NVFP4 quantise-dequantise of BF16-valued rows in 16-element blocks, written independently of
    the oracle: the block scale through torch's float8_e4m3fn cast of the FP32 quotient amax / 6, the
    FP32 quotient a / s by torch's float32 division (the scale saturates at 448, where torch's cast
    would give NaN), and the E2M1 code by round-half-even on the
    binade's quantum (0.5 below 2, 1 below 4, 2 above) saturating at 6."""
    n, K = A.shape
    B = A.reshape(n, K // 16, 16)
    amax = B.abs().amax(dim=-1)
    s = torch.clamp(amax.to(torch.float32) / 6.0, max=448.0).to(torch.float8_e4m3fn).to(torch.float32)  # saturating
    y = B.to(torch.float32) / s[..., None]
    ay = y.abs().to(torch.float64)
    quantum = torch.where(ay < 2, 0.5, torch.where(ay < 4, 1.0, 2.0))
    v = torch.clamp(torch.round(ay / quantum) * quantum, max=6.0) * torch.sign(y).to(torch.float64)
    v = torch.where(s[..., None] > 0, v, torch.zeros_like(v))
    return (v * s[..., None].to(torch.float64)).reshape(n, K)


def _torch_w4a4_mlp(Wg, Wu, Wd, X, quant=None):
    """The W4A4 lever's order: x quantised, gate and up, h = bf16(silu(g) * u), h quantised, down."""
    quant = quant or _torch_nvfp4_fake_quant
    Xq = quant(X)
    g = Xq @ Wg.T
    u = Xq @ Wu.T
    h = torch.from_numpy(F.round_bf16((torch.nn.functional.silu(g) * u).numpy()))
    return quant(h) @ Wd.T


@pytest.mark.parametrize("fmt,H,I,aq", [(FMT_NVFP4, 256, 128, 1), (FMT_MXFP4, 256, 128, 1),
                                        (FMT_MXFP4, 256, 128, 2)])
def test_w4a4_single_expert_equals_quantised_swiglu_mlp(fmt, H, I, aq):
    # one expert, top-1, weight 1: the W4A4 mode is the SwiGLU MLP with x and h replaced by their
    # NVFP4 (aq 1) or MXFP4 (aq 2) quantise-dequantise (activations, page 5 weekly update: W4A4
    # prefill is opt-in)
    cfg = _small(fmt, H=H, I=I)
    lay = synth.make_layer(cfg, seed=8)
    x = synth.make_tokens(cfg, 24, seed=8)
    out = M.layer_forward(lay, x, act_quant=aq)
    X = torch.from_numpy(F.bf16_to_f64(x))
    y_ref = _torch_w4a4_mlp(_torch_decode(lay.gate), _torch_decode(lay.up), _torch_decode(lay.down), X,
                            _torch_mxfp4_fake_quant if aq == 2 else None).numpy()
    ok = M.within_tolerance(F.bf16_to_f64(out["y_bits"]), y_ref, ulps=1.0, abs_tol=1e-6)
    assert ok.all(), np.abs(F.bf16_to_f64(out["y_bits"]) - y_ref).max()
    # and the lever changes the result: the exact chain differs from it
    exact = M.layer_forward(lay, x)
    assert not np.array_equal(exact["y_bits"], out["y_bits"])


def test_mxfp4_fake_quant_matches_torch_on_hard_blocks():
    rng = np.random.default_rng(13)
    A = F.round_bf16(rng.standard_normal((40, 64)) * np.exp(rng.uniform(-30, 30, (40, 1))))
    A[0, :32] = 0.0
    A[1, :32] = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 4) * np.array([1, -1] * 16)  # 2^0, ties
    A[2, :32] = np.array([4.0, 5.0, 6.0, -6.0] * 8) * 8.0                   # 2^3: ties at 5 * 8
    got = M.mxfp4_fake_quant(A)
    ref = _torch_mxfp4_fake_quant(torch.from_numpy(A)).numpy()
    assert np.array_equal(got, ref)


def test_w4a4_fake_quant_matches_torch_on_hard_blocks():
    # zero blocks, blocks at the E2M1 tie points and at saturation, huge and tiny binades
    rng = np.random.default_rng(12)
    A = F.round_bf16(rng.standard_normal((40, 64)) * np.exp(rng.uniform(-20, 20, (40, 1))))
    A[0, :16] = 0.0
    A[1, :16] = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 2) * np.array([1, -1] * 8)  # amax 6: s = 1
    A[2, :16] = np.array([4.0, 5.0, 6.0, -6.0] * 4) * 3.0                  # s = 3: ties at 5 * 3
    got = M.nvfp4_fake_quant(A)
    ref = _torch_nvfp4_fake_quant(torch.from_numpy(A)).numpy()
    assert np.array_equal(got, ref)


# --------------------------------------------------- planted mistakes ----

def _run_pin(fn, *args):
    try:
        fn(*args)
        return True
    except Exception:
        return False


def _swapped_nibbles(data):
    d = np.asarray(data, dtype=np.uint8)
    out = np.empty(d.shape[:-1] + (d.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = d >> 4
    out[..., 1::2] = d & 0x0F
    return out


def _topk_ids_descending(l32, k):
    ids = -np.arange(l32.shape[1])
    return np.stack([np.lexsort((ids, -l32[t].astype(np.float64)))[:k] for t in range(l32.shape[0])]).astype(np.int32)


def _unnormalised_weights(l32, idx):
    sel = np.take_along_axis(l32.astype(np.float64), idx.astype(np.int64), axis=1)
    return np.exp(sel - l32.astype(np.float64).max(axis=1, keepdims=True)).astype(np.float32)


def _unstable_dispatch(idx, E):
    cnt, off, pair = _ORIG["dispatch"](idx, E)
    return cnt, off, np.concatenate([pair[off[e]:off[e + 1]][::-1] for e in range(E)]).astype(np.int32)


def _w4a4_variant(Wg, Wu, Wd, X, act_quant=False, quant_x=True, round_first=True, quant_h=True):
    if act_quant and quant_x:
        X = M.nvfp4_fake_quant(X)
    g = X @ Wg.T
    u = X @ Wu.T
    raw = M.silu(g) * u
    h = F.round_bf16(raw)
    if act_quant and quant_h:
        hq = M.nvfp4_fake_quant(h if round_first else raw)
    else:
        hq = h
    return h, hq @ Wd.T


def _w4a4_h_unrounded(Wg, Wu, Wd, X, act_quant=False):
    return _w4a4_variant(Wg, Wu, Wd, X, act_quant, round_first=False)


def _w4a4_x_unquantised(Wg, Wu, Wd, X, act_quant=False):
    return _w4a4_variant(Wg, Wu, Wd, X, act_quant, quant_x=False)


def _w4a4_h_unquantised(Wg, Wu, Wd, X, act_quant=False):
    return _w4a4_variant(Wg, Wu, Wd, X, act_quant, quant_h=False)


def _router_logits_bound_mask(x_bits, Wr, bias=None):
    # the mask computed from the FP64 result and its error bound, without settling the uncertain ones
    l32, _ = _ORIG["router_logits"](x_bits, Wr, bias)
    X = F.bf16_to_f64(x_bits)
    W = np.asarray(Wr, dtype=np.float32).astype(np.float64)
    d = X @ W.T
    bound = X.shape[1] * 2.0 ** -53 * (np.abs(X) @ np.abs(W).T)
    l0 = d.astype(np.float32)
    return l32, M.midpoint_distance(d, l0) <= 2.0 ** -40 * np.abs(d) + bound


def _route_bias_always_weighs(x_bits, Wr, bias, k, bias_select=False):
    return _ORIG["route"](x_bits, Wr, bias, k, False)


def _mxfp4_exponent_low(a):
    """floor(log2(amax / 6)) instead of the ceiling: values above 6 * 2^e saturate."""
    a = np.asarray(a, dtype=np.float64)
    *lead, K = a.shape
    blk = a.reshape(*lead, K // 32, 32)
    amax = np.abs(blk).max(axis=-1)
    _, p = np.frexp(np.where(amax > 0, amax, 1.0))
    e = np.where(amax > 0, p - 3, 0)
    s_code = np.clip(e + 127, 0, 254)
    codes = F.e2m1_encode_rne(blk / np.ldexp(1.0, s_code - 127)[..., None])
    return codes.reshape(*lead, K).astype(np.uint8), s_code.astype(np.uint8)


_ORIG = {"dispatch": M.dispatch, "decode": F.decode, "swiglu": M.swiglu_mlp, "router_logits": M.router_logits,
         "route": M.route, "shared_gate": M.shared_gate, "layer_forward": M.layer_forward,
         "act_fake_quant": M.act_fake_quant, "fp8": M.fp8_quantize_act}


def test_planted_mistakes_are_caught(monkeypatch):
    """Each plausible oracle mistake fails at least one pin (mistakes planted in the oracle, on the CPU)."""
    import tests.test_oracle_formats as TF
    import tests.test_oracle_router as TR

    single = (test_single_expert_equals_plain_swiglu_mlp, FMT_NVFP4, 128, 64)
    w4a4 = (test_w4a4_single_expert_equals_quantised_swiglu_mlp, FMT_NVFP4, 256, 128, 1)
    w4a4_mx = (test_w4a4_single_expert_equals_quantised_swiglu_mlp, FMT_MXFP4, 256, 128, 2)
    mistakes = {
        "nibble order": (F, "unpack_nibbles", _swapped_nibbles, [(TF.test_nvfp4_layout_hand_built,), single]),
        "silu sign": (M, "silu", lambda z: z / (1.0 + np.exp(z)), [single]),
        "dropped tensor scale": (F, "decode", lambda fmt, d, s, ts, N, K: _ORIG["decode"](fmt, d, s, 1.0, N, K),
                                 [(TF.test_nvfp4_layout_hand_built,)]),
        "tie-break reversed": (M, "topk", _topk_ids_descending, [(TR.test_topk_order_descending_then_id,)]),
        "unnormalised weights": (M, "topk_weights", _unnormalised_weights, [(TR.test_weights_identity_and_sum,)]),
        "unstable dispatch": (M, "dispatch", _unstable_dispatch, [(TR.test_dispatch_matches_plain_loop,)]),
        "gate/up swapped": (M, "swiglu_mlp", lambda Wg, Wu, Wd, X, act_quant=False: _ORIG["swiglu"](
            Wu, Wg, Wd, X, act_quant), [single]),
        "W4A4: h quantised before its BF16 rounding": (M, "swiglu_mlp", _w4a4_h_unrounded, [w4a4]),
        "W4A4: x not quantised": (M, "swiglu_mlp", _w4a4_x_unquantised, [w4a4]),
        "W4A4: h not re-quantised": (M, "swiglu_mlp", _w4a4_h_unquantised, [w4a4]),
        "MXFP4 activations: exponent one too small": (M, "mxfp4_quantize_act", _mxfp4_exponent_low,
                                                      [(test_mxfp4_act_quantizer_pins,)]),
        "MXFP4 W4A4 quantised as NVFP4": (M, "act_fake_quant", lambda a, aq: _ORIG["act_fake_quant"](
            a, 1 if aq else 0), [w4a4_mx]),
        "mask window 2^-4": (M, "near_midpoint", lambda d, l: M.midpoint_distance(d, l) <= 2.0 ** -4 * np.abs(d),
                             [(TR.test_near_midpoint_mask_flags_only_the_window, 1.0),
                              (TR.test_near_midpoint_mask_empty_at_the_decode_seeds,)]),
        "mask never set": (M, "near_midpoint", lambda d, l: np.zeros(d.shape, dtype=bool),
                           [(TR.test_near_midpoint_mask_flags_only_the_window, 1.0)]),
        "mask widened by the FP64 error bound": (M, "router_logits", _router_logits_bound_mask,
                                                 [(TR.test_near_midpoint_mask_empty_at_the_decode_seeds,)]),
        "bias weighs the mixture in bias_select mode": (M, "route", _route_bias_always_weighs,
                                                        [(TR.test_bias_select_routes_by_biased_and_weighs_by_unbiased,
                                                          8, 2)]),
        "shared gate sign (sigmoid(-g))": (M, "shared_gate", lambda x, w: 1.0 - _ORIG["shared_gate"](x, w),
                                           [(test_sigmoid_gated_shared_expert,)]),
        "bf16 partials not rounded": (M, "layer_forward", lambda *a, **kw: _ORIG["layer_forward"](
            *a, **{**kw, "bf16_partials": False}), [(test_bf16_partials_round_each_expert_output,)]),
        "FP8 activations: scale from 240 (E4M3 fnuz) instead of 448": (
            M, "fp8_quantize_act", _fp8_scale_240, [(test_fp8_act_quantizer_pins,)]),
        "FP8 activations: truncated instead of nearest-even": (
            M, "fp8_quantize_act", _fp8_truncating, [(test_fp8_act_quantizer_pins,)]),
        "FP8 lever: h not re-quantised": (M, "act_fake_quant", lambda a, aq: _ORIG["act_fake_quant"](
            a, aq) if aq != M.ACT_FP8 or a.shape[-1] != 128 else a, [(test_fp8_act_lever_equals_quantised_mlp, False)]),
        "shared expert dropped": (M, "swiglu_mlp", lambda Wg, Wu, Wd, X, act_quant=False: (
            lambda h, P: (h, P * (Wg.shape[0] != 128)))(*_ORIG["swiglu"](Wg, Wu, Wd, X, act_quant)),
            [(test_shared_expert_adds_plain_mlp, FMT_FP8_B128)]),
    }
    for name, (mod, attr, bad, pins) in mistakes.items():
        with monkeypatch.context() as mp:
            mp.setattr(mod, attr, bad)
            caught = [not _run_pin(*p) for p in pins]
        assert any(caught), f"planted mistake not caught: {name}"
