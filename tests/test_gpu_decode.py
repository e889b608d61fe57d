"""GPU parity of the decode path against the FP64 oracle, through the C ABI.

Bit-exact: decoded weights (moe_dequantize), routing indices, expert counts,
offsets and pair lists, NVFP4 activation codes.  Layer output y within
max(2 BF16 ulp, 1e-3) per element of the oracle's value.  Full sizes of the
decode workloads plus small shapes with ragged expert loads.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import formats as F
from oracle import moe as M
from quantized_moe_decode_router_gb300 import _binding as B
from quantized_moe_decode_router_gb300.device import qweight_to_device, to_device
from synth.configs import (FMT_FP8_B128, FMT_INT4_G64, FMT_INT4_G128, FMT_INT8_G64, FMT_MXFP4, FMT_NVFP4,
                           LayerConfig)
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    G.lib()


# ------------------------------------------------------------ format decode ----

def _f32_bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("fmt,N,K", [(FMT_NVFP4, 256, 512), (FMT_MXFP4, 256, 512), (FMT_INT4_G64, 256, 512),
                                     (FMT_INT8_G64, 256, 512), (FMT_FP8_B128, 256, 512), (FMT_INT4_G128, 256, 512)])
def test_dequantize_bit_exact(fmt, N, K):
    qm = synth.make_stack(fmt, 11, synth.KIND_ROUTED, 0, 0, 3, N, K)
    # adversarial codes: zero blocks, -0 nibbles, subnormal / NaN / signed scales, extreme exponents
    rng = np.random.default_rng(fmt)
    if fmt == FMT_NVFP4:
        qm.scales[1, :4, :] = np.array([0x00, 0x01, 0x07, 0x80], dtype=np.uint8)[:, None]   # 0, subnormals, -0
        qm.scales[1, 4, 0] = 0x7F                                                          # NaN scale
        qm.scales[1, 5, :] = 0xBE                                                          # negative scale
        qm.data[1, 6, :] = 0x88                                                            # -0 codes
    elif fmt == FMT_MXFP4:
        qm.scales[1, :3, :] = np.array([0, 1, 254], dtype=np.uint8)[:, None] * np.ones((1, K // 32), np.uint8)
        qm.data[1, 2, :] = rng.integers(0, 256, K // 2).astype(np.uint8) & 0x33            # avoid fp32 overflow
        qm.scales[1, 3, 0] = 255                                                           # NaN
    elif fmt == FMT_INT4_G128:
        qm.scales[1, 0, :] = 0x8000                                                        # -0 scale
        qm.scales[1, 1, :] = 0x0001                                                        # f16 subnormal
        qm.scales[1, 2, :] = 0xC2F7                                                        # negative
        qm.data[1, 3, :] = 0x08                                                            # codes 8 and 0: 0 and -8
    elif fmt in (FMT_INT4_G64, FMT_INT8_G64):
        qm.scales[1, 0, :] = 0x8000                                                        # -0 scale
        qm.scales[1, 1, :] = 0x0001                                                        # bf16 subnormal
        qm.scales[1, 2, :] = 0xC2F7                                                        # negative
    else:
        qm.scales[1, 0, :] = 0.0
        qm.data[1, 5, :] = 0x7F                                                            # NaN codes
    dev = qweight_to_device(qm)
    for e in (0, 1, 2):
        out = torch.empty((N, K), dtype=torch.float32, device="cuda")
        B.moe_dequantize(fmt, dev, N, K, e, 0, N, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        ref = F.decode(fmt, qm.data[e], qm.scales[e], float(qm.ts[e]), N, K).astype(np.float32)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(_f32_bits(got)[~nan], _f32_bits(ref)[~nan]), f"expert {e}"


def test_dequantize_row_window():
    qm = synth.make_stack(FMT_NVFP4, 12, synth.KIND_ROUTED, 0, 0, 2, 512, 2048)
    dev = qweight_to_device(qm)
    out = torch.empty((48, 2048), dtype=torch.float32, device="cuda")
    B.moe_dequantize(FMT_NVFP4, dev, 512, 2048, 1, 400, 48, out)
    ref = F.decode(FMT_NVFP4, qm.data[1], qm.scales[1], float(qm.ts[1]), 512, 2048)[400:448].astype(np.float32)
    assert np.array_equal(_f32_bits(out.cpu().numpy()), _f32_bits(ref))


def test_quantize_act_nvfp4_bit_exact():
    rng = np.random.default_rng(21)
    rows, K = 37, 512
    a = rng.standard_normal((rows, K)) * np.exp(rng.uniform(-6, 6, (rows, 1)))
    a[0, :16] = 0.0                                  # zero block -> zero scale and codes
    a[1, :16] = 1e-30                                # scale underflows to zero
    a[2, :16] = 5000.0                               # amax / 6 above 448: saturated scale
    a[3, 16:32] = -0.0
    bits = F.f64_to_bf16_bits(a)
    x = G.x_device(bits)
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    sc = torch.empty((rows, K // 16), dtype=torch.uint8, device="cuda")
    B.moe_quantize_act_nvfp4(x, rows, K, codes, sc)
    torch.cuda.synchronize()
    q_ref, s_ref = M.nvfp4_quantize_act(F.bf16_to_f64(bits))
    packed = (q_ref[:, 0::2] | (q_ref[:, 1::2] << 4)).astype(np.uint8)
    np.testing.assert_array_equal(sc.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(codes.cpu().numpy(), packed)


def test_quantize_act_mxfp4_bit_exact():
    rng = np.random.default_rng(22)
    rows, K = 37, 512
    a = rng.standard_normal((rows, K)) * np.exp(rng.uniform(-30, 30, (rows, 1)))
    a[0, :32] = 0.0                                  # zero block -> scale code 127, zero codes
    a[1, :32] = np.linspace(-6.0, 6.0, 32) * 2.0 ** -4    # amax exactly 6 * 2^-4: exponent -4
    a[2, :32] = a[1, :32] * (1 + 2.0 ** -7)          # just above: exponent -3
    a[3, 32:64] = -0.0
    a[4, :32] = 1e-40                                # below FP32's normal range
    bits = F.f64_to_bf16_bits(a)
    x = G.x_device(bits)
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    sc = torch.empty((rows, K // 32), dtype=torch.uint8, device="cuda")
    B.moe_quantize_act_mxfp4(x, rows, K, codes, sc)
    torch.cuda.synchronize()
    q_ref, s_ref = M.mxfp4_quantize_act(F.bf16_to_f64(bits))
    packed = (q_ref[:, 0::2] | (q_ref[:, 1::2] << 4)).astype(np.uint8)
    np.testing.assert_array_equal(sc.cpu().numpy(), s_ref)
    np.testing.assert_array_equal(codes.cpu().numpy(), packed)


# ------------------------------------------------------------------ routing ----

DECODE_CASES = [("tiny_nvfp4", 1), ("decode_nvfp4", 1), ("decode_nvfp4", 4), ("decode_nvfp4", 8),
                ("decode_mxfp4", 1), ("decode_mxfp4", 8), ("decode_int4", 8)]


@pytest.mark.parametrize("name,T", DECODE_CASES)
def test_route_matches_oracle(name, T):
    hl = G.host_layer(name)
    dl = G.device_layer(name)
    x = synth.make_tokens(hl.cfg, T, seed=0, batch=T)
    got = G.route(dl, x)
    l32, near, idx, w = M.route(x, hl.router_w, hl.router_b, hl.cfg.k)
    cnt, off, pair = M.dispatch(idx, hl.cfg.E)
    ref = {"logits": l32, "topk_idx": idx, "topk_w": w, "expert_cnt": cnt, "expert_off": off, "pair_list": pair}
    G.assert_routing_matches(got, ref, near)


def test_route_ties_break_to_lower_id():
    # identical router rows -> identical logits; the tie rule picks ascending ids
    cfg = LayerConfig("ties", FMT_NVFP4, H=256, E=16, k=4, I=128)
    hl = synth.make_layer(cfg, seed=3)
    hl.router_w[5] = hl.router_w[2]
    hl.router_w[9] = hl.router_w[2]
    hl.router_w[2] *= 4.0
    hl.router_w[5] *= 4.0
    hl.router_w[9] *= 4.0
    dl = to_device(hl)
    x = synth.make_tokens(cfg, 6, seed=3)
    got = G.route(dl, x)
    l32, near, idx, w = M.route(x, hl.router_w, None, cfg.k)
    cnt, off, pair = M.dispatch(idx, cfg.E)
    G.assert_routing_matches(got, {"logits": l32, "topk_idx": idx, "topk_w": w, "expert_cnt": cnt,
                                   "expert_off": off, "pair_list": pair}, near)


# -------------------------------------------------------------------- layer ----

def _check_y(y_bits, ref_bits, tokens=None):
    y = F.bf16_to_f64(y_bits if tokens is None else y_bits[tokens])
    r = F.bf16_to_f64(ref_bits)
    ok = M.within_tolerance(y, r)
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        raise AssertionError(f"{int((~ok).sum())} of {ok.size} outputs outside tolerance; e.g. "
                             + ", ".join(f"{tuple(b)}: {y[tuple(b)]} vs {r[tuple(b)]}" for b in bad))


@pytest.mark.parametrize("name,T", DECODE_CASES)
def test_decode_matches_oracle(name, T):
    # every token of the batch, seed 0, on the full layer
    hl = G.host_layer(name)
    dl = G.device_layer(name)
    x = synth.make_tokens(hl.cfg, T, seed=0, batch=T)
    y, routing = G.decode(dl, x)
    ref = M.layer_forward(hl, x)
    _check_y(y, ref["y_bits"])
    G.assert_routing_matches(routing, ref, ref["near_midpoint"])


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("name,T", [c for c in DECODE_CASES if c[0] != "tiny_nvfp4"])
def test_decode_matches_oracle_more_seeds(name, T, seed):
    # seeds 1-3: every token, on the seed's layer with only the selected experts generated
    cfg = synth.CONFIGS[name]
    x = synth.make_tokens(cfg, T, seed=seed, batch=T)
    hl = G.sparse_host_layer(name, seed, x)
    dl = to_device(hl)
    y, routing = G.decode(dl, x)
    ref = M.layer_forward(hl, x)
    _check_y(y, ref["y_bits"])
    G.assert_routing_matches(routing, ref, ref["near_midpoint"])
    del dl
    torch.cuda.empty_cache()


def _spread_scales(qm, fmt, rows_every=3):
    """Push one scale block per 128-column unit of every third row far below the others of its
    row group: 2^-24 for MXFP4 (limit 2^-20), 2^-26 for int4 g64 (limit 2^-24).  The decode
    kernels' scale fold is not exact there, so those units take the exact 4-MMA path."""
    qm = synth.QMat(qm.fmt, qm.N, qm.K, qm.data.copy(), qm.scales.copy(), qm.ts.copy())
    rows = np.arange(0, qm.N, rows_every)
    if fmt == FMT_MXFP4:
        blk = np.arange(0, qm.K // 32, 4)                            # lane 0's block of each unit
        sub = qm.scales[:, rows[:, None], blk[None, :]].astype(np.int32)
        qm.scales[:, rows[:, None], blk[None, :]] = np.maximum(sub - 24, 1).astype(np.uint8)
    else:
        grp = np.arange(0, qm.K // 64, 2)                            # lanes 0-1's group of each unit
        s = qm.scales[:, rows[:, None], grp[None, :]].astype(np.int32)
        ex = (s >> 7) & 0xFF
        ex = np.where(ex > 27, ex - 26, ex)
        qm.scales[:, rows[:, None], grp[None, :]] = ((s & 0x807F) | (ex << 7)).astype(np.uint16)
    return qm


@pytest.mark.parametrize("fmt", [FMT_MXFP4, FMT_INT4_G64])
@pytest.mark.parametrize("T", [1, 8])
def test_decode_exact_path_for_wide_scale_spreads(fmt, T):
    cfg = LayerConfig(f"spread_{fmt}", fmt, H=1024, E=12, k=4, I=512,
                      shared_fmt=fmt, shared_I=256)
    hl = synth.make_layer(cfg, seed=6)
    for attr in ("gate", "up", "down", "shared_gate", "shared_up", "shared_down"):
        setattr(hl, attr, _spread_scales(getattr(hl, attr), fmt))
    dl = to_device(hl)
    x = synth.make_tokens(cfg, T, seed=6, batch=T)
    y, routing = G.decode(dl, x)
    ref = M.layer_forward(hl, x)
    _check_y(y, ref["y_bits"])
    G.assert_routing_matches(routing, ref, ref["near_midpoint"])
    # the spread blocks are tiny but not zero: the decoded weights keep them bit for bit
    out = torch.empty((16, cfg.H), dtype=torch.float32, device="cuda")
    B.moe_dequantize(fmt, dl.gate, cfg.I, cfg.H, 1, 0, 16, out)
    torch.cuda.synchronize()
    ref_w = F.decode(fmt, hl.gate.data[1], hl.gate.scales[1], 1.0, cfg.I, cfg.H)[:16].astype(np.float32)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref_w.view(np.uint32))


SMALL = [
    LayerConfig("s_nvfp4_fp8", FMT_NVFP4, H=512, E=24, k=5, I=256, shared_fmt=FMT_FP8_B128, shared_I=384),
    LayerConfig("s_mxfp4", FMT_MXFP4, H=640, E=12, k=3, I=384),
    LayerConfig("s_int4_int8", FMT_INT4_G64, H=768, E=16, k=4, I=256, shared_fmt=FMT_INT8_G64, shared_I=512),
    LayerConfig("s_int8", FMT_INT8_G64, H=512, E=9, k=2, I=128, shared_fmt=FMT_NVFP4, shared_I=256),
    LayerConfig("s_fp8", FMT_FP8_B128, H=384, E=6, k=6, I=256, shared_fmt=FMT_MXFP4, shared_I=128),
    LayerConfig("s_nvfp4_k1", FMT_NVFP4, H=256, E=3, k=1, I=128),
    LayerConfig("s_g128_int8", FMT_INT4_G128, H=768, E=10, k=3, I=256, shared_fmt=FMT_INT8_G64, shared_I=256),
    LayerConfig("s_nvfp4_g128", FMT_NVFP4, H=512, E=8, k=2, I=128, shared_fmt=FMT_INT4_G128, shared_I=384),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c.name for c in SMALL])
@pytest.mark.parametrize("T", [1, 3, 8])
def test_decode_small_shapes(cfg, T):
    hl = synth.make_layer(cfg, seed=5)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, T, seed=5, batch=T)
    y, routing = G.decode(dl, x)
    ref = M.layer_forward(hl, x)
    _check_y(y, ref["y_bits"])
    G.assert_routing_matches(routing, ref, ref["near_midpoint"])


def test_decode_deterministic_and_batch_invariant():
    hl = G.host_layer("decode_nvfp4")
    dl = G.device_layer("decode_nvfp4")
    x = synth.make_tokens(hl.cfg, 8, seed=9, batch=99)
    y1, _ = G.decode(dl, x)
    y2, _ = G.decode(dl, x)
    assert np.array_equal(y1, y2)
    for t in (0, 5):
        y_one, _ = G.decode(dl, x[t:t + 1])
        assert np.array_equal(y_one[0], y1[t])


def test_workspace_reuse_across_calls_and_sizes():
    hl = G.host_layer("tiny_nvfp4")
    dl = G.device_layer("tiny_nvfp4")
    ws = G.new_ws(dl, 8)
    for T in (8, 1, 5, 8):
        x = synth.make_tokens(hl.cfg, T, seed=1, batch=T)
        y, _ = G.decode(dl, x, ws=ws)
        _check_y(y, M.layer_forward(hl, x)["y_bits"])
