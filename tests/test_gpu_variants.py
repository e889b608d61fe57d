"""GPU parity of the layer variants and levers, and the device-side failure
reports, through the C ABI.

* caller routing (moe_experts_forward): bit for bit moe_decode_forward when fed
  moe_route's own choice; the oracle's layer on an arbitrary routing; an expert
  id out of range reported as MOE_ERR_DEVICE_BAD_INDEX with no fault;
* the router bias steering the selection only (layer.bias_select), decode and
  prefill;
* a sigmoid-gated shared expert (layer.shared_expert_gate);
* the bf16-partials lever, decode and prefill;
* the prefill kernels' bounded waits made to run out (a 1 us limit): the call
  reports MOE_ERR_DEVICE_TIMEOUT through moe_check and the next call is exact.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import formats as F
from oracle import moe as M
from quantized_moe_decode_router_gb300 import _binding as B
from quantized_moe_decode_router_gb300.device import to_device
from synth.configs import FMT_FP8_B128, FMT_INT8_G64, FMT_MXFP4, FMT_NVFP4, LayerConfig
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    G.lib()


def _check_y(y_bits, ref_bits):
    y, r = F.bf16_to_f64(y_bits), F.bf16_to_f64(ref_bits)
    ok = M.within_tolerance(y, r)
    assert ok.all(), f"{int((~ok).sum())} of {ok.size} outputs outside tolerance; max |d| {np.abs(y - r).max()}"


def _experts(dl, x_bits, idx, w, ws=None, **kw):
    T, H = x_bits.shape
    if ws is None:
        ws = G.new_ws(dl, T)
    x = G.x_device(x_bits)
    y = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    ti = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).cuda()
    tw = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32)).cuda()
    B.moe_experts_forward(dl, x, T, ti, tw, y, ws, **kw)
    torch.cuda.synchronize()
    return y.cpu().numpy().view(np.uint16), ws


# ------------------------------------------------------------ caller routing ----

@pytest.mark.parametrize("name,T", [("decode_nvfp4", 1), ("decode_nvfp4", 8), ("decode_mxfp4", 8)])
def test_experts_forward_on_routers_choice_equals_decode_forward(name, T):
    hl = G.host_layer(name)
    dl = G.device_layer(name)
    x = synth.make_tokens(hl.cfg, T, seed=3, batch=T)
    y_ref, routing = G.decode(dl, x)
    y, ws = _experts(dl, x, routing["topk_idx"], routing["topk_w"])
    assert B.moe_check(ws) == 0
    assert np.array_equal(y, y_ref)


def test_experts_forward_on_any_routing_matches_oracle():
    # a routing no softmax router makes: sigmoid scores of random ids, repeated experts across tokens
    cfg = LayerConfig("ext", FMT_NVFP4, H=512, E=16, k=4, I=256, shared_fmt=FMT_FP8_B128, shared_I=256)
    hl = synth.make_layer(cfg, seed=21)
    dl = to_device(hl)
    rng = np.random.default_rng(21)
    T = 7
    idx = np.stack([rng.choice(cfg.E, cfg.k, replace=False) for _ in range(T)]).astype(np.int32)
    idx[3] = idx[1]
    w = (1.0 / (1.0 + np.exp(-rng.standard_normal((T, cfg.k))))).astype(np.float32)
    x = synth.make_tokens(cfg, T, seed=21)
    y, ws = _experts(dl, x, idx, w)
    assert B.moe_check(ws) == 0
    ref = M.layer_forward(hl, x, routing=(idx, w))
    _check_y(y, ref["y_bits"])


def test_experts_forward_reports_an_expert_id_out_of_range():
    cfg = LayerConfig("bad", FMT_NVFP4, H=256, E=8, k=2, I=128)
    hl = synth.make_layer(cfg, seed=22)
    dl = to_device(hl)
    T = 4
    x = synth.make_tokens(cfg, T, seed=22)
    idx = np.array([[0, 1], [2, 8], [3, -1], [4, 5]], dtype=np.int32)     # 8 and -1 are not experts
    w = np.full((T, cfg.k), 0.5, dtype=np.float32)
    _, ws = _experts(dl, x, idx, w)
    assert B.moe_check(ws) == B.MOE_ERR_DEVICE_BAD_INDEX
    assert B.moe_check(ws) == 0                                            # read and cleared
    # the context and the workspace stay usable: a valid routing is exact afterwards
    idx[1, 1], idx[2, 1] = 7, 6
    y, ws = _experts(dl, x, idx, w, ws=ws)
    assert B.moe_check(ws) == 0
    _check_y(y, M.layer_forward(hl, x, routing=(idx, w))["y_bits"])


# ------------------------------------------------------------ router variants ----

def _biased_layer(cfg, seed, bias_select):
    hl = synth.make_layer(cfg, seed=seed)
    hl.router_b = (np.random.default_rng(seed).standard_normal(cfg.E) * 0.7).astype(np.float32)
    hl.extra["bias_select"] = bias_select
    return hl


@pytest.mark.parametrize("T", [1, 8])
def test_decode_bias_steers_selection_only(T):
    cfg = LayerConfig("bsel", FMT_NVFP4, H=1024, E=64, k=6, I=256)
    hl = _biased_layer(cfg, 23, 1)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, T, seed=23, batch=T)
    y, routing = G.decode(dl, x)
    ref = M.layer_forward(hl, x, bias_select=True)
    G.assert_routing_matches(routing, ref, ref["near_midpoint"])
    _check_y(y, ref["y_bits"])
    assert not np.allclose(ref["topk_w"], M.layer_forward(hl, x)["topk_w"])   # the mode matters here


@pytest.mark.parametrize("T", [17, 300])
def test_prefill_bias_steers_selection_only(T):
    cfg = LayerConfig("bselp", FMT_NVFP4, H=512, E=32, k=4, I=256)
    hl = _biased_layer(cfg, 24, 1)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, T, seed=24, batch=T)
    y, routing = G.decode(dl, x, prefill=True)
    ref = M.layer_forward(hl, x, bias_select=True)
    np.testing.assert_array_equal(routing["topk_idx"], ref["topk_idx"])
    np.testing.assert_allclose(routing["topk_w"], ref["topk_w"], rtol=8 * 2.0 ** -24, atol=2.0 ** -30)
    _check_y(y, ref["y_bits"])


@pytest.mark.parametrize("shared_fmt", [FMT_FP8_B128, FMT_INT8_G64])
@pytest.mark.parametrize("T", [1, 5])
def test_decode_sigmoid_gated_shared_expert(shared_fmt, T):
    cfg = LayerConfig("sg", FMT_NVFP4, H=512, E=16, k=4, I=256, shared_fmt=shared_fmt, shared_I=256)
    hl = synth.make_layer(cfg, seed=25)
    hl.extra["shared_gate_w"] = (np.random.default_rng(25).standard_normal(cfg.H) * 0.1).astype(np.float32)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, T, seed=25, batch=T)
    y, _ = G.decode(dl, x)
    _check_y(y, M.layer_forward(hl, x)["y_bits"])
    # and through the caller-routing entry point
    ref = M.layer_forward(hl, x)
    y2, ws = _experts(dl, x, ref["topk_idx"], ref["topk_w"])
    assert B.moe_check(ws) == 0
    assert np.array_equal(y2, y)


@pytest.mark.parametrize("shared_fmt", [FMT_FP8_B128, FMT_NVFP4])
def test_prefill_sigmoid_gated_shared_expert(shared_fmt):
    cfg = LayerConfig("psg", FMT_NVFP4, H=512, E=16, k=4, I=256, shared_fmt=shared_fmt, shared_I=256)
    hl = synth.make_layer(cfg, seed=29)
    hl.extra["shared_gate_w"] = (np.random.default_rng(29).standard_normal(cfg.H) * 0.1).astype(np.float32)
    dl = to_device(hl)
    T = 150
    x = synth.make_tokens(cfg, T, seed=29, batch=T)
    y, _ = G.decode(dl, x, prefill=True)
    _check_y(y, M.layer_forward(hl, x)["y_bits"])


# --------------------------------------------------------------- bf16 partials ----

@pytest.mark.parametrize("name,T", [("decode_nvfp4", 8), ("tiny_nvfp4", 1)])
def test_decode_bf16_partials(name, T):
    hl = G.host_layer(name)
    dl = G.device_layer(name)
    x = synth.make_tokens(hl.cfg, T, seed=26, batch=T)
    ws = G.new_ws(dl, T)
    y = torch.zeros((T, hl.cfg.H), dtype=torch.int16, device="cuda")
    B.moe_decode_forward(dl, G.x_device(x), T, y, ws, bf16_partials=1)
    torch.cuda.synchronize()
    assert B.moe_check(ws) == 0
    _check_y(y.cpu().numpy().view(np.uint16), M.layer_forward(hl, x, bf16_partials=True)["y_bits"])


@pytest.mark.parametrize("T,shared_fmt", [(17, 0), (300, 0), (200, FMT_INT8_G64)])
def test_prefill_bf16_partials(T, shared_fmt):
    cfg = LayerConfig("pbf", FMT_NVFP4, H=512, E=24, k=4, I=256, zipf_s=1.1, shared_fmt=shared_fmt,
                      shared_I=256 if shared_fmt else 0)
    hl = synth.make_layer(cfg, seed=27)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, T, seed=27, batch=T)
    ws = G.new_ws(dl, T)
    y = torch.zeros((T, cfg.H), dtype=torch.int16, device="cuda")
    B.moe_prefill_forward(dl, G.x_device(x), T, y, ws, bf16_partials=1)
    torch.cuda.synchronize()
    assert B.moe_check(ws) == 0
    y_bits = y.cpu().numpy().view(np.uint16)
    _check_y(y_bits, M.layer_forward(hl, x, bf16_partials=True)["y_bits"])


# --------------------------------------------------------- bounded device waits ----

@pytest.mark.parametrize("sfmt", [0, FMT_INT8_G64])
def test_prefill_wait_limit_runs_out_and_is_reported(sfmt):
    # a 1 us limit on every pipeline wait of the prefill GEMMs (each try_wait suspends at most that
    # long): the epilogue's wait for a whole tile's MMAs (8 K steps of the NVFP4 routed experts) cannot
    # be met in time, so it gives up; every CTA drains what it issued and returns, and moe_check reports
    # the timeout.  With an int8 g64 shared expert the per-group accumulation's waits run under the same
    # limit in the same call (they may or may not run out; the call must still end and report).
    cfg = LayerConfig("waits", FMT_NVFP4, H=512, E=24, k=4, I=256, shared_fmt=sfmt, shared_I=256 if sfmt else 0)
    hl = synth.make_layer(cfg, seed=28)
    dl = to_device(hl)
    T = 300
    x = synth.make_tokens(cfg, T, seed=28, batch=T)
    ws = G.new_ws(dl, T)
    y = torch.zeros((T, cfg.H), dtype=torch.int16, device="cuda")
    B.moe_prefill_forward(dl, G.x_device(x), T, y, ws, wait_limit_us=1)
    torch.cuda.synchronize()
    assert B.moe_check(ws) == B.MOE_ERR_DEVICE_TIMEOUT
    # the context stays usable: the same call with the default limit is exact
    y2, routing = G.decode(dl, x, ws=ws, prefill=True)
    _check_y(y2, M.layer_forward(hl, x)["y_bits"])
