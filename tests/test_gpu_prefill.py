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
from synth.configs import FMT_MXFP4, FMT_NVFP4, LayerConfig
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


def test_prefill_unsupported_format_is_reported():
    cfg = LayerConfig("p_mx", FMT_MXFP4, H=256, E=4, k=2, I=128)
    dl = to_device(synth.make_layer(cfg, seed=1))
    x = G.x_device(synth.make_tokens(cfg, 20, seed=1))
    y = torch.zeros((20, cfg.H), dtype=torch.int16, device="cuda")
    ws = G.new_ws(dl, 20)
    st = B.moe_prefill_forward(dl, x, 20, y, ws, raise_on_error=False)
    assert st == B.MOE_ERR_UNSUPPORTED


# ------------------------------------------------------------ W4A4 lever ----

W4A4 = [
    LayerConfig("w4_small", FMT_NVFP4, H=512, E=6, k=2, I=256),
    LayerConfig("w4_skew", FMT_NVFP4, H=768, E=20, k=4, I=512, zipf_s=1.1),
]


def _check_w4a4(y_bits, ref_bits, tokens=None):
    """W4A4 against the oracle's act_quant mode.  x is quantised identically on
    both sides (same rule, same BF16 input); h is re-quantised from a BF16 value
    that the GPU reaches with FP32 accumulation, so a rare h can land on the
    other side of a BF16 or E2M1 rounding boundary.  Bar: every element within
    max(2 BF16 ulp, 1e-3) except at most 0.1 %, and those within 2^-5 relative."""
    y = F.bf16_to_f64(y_bits if tokens is None else y_bits[tokens])
    r = F.bf16_to_f64(ref_bits)
    ok = M.within_tolerance(y, r)
    assert np.isfinite(y).all()
    frac_bad = float((~ok).mean())
    assert frac_bad <= 1e-3, f"{int((~ok).sum())} of {ok.size} outputs outside the 2-ulp bar"
    loose = np.abs(y - r) <= np.maximum(2.0 ** -5 * np.abs(r), 1e-2)
    assert loose.all(), f"{int((~loose).sum())} outputs outside the loose bar"


@pytest.mark.parametrize("cfg", W4A4, ids=[c.name for c in W4A4])
@pytest.mark.parametrize("T", [1, 37, 300])
def test_prefill_w4a4_matches_oracle(cfg, T):
    hl = synth.make_layer(cfg, seed=9)
    dl = to_device(hl)
    x = synth.make_tokens(cfg, T, seed=9, batch=T)
    y, routing = G.decode(dl, x, prefill=True, act_quant=1)
    ref = M.layer_forward(hl, x, act_quant=True)
    _check_w4a4(y, ref["y_bits"])
    assert_prefill_routing(routing, ref, ref["near_midpoint"])


def test_prefill_w4a4_workload_sampled():
    hl = G.host_layer("prefill_nvfp4")
    dl = G.device_layer("prefill_nvfp4")
    T, tokens = 4096, [0, 5, 2047, 4095]
    x = synth.make_tokens(hl.cfg, T, seed=0, batch=T)
    y, _ = G.decode(dl, x, prefill=True, act_quant=1)
    ref = M.layer_forward(hl, x, act_quant=True, tokens=tokens)
    _check_w4a4(y, ref["y_bits"], tokens)


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
