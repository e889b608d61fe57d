"""Helpers shared by the GPU tests: build once, cache synthetic layers, run the
C ABI on device buffers and bring results back as numpy arrays."""
from __future__ import annotations

import functools

import numpy as np
import torch

import synth
from quantized_moe_decode_router_gb300 import _binding as B
from quantized_moe_decode_router_gb300 import build as qbuild
from quantized_moe_decode_router_gb300.device import to_device


@functools.lru_cache(maxsize=1)
def lib():
    qbuild.build()
    return B.load()


@functools.lru_cache(maxsize=6)
def host_layer(name: str, seed: int = 0):
    return synth.make_layer(synth.CONFIGS[name], seed)


_dev_cache = {}


def device_layer(name: str, seed: int = 0):
    key = (name, seed)
    if key not in _dev_cache:
        if len(_dev_cache) >= 2:
            _dev_cache.clear()
            torch.cuda.empty_cache()
        _dev_cache[key] = to_device(host_layer(name, seed))
    return _dev_cache[key]


def sparse_host_layer(name: str, seed: int, x_bits: np.ndarray):
    """The layer of workload `name` at `seed` with only the routed experts these tokens
    select filled in (the others all-zero codes and scales): the router, the shared
    expert and every selected expert are the seed's own, so the outputs for these
    tokens equal those of the full layer, at a fraction of the generation cost."""
    import concurrent.futures as cf
    from oracle import moe as M
    cfg = synth.CONFIGS[name]
    rw = synth.normal_f32(synth.stream_key(seed, synth.KIND_ROUTER, 0, 0), cfg.E * cfg.H,
                          synth.configs.WEIGHT_SIGMA).reshape(cfg.E, cfg.H)
    rb = synth.zipf_bias(cfg, seed) if cfg.zipf_s else None
    _, _, idx, _ = M.route(x_bits, rw, rb, cfg.k)
    touched = sorted(set(int(e) for e in idx.reshape(-1)))

    def empty(N, K):
        sshape, sdt = synth.scale_shape(cfg.fmt, N, K)
        return synth.QMat(cfg.fmt, N, K, np.zeros((cfg.E,) + synth.data_shape(cfg.fmt, N, K), np.uint8),
                          np.zeros((cfg.E,) + sshape, sdt), np.ones(cfg.E, np.float32))
    gate, up, down = empty(cfg.I, cfg.H), empty(cfg.I, cfg.H), empty(cfg.H, cfg.I)
    with cf.ThreadPoolExecutor(max_workers=16) as ex:
        for e, mats in zip(touched, ex.map(lambda e: synth.make_expert(cfg, seed, e), touched)):
            for dst, src in zip((gate, up, down), mats):
                dst.data[e], dst.scales[e], dst.ts[e] = src.data[0], src.scales[0], src.ts[0]
    full = synth.make_layer(cfg.with_(E=1, k=1), seed) if cfg.shared_fmt else None
    return synth.HostLayer(cfg, seed, rw, rb, gate, up, down,
                           full.shared_gate if full else None, full.shared_up if full else None,
                           full.shared_down if full else None)


def x_device(x_bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()


def new_ws(layer, T: int, act_quant: int = 0) -> torch.Tensor:
    n = B.workspace_size(layer, T, act_quant)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    B.workspace_init(ws)
    return ws


def ws_read(ws: torch.Tensor, off: int, dtype, count: int) -> np.ndarray:
    nbytes = np.dtype(dtype).itemsize * count
    return ws[off:off + nbytes].cpu().numpy().view(dtype).copy()


def decode(layer, x_bits: np.ndarray, ws=None, prefill: bool = False, act_quant: int = 0, fold_scales: int = 0,
           fp8_act: int = 0):
    """Run one forward call; returns (y bits uint16 [T, H], routing dict read from the workspace)."""
    T, H = x_bits.shape
    if ws is None:
        ws = new_ws(layer, T, act_quant)
    x = x_device(x_bits)
    y = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    if prefill:
        B.moe_prefill_forward(layer, x, T, y, ws, act_quant=act_quant, fold_scales=fold_scales, fp8_act=fp8_act)
    else:
        B.moe_decode_forward(layer, x, T, y, ws, act_quant=act_quant)
    torch.cuda.synchronize()
    assert B.moe_check(ws) == 0
    maxT = _ws_tokens(layer, ws)
    lo = B.workspace_layout(layer, maxT, act_quant)
    E, k = layer.n_experts, layer.top_k
    routing = {
        "logits": ws_read(ws, lo.logits, np.float32, T * E).reshape(T, E),
        "topk_idx": ws_read(ws, lo.topk_idx, np.int32, T * k).reshape(T, k),
        "topk_w": ws_read(ws, lo.topk_w, np.float32, T * k).reshape(T, k),
        "expert_cnt": ws_read(ws, lo.expert_cnt, np.int32, E),
        "expert_off": ws_read(ws, lo.expert_off, np.int32, E + 1),
        "pair_list": ws_read(ws, lo.pair_list, np.int32, T * k),
    }
    if act_quant:
        I = layer.inter
        routing["h_codes"] = ws_read(ws, lo.h_codes, np.uint8, T * k * I // 2).reshape(T * k, I // 2)
        blk = 32 if act_quant == 2 else 16   # MXFP4 / NVFP4 block scales of h
        routing["h_scales"] = ws_read(ws, lo.h_scales, np.uint8, T * k * I // blk).reshape(T * k, I // blk)
    return y.cpu().numpy().view(np.uint16), routing


def _ws_tokens(layer, ws) -> int:
    n = ws.numel()
    lo, hi = 1, 1
    while B.workspace_size(layer, hi * 2) <= n and hi < (1 << 22):
        hi *= 2
    lo = hi
    hi = hi * 2
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if B.workspace_size(layer, mid) <= n:
            lo = mid
        else:
            hi = mid
    return lo


def route(layer, x_bits: np.ndarray):
    T = x_bits.shape[0]
    E, k = layer.n_experts, layer.top_k
    ws = new_ws(layer, T)
    x = x_device(x_bits)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    cnt = torch.empty(E, dtype=torch.int32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pair = torch.empty(T * k, dtype=torch.int32, device="cuda")
    B.moe_route(layer, x, T, idx, w, cnt, off, pair, ws)
    torch.cuda.synchronize()
    lo = B.workspace_layout(layer, T)
    logits = ws_read(ws, lo.logits, np.float32, T * E).reshape(T, E)
    return {"logits": logits, "topk_idx": idx.cpu().numpy(), "topk_w": w.cpu().numpy(),
            "expert_cnt": cnt.cpu().numpy(), "expert_off": off.cpu().numpy(), "pair_list": pair.cpu().numpy()}


def assert_routing_matches(got: dict, ref: dict, near: np.ndarray):
    """Bit-exact indices and dispatch.  The router recomputes exactly every expert that
    can still reach the top-k (the others hold -inf in the workspace's logits): those
    logits are the correctly rounded value, except oracle-flagged near-midpoint ones, and
    every selected expert is among them.  At decode sizes (a few thousand logits, about
    2^-15 flagged per logit) none may be flagged, so every recomputed logit is compared
    bit for bit."""
    lg, lr = got["logits"], ref["logits"]
    if lg.size <= 8 * 1024:
        assert not near.any(), f"{int(near.sum())} logits within 2^-40 of an FP32 midpoint at this seed"
    recomputed = ~np.isneginf(lg)
    diff = (lg.view(np.uint32) != lr.view(np.uint32)) & recomputed
    assert not np.any(diff & ~near), f"{int(np.sum(diff & ~near))} recomputed logits differ from the correctly rounded value"
    T, k = ref["topk_idx"].shape
    assert np.all(recomputed[np.arange(T)[:, None], ref["topk_idx"]]), "a selected expert was not recomputed"
    np.testing.assert_array_equal(got["topk_idx"], ref["topk_idx"])
    np.testing.assert_array_equal(got["expert_cnt"], ref["expert_cnt"])
    np.testing.assert_array_equal(got["expert_off"], ref["expert_off"])
    np.testing.assert_array_equal(got["pair_list"], ref["pair_list"])
    np.testing.assert_allclose(got["topk_w"], ref["topk_w"], rtol=8 * 2.0 ** -24, atol=2.0 ** -30)
