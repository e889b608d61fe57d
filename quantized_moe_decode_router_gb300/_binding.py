"""ctypes binding of libqmoe.so (include/moe.h): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels.  PyTorch is used
only to own device memory and to supply the current CUDA stream; there is no
fallback: if the library is missing or fails to load, importing raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_MISALIGNED = -3
MOE_ERR_WORKSPACE = -4
MOE_ERR_CUDA = -5
MOE_ERR_DEVICE_TIMEOUT = -6
MOE_ERR_DEVICE_BAD_INDEX = -7

MOE_FMT_NONE, MOE_FMT_NVFP4, MOE_FMT_MXFP4, MOE_FMT_INT4_G64, MOE_FMT_INT8_G64, MOE_FMT_FP8_B128, MOE_FMT_INT4_G128 = \
    range(7)
MOE_DECODE_MAX_TOKENS = 8


class moe_qweight(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p)]


class moe_layer(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("n_experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32), ("fmt", ctypes.c_int32),
        ("router_w", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
        ("gate", moe_qweight), ("up", moe_qweight), ("down", moe_qweight),
        ("shared_fmt", ctypes.c_int32), ("shared_inter", ctypes.c_int32),
        ("shared_gate", moe_qweight), ("shared_up", moe_qweight), ("shared_down", moe_qweight),
        ("shared_expert_gate", ctypes.c_void_p), ("bias_select", ctypes.c_int32),
    ]


class moe_options(ctypes.Structure):
    _fields_ = [("act_quant", ctypes.c_int32), ("bf16_partials", ctypes.c_int32), ("wait_limit_us", ctypes.c_int32),
                ("fold_scales", ctypes.c_int32), ("fp8_act", ctypes.c_int32), ("reserved", ctypes.c_int32 * 3)]


class moe_ws_layout(ctypes.Structure):
    _fields_ = [("logits", ctypes.c_size_t), ("topk_idx", ctypes.c_size_t), ("topk_w", ctypes.c_size_t),
                ("expert_cnt", ctypes.c_size_t), ("expert_off", ctypes.c_size_t), ("pair_list", ctypes.c_size_t),
                ("total", ctypes.c_size_t), ("h_codes", ctypes.c_size_t), ("h_scales", ctypes.c_size_t)]


class moe_decode_plan_info(ctypes.Structure):
    _fields_ = [("gu_slices", ctypes.c_int32), ("gu_slices_shared", ctypes.c_int32),
                ("gu_slices_tail", ctypes.c_int32), ("gu_tail_cap", ctypes.c_int32),
                ("dn_slices", ctypes.c_int32), ("dn_segs", ctypes.c_int32), ("gu_ctas_per_sm", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("gu_smem", ctypes.c_size_t), ("dn_smem", ctypes.c_size_t),
                ("gu_split_blocks", ctypes.c_size_t), ("dn_split_blocks", ctypes.c_size_t),
                ("split_block_capacity", ctypes.c_size_t)]


# (name, restype, argtypes) of every entry point declared in include/moe.h
_P = ctypes.POINTER
_SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int32]),
    "moe_workspace_size": (ctypes.c_size_t, [_P(moe_layer), ctypes.c_int32, _P(moe_options)]),
    "moe_workspace_init": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_route": (ctypes.c_int32, [_P(moe_layer), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_decode_forward": (ctypes.c_int32, [_P(moe_layer), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                            _P(moe_options), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_prefill_forward": (ctypes.c_int32, [_P(moe_layer), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                             _P(moe_options), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_decode_forward_timed": (ctypes.c_int32, [_P(moe_layer), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                  _P(moe_options), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                                  ctypes.POINTER(ctypes.c_void_p)]),
    "moe_prefill_forward_timed": (ctypes.c_int32, [_P(moe_layer), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                   _P(moe_options), ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                                   ctypes.POINTER(ctypes.c_void_p)]),
    "moe_experts_forward": (ctypes.c_int32, [_P(moe_layer), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p, _P(moe_options), ctypes.c_void_p,
                                             ctypes.c_size_t, ctypes.c_void_p]),
    "moe_decode_forward_noalloc": (ctypes.c_int32, [_P(moe_layer), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                                    _P(moe_options), ctypes.c_void_p]),
    "moe_check": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_decode_plan": (ctypes.c_int32, [_P(moe_layer), ctypes.c_int32, ctypes.c_int32, _P(moe_decode_plan_info)]),
    "moe_workspace_layout": (ctypes.c_int32, [_P(moe_layer), ctypes.c_int32, _P(moe_options), _P(moe_ws_layout)]),
    "moe_dequantize": (ctypes.c_int32, [ctypes.c_int32, _P(moe_qweight), ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                        ctypes.c_void_p]),
    "moe_quantize_act_nvfp4": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_void_p]),
    "moe_quantize_act_mxfp4": (ctypes.c_int32, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_void_p]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load libqmoe.so (raises OSError if it is missing: build it with build.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise OSError(f"{path} not found; run quantized_moe_decode_router_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = load().moe_status_string(status).decode()
        super().__init__(f"{what}: {msg}" if what else msg)


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)
    return status


def status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


@dataclass
class QWeight:
    data: object          # torch uint8 tensor (device)
    scales: object        # torch tensor (device)
    tensor_scale: object = None   # torch float32 [count] (NVFP4)

    def c(self) -> moe_qweight:
        return moe_qweight(_ptr(self.data), _ptr(self.scales), _ptr(self.tensor_scale))


@dataclass
class Layer:
    """Device-resident layer description; tensors must stay alive while in use."""
    hidden: int
    inter: int
    n_experts: int
    top_k: int
    fmt: int
    router_w: object
    router_bias: object
    gate: QWeight
    up: QWeight
    down: QWeight
    shared_fmt: int = 0
    shared_inter: int = 0
    shared_gate: Optional[QWeight] = None
    shared_up: Optional[QWeight] = None
    shared_down: Optional[QWeight] = None
    shared_expert_gate: object = None   # torch float32 [H] (device) or None
    bias_select: int = 0                # 1: the router bias steers the selection only

    def c(self) -> moe_layer:
        z = moe_qweight(None, None, None)
        return moe_layer(self.hidden, self.inter, self.n_experts, self.top_k, self.fmt, _ptr(self.router_w),
                         _ptr(self.router_bias), self.gate.c(), self.up.c(), self.down.c(), self.shared_fmt,
                         self.shared_inter, self.shared_gate.c() if self.shared_gate else z,
                         self.shared_up.c() if self.shared_up else z,
                         self.shared_down.c() if self.shared_down else z, _ptr(self.shared_expert_gate),
                         self.bias_select)


def _opts(act_quant: int = 0, bf16_partials: int = 0, wait_limit_us: int = 0, fold_scales: int = 0,
          fp8_act: int = 0):
    return moe_options(act_quant, bf16_partials, wait_limit_us, fold_scales, fp8_act, (ctypes.c_int32 * 3)())


def workspace_size(layer: Layer, max_tokens: int, act_quant: int = 0) -> int:
    lc, o = layer.c(), _opts(act_quant)
    return int(load().moe_workspace_size(ctypes.byref(lc), max_tokens, ctypes.byref(o)))


def workspace_layout(layer: Layer, max_tokens: int, act_quant: int = 0) -> moe_ws_layout:
    lc, o, out = layer.c(), _opts(act_quant), moe_ws_layout()
    _check(load().moe_workspace_layout(ctypes.byref(lc), max_tokens, ctypes.byref(o), ctypes.byref(out)),
           "moe_workspace_layout")
    return out


def decode_plan(layer: Layer, T: int, num_sms: int) -> moe_decode_plan_info:
    """Launch plan of a decode call (K splits, staged shared memory); host only."""
    lc, out = layer.c(), moe_decode_plan_info()
    _check(load().moe_decode_plan(ctypes.byref(lc), T, num_sms, ctypes.byref(out)), "moe_decode_plan")
    return out


def workspace_init(ws, stream=None):
    return _check(load().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream_handle(stream)),
                  "moe_workspace_init")


def moe_route(layer: Layer, x, T: int, topk_idx=None, topk_w=None, expert_cnt=None, expert_off=None,
              pair_list=None, ws=None, stream=None, raise_on_error: bool = True) -> int:
    lc = layer.c()
    st = load().moe_route(ctypes.byref(lc), _ptr(x), T, _ptr(topk_idx), _ptr(topk_w), _ptr(expert_cnt),
                          _ptr(expert_off), _ptr(pair_list), _ptr(ws),
                          0 if ws is None else ws.numel() * ws.element_size(), _stream_handle(stream))
    return _check(st, "moe_route") if raise_on_error else st


def moe_decode_forward(layer: Layer, x, T: int, y, ws, stream=None, act_quant: int = 0,
                       raise_on_error: bool = True, bf16_partials: int = 0, fold_scales: int = 0,
                       fp8_act: int = 0) -> int:
    lc, o = layer.c(), _opts(act_quant, bf16_partials, 0, fold_scales, fp8_act)
    st = load().moe_decode_forward(ctypes.byref(lc), _ptr(x), T, _ptr(y), ctypes.byref(o), _ptr(ws),
                                   0 if ws is None else ws.numel() * ws.element_size(), _stream_handle(stream))
    return _check(st, "moe_decode_forward") if raise_on_error else st


def moe_experts_forward(layer: Layer, x, T: int, topk_idx, topk_w, y, ws, stream=None, raise_on_error: bool = True,
                        bf16_partials: int = 0) -> int:
    """The expert half of the decode forward on caller routing (topk_idx i32 [T, k], topk_w f32 [T, k])."""
    lc, o = layer.c(), _opts(0, bf16_partials)
    st = load().moe_experts_forward(ctypes.byref(lc), _ptr(x), T, _ptr(topk_idx), _ptr(topk_w), _ptr(y),
                                    ctypes.byref(o), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                    _stream_handle(stream))
    return _check(st, "moe_experts_forward") if raise_on_error else st


def moe_decode_forward_timed(layer: Layer, x, T: int, y, ws, events, stream=None, bf16_partials: int = 0) -> int:
    """moe_decode_forward recording torch.cuda.Event objects (4, or None entries) between its kernels."""
    lc, o = layer.c(), _opts(0, bf16_partials)
    arr = (ctypes.c_void_p * 4)(*[None if e is None else int(e.cuda_event) for e in events])
    st = load().moe_decode_forward_timed(ctypes.byref(lc), _ptr(x), T, _ptr(y), ctypes.byref(o), _ptr(ws),
                                         ws.numel() * ws.element_size(), _stream_handle(stream), arr)
    return _check(st, "moe_decode_forward_timed")


def moe_decode_forward_noalloc(layer: Layer, x, T: int, y, stream=None, raise_on_error: bool = True) -> int:
    """moe_decode_forward on the library's fixed device workspace (no caller workspace, no allocation)."""
    lc, o = layer.c(), _opts(0)
    st = load().moe_decode_forward_noalloc(ctypes.byref(lc), _ptr(x), T, _ptr(y), ctypes.byref(o),
                                           _stream_handle(stream))
    return _check(st, "moe_decode_forward_noalloc") if raise_on_error else st


def moe_prefill_forward(layer: Layer, x, T: int, y, ws, stream=None, act_quant: int = 0,
                        raise_on_error: bool = True, bf16_partials: int = 0, wait_limit_us: int = 0,
                        fold_scales: int = 0, fp8_act: int = 0) -> int:
    lc, o = layer.c(), _opts(act_quant, bf16_partials, wait_limit_us, fold_scales, fp8_act)
    st = load().moe_prefill_forward(ctypes.byref(lc), _ptr(x), T, _ptr(y), ctypes.byref(o), _ptr(ws),
                                    0 if ws is None else ws.numel() * ws.element_size(), _stream_handle(stream))
    return _check(st, "moe_prefill_forward") if raise_on_error else st


def moe_prefill_forward_timed(layer: Layer, x, T: int, y, ws, events, stream=None, act_quant: int = 0,
                              bf16_partials: int = 0, fold_scales: int = 0, fp8_act: int = 0) -> int:
    """moe_prefill_forward recording torch.cuda.Event objects (8, or None entries) between its kernels."""
    lc, o = layer.c(), _opts(act_quant, bf16_partials, 0, fold_scales, fp8_act)
    arr = (ctypes.c_void_p * 8)(*[None if e is None else int(e.cuda_event) for e in events])
    st = load().moe_prefill_forward_timed(ctypes.byref(lc), _ptr(x), T, _ptr(y), ctypes.byref(o), _ptr(ws),
                                          ws.numel() * ws.element_size(), _stream_handle(stream), arr)
    return _check(st, "moe_prefill_forward_timed")


def moe_check(ws, stream=None) -> int:
    return int(load().moe_check(_ptr(ws), ws.numel() * ws.element_size(), _stream_handle(stream)))


def moe_check_noalloc(stream=None) -> int:
    """moe_check of the allocation-free entry point's fixed array on the current device."""
    return int(load().moe_check(None, 0, _stream_handle(stream)))


def moe_dequantize(fmt: int, w: QWeight, N: int, K: int, expert: int, row0: int, nrows: int, out,
                   stream=None) -> int:
    qc = w.c()
    return _check(load().moe_dequantize(fmt, ctypes.byref(qc), N, K, expert, row0, nrows, _ptr(out),
                                        _stream_handle(stream)), "moe_dequantize")


def moe_quantize_act_nvfp4(x, rows: int, K: int, codes, scales, stream=None) -> int:
    return _check(load().moe_quantize_act_nvfp4(_ptr(x), rows, K, _ptr(codes), _ptr(scales),
                                                _stream_handle(stream)), "moe_quantize_act_nvfp4")


def moe_quantize_act_mxfp4(x, rows: int, K: int, codes, scales, stream=None) -> int:
    return _check(load().moe_quantize_act_mxfp4(_ptr(x), rows, K, _ptr(codes), _ptr(scales),
                                                _stream_handle(stream)), "moe_quantize_act_mxfp4")
