"""Seeded synthetic inputs for the quantized MoE layer.

A module of its own, shared by the CUDA path's tests and benchmark and by the
oracle's tests: it draws Gaussian weights and activations from a counter-based
generator and encodes the weights into the checkpoint formats the DGPP pages
serve (page 1 README "Serves checkpoints as published"; page 4 forum post 1,
quantisation table: NVFP4 / MXFP4 routed experts, int4 g64 routed with int8
g64 shared experts, FP8 shared experts).  It holds none of the layer's own
arithmetic: no decoding, routing, projection or combine happens here.

The heavy lifting is in ``qmoe_synth.c`` (compiled on first use with the
host C compiler); this file only marshals numpy buffers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from .configs import (CONFIGS, FMT_FP8_B128, FMT_INT4_G64, FMT_INT4_G128, FMT_INT8_G64, FMT_MXFP4, FMT_NVFP4,
                      LayerConfig,
                      KIND_ROUTED, KIND_ROUTER, KIND_SHARED, KIND_TOKENS, KIND_ZIPF, WEIGHT_SIGMA)

__all__ = [
    "CONFIGS", "LayerConfig", "QMat", "HostLayer", "make_layer", "make_tokens", "lib", "quantize",
    "normal_f32", "normal_bf16", "data_shape", "scale_shape", "FMT_NVFP4", "FMT_MXFP4", "FMT_INT4_G64",
    "FMT_INT8_G64", "FMT_FP8_B128", "FMT_INT4_G128", "make_expert", "stream_key",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmoe_synth.c")
_LIB = os.path.join(_HERE, "libqmoe_synth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the generator library in place (gcc, -O2, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
               "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            u64, u32, i32, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p
            L.qs_stream_key.restype = u64
            L.qs_stream_key.argtypes = [u64, u32, u32, u32]
            L.qs_draw_u64.restype = u64
            L.qs_draw_u64.argtypes = [u64, u64]
            L.qs_normal_f32.argtypes = [u64, u64, u64, ctypes.c_double, vp]
            L.qs_normal_bf16.argtypes = [u64, u64, u64, ctypes.c_double, vp]
            L.qs_quantize.restype = i32
            L.qs_quantize.argtypes = [i32, vp, i32, i32, vp, vp, vp]
            L.qs_make_stack.restype = i32
            L.qs_make_stack.argtypes = [i32, u64, u32, u32, u32, i32, i32, i32, ctypes.c_double, vp, vp, vp, i32]
            L.qs_permutation.argtypes = [u64, i32, vp]
            L.qs_num_threads.restype = i32
            _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def stream_key(seed: int, kind: int, expert: int, proj: int) -> int:
    return int(lib().qs_stream_key(seed, kind, expert, proj))


def normal_f32(key: int, n: int, sigma: float, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().qs_normal_f32(key, start, n, sigma, _ptr(out))
    return out


def normal_bf16(key: int, n: int, sigma: float, start: int = 0) -> np.ndarray:
    """N(0, sigma) rounded to bf16; returned as raw uint16 bit patterns."""
    out = np.empty(n, dtype=np.uint16)
    lib().qs_normal_bf16(key, start, n, sigma, _ptr(out))
    return out


def data_shape(fmt: int, N: int, K: int) -> tuple:
    if fmt in (FMT_NVFP4, FMT_MXFP4, FMT_INT4_G64, FMT_INT4_G128):
        return (N, K // 2)
    if fmt in (FMT_INT8_G64, FMT_FP8_B128):
        return (N, K)
    raise ValueError(f"unknown format {fmt}")


def scale_shape(fmt: int, N: int, K: int) -> tuple:
    """Scale array shape and numpy dtype for one matrix."""
    if fmt == FMT_NVFP4:
        return (N, K // 16), np.uint8
    if fmt == FMT_MXFP4:
        return (N, K // 32), np.uint8
    if fmt in (FMT_INT4_G64, FMT_INT8_G64):
        return (N, K // 64), np.uint16  # bf16 bit patterns
    if fmt == FMT_FP8_B128:
        return (N // 128, K // 128), np.float32
    if fmt == FMT_INT4_G128:
        return (N, K // 128), np.uint16  # f16 bit patterns
    raise ValueError(f"unknown format {fmt}")


def quantize(fmt: int, W: np.ndarray):
    """Encode one FP32 matrix W[N, K]; returns (data, scales, tensor_scale)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    data = np.zeros(data_shape(fmt, N, K), dtype=np.uint8)
    sshape, sdt = scale_shape(fmt, N, K)
    scales = np.zeros(sshape, dtype=sdt)
    ts = np.ones(1, dtype=np.float32)
    rc = lib().qs_quantize(fmt, _ptr(W), N, K, _ptr(data), _ptr(scales), _ptr(ts))
    if rc != 0:
        raise ValueError(f"shape {W.shape} not valid for format {fmt}")
    return data, scales, float(ts[0])


@dataclass
class QMat:
    """A stack of E quantized matrices W_e[N, K] in one format."""
    fmt: int
    N: int
    K: int
    data: np.ndarray      # [E, *data_shape]
    scales: np.ndarray    # [E, *scale_shape]
    ts: np.ndarray        # [E] float32 (NVFP4 tensor scale; 1.0 otherwise)

    @property
    def E(self) -> int:
        return self.data.shape[0]

    def nbytes(self) -> int:
        return self.data.nbytes + self.scales.nbytes + (self.ts.nbytes if self.fmt == FMT_NVFP4 else 0)

    def expert(self, e: int) -> "QMat":
        return QMat(self.fmt, self.N, self.K, self.data[e:e + 1], self.scales[e:e + 1], self.ts[e:e + 1])


def make_stack(fmt: int, seed: int, kind: int, proj: int, expert0: int, E: int, N: int, K: int,
               sigma: float = WEIGHT_SIGMA, nthreads: int = 0) -> QMat:
    data = np.empty((E,) + data_shape(fmt, N, K), dtype=np.uint8)
    sshape, sdt = scale_shape(fmt, N, K)
    scales = np.empty((E,) + sshape, dtype=sdt)
    ts = np.ones(E, dtype=np.float32)
    rc = lib().qs_make_stack(fmt, seed, kind, proj, expert0, E, N, K, sigma, _ptr(data), _ptr(scales), _ptr(ts),
                             nthreads)
    if rc != 0:
        raise RuntimeError(f"qs_make_stack failed ({rc})")
    return QMat(fmt, N, K, data, scales, ts)


@dataclass
class HostLayer:
    """One MoE layer's parameters in host memory (checkpoint formats)."""
    cfg: LayerConfig
    seed: int
    router_w: np.ndarray                 # [E, H] float32
    router_b: Optional[np.ndarray]       # [E] float32 or None
    gate: QMat                           # [E] x [I, H]
    up: QMat                             # [E] x [I, H]
    down: QMat                           # [E] x [H, I]
    shared_gate: Optional[QMat] = None   # [1] x [Is, H]
    shared_up: Optional[QMat] = None
    shared_down: Optional[QMat] = None   # [1] x [H, Is]
    extra: dict = field(default_factory=dict)

    def expert_bytes(self) -> int:
        """Packed bytes of one routed expert (gate + up + down, data + scales + tensor scales)."""
        return sum(m.nbytes() // m.E for m in (self.gate, self.up, self.down))

    def router_bytes(self) -> int:
        return self.router_w.nbytes + (self.router_b.nbytes if self.router_b is not None else 0)

    def shared_bytes(self) -> int:
        if self.shared_gate is None:
            return 0
        return sum(m.nbytes() for m in (self.shared_gate, self.shared_up, self.shared_down))


def zipf_bias(cfg: LayerConfig, seed: int) -> np.ndarray:
    """Router bias b[e] = -s * ln(pi(e) + 1) for a seeded permutation pi (Zipf load skew)."""
    perm = np.empty(cfg.E, dtype=np.int32)
    lib().qs_permutation(stream_key(seed, KIND_ZIPF, 0, 0), cfg.E, _ptr(perm))
    return (-cfg.zipf_s * np.log(perm.astype(np.float64) + 1.0)).astype(np.float32)


def make_expert(cfg: LayerConfig, seed: int, e: int):
    """Regenerate only routed expert e: (gate, up, down) as single-expert QMat stacks."""
    return tuple(make_stack(cfg.fmt, seed, KIND_ROUTED, p, e, 1, N, K, nthreads=1)
                 for p, (N, K) in enumerate(((cfg.I, cfg.H), (cfg.I, cfg.H), (cfg.H, cfg.I))))


def make_layer(cfg: LayerConfig, seed: int = 0, nthreads: int = 0) -> HostLayer:
    H, E, I = cfg.H, cfg.E, cfg.I
    rw = normal_f32(stream_key(seed, KIND_ROUTER, 0, 0), E * H, WEIGHT_SIGMA).reshape(E, H)
    rb = zipf_bias(cfg, seed) if cfg.zipf_s else None
    gate = make_stack(cfg.fmt, seed, KIND_ROUTED, 0, 0, E, I, H, nthreads=nthreads)
    up = make_stack(cfg.fmt, seed, KIND_ROUTED, 1, 0, E, I, H, nthreads=nthreads)
    down = make_stack(cfg.fmt, seed, KIND_ROUTED, 2, 0, E, H, I, nthreads=nthreads)
    sg = su = sd = None
    if cfg.shared_fmt:
        Is = cfg.shared_I
        sg = make_stack(cfg.shared_fmt, seed, KIND_SHARED, 0, 0, 1, Is, H, nthreads=nthreads)
        su = make_stack(cfg.shared_fmt, seed, KIND_SHARED, 1, 0, 1, Is, H, nthreads=nthreads)
        sd = make_stack(cfg.shared_fmt, seed, KIND_SHARED, 2, 0, 1, H, Is, nthreads=nthreads)
    return HostLayer(cfg, seed, rw, rb, gate, up, down, sg, su, sd)


def make_tokens(cfg: LayerConfig, T: int, seed: int = 0, batch: int = 0) -> np.ndarray:
    """Activations x[T, H]: N(0, 1) rounded to bf16, as uint16 bit patterns."""
    return normal_bf16(stream_key(seed, KIND_TOKENS, batch, 0), T * cfg.H, 1.0).reshape(T, cfg.H)
