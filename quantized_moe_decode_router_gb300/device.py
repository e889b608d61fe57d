"""Place checkpoint-format weights in device memory as a binding ``Layer``.

Takes any host object with the layer's fields (router weights and bias,
stacked gate / up / down matrices as ``data`` / ``scales`` / ``ts`` numpy
arrays, optional shared expert) and copies the bytes unchanged: weights
stay in their published encoding, there is no conversion step.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from ._binding import MOE_FMT_NVFP4, Layer, QWeight


def _dev(a: np.ndarray, device) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.uint8).reshape(-1) if a.dtype != np.float32 else a.reshape(-1))
    return t.to(device, non_blocking=False)


def qweight_to_device(qm, device="cuda") -> QWeight:
    """One stacked weight (data / scales / tensor scales) copied to the device unchanged."""
    ts = torch.from_numpy(np.ascontiguousarray(qm.ts, dtype=np.float32)).to(device) if qm.fmt == MOE_FMT_NVFP4 \
        else None
    return QWeight(_dev(qm.data, device), _dev(qm.scales, device), ts)


@dataclass
class DeviceLayer:
    layer: Layer
    nbytes: int

    def __getattr__(self, name):
        return getattr(self.layer, name)


def to_device(host, device: Optional[str] = "cuda") -> Layer:
    cfg = host.cfg
    rw = torch.from_numpy(np.ascontiguousarray(host.router_w, dtype=np.float32)).to(device)
    rb = None if host.router_b is None else torch.from_numpy(
        np.ascontiguousarray(host.router_b, dtype=np.float32)).to(device)
    lay = Layer(hidden=cfg.H, inter=cfg.I, n_experts=cfg.E, top_k=cfg.k, fmt=cfg.fmt, router_w=rw, router_bias=rb,
                gate=qweight_to_device(host.gate, device), up=qweight_to_device(host.up, device), down=qweight_to_device(host.down, device))
    if host.shared_gate is not None:
        lay.shared_fmt = cfg.shared_fmt
        lay.shared_inter = cfg.shared_I
        lay.shared_gate = qweight_to_device(host.shared_gate, device)
        lay.shared_up = qweight_to_device(host.shared_up, device)
        lay.shared_down = qweight_to_device(host.shared_down, device)
        gw = getattr(host, "extra", {}).get("shared_gate_w")
        if gw is not None:
            lay.shared_expert_gate = torch.from_numpy(np.ascontiguousarray(gw, dtype=np.float32)).to(device)
    lay.bias_select = int(getattr(host, "extra", {}).get("bias_select", 0))
    return lay
