"""moe_decode_forward_noalloc: the decode forward for callers that cannot
allocate device memory (a host framework that owns every device buffer and
gives plugins no allocator, or a serving loop that forbids allocation once it
runs).  It uses the library's fixed 32 MiB device array as its workspace.

Checked through the C ABI: two calls in a row give the same outputs as
moe_decode_forward with a caller workspace (within the layer tolerance the
other tests use), and a layer whose workspace would exceed the fixed array is
rejected before anything is launched.  Runs last (file name) so a failure here
cannot stop the rest of a -x run; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from oracle import formats as F
from oracle import moe as M
from quantized_moe_decode_router_gb300 import _binding as B
from quantized_moe_decode_router_gb300 import build as qbuild
from quantized_moe_decode_router_gb300.device import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return B.load()


@pytest.mark.parametrize("name,T", [("tiny_nvfp4", 1), ("decode_nvfp4", 8), ("decode_nvfp4", 3)])
def test_noalloc_matches_workspace_entry_point(lib, name, T):
    cfg = synth.CONFIGS[name]
    host = synth.make_layer(cfg, seed=2)
    dev = to_device(host)
    ws = torch.empty(B.workspace_size(dev, T), dtype=torch.uint8, device="cuda")
    B.workspace_init(ws)
    for call in range(2):  # two calls in a row: the shared array must not carry state over
        xb = synth.make_tokens(cfg, T, seed=2, batch=10 * T + call)
        x = torch.from_numpy(xb.view(np.int16)).cuda()
        y_ref = torch.zeros((T, cfg.H), dtype=torch.int16, device="cuda")
        y_na = torch.zeros((T, cfg.H), dtype=torch.int16, device="cuda")
        B.moe_decode_forward(dev, x, T, y_ref, ws)
        B.moe_decode_forward_noalloc(dev, x, T, y_na)
        torch.cuda.synchronize()
        a = F.bf16_to_f64(y_na.cpu().numpy().view(np.uint16))
        r = F.bf16_to_f64(y_ref.cpu().numpy().view(np.uint16))
        assert np.all(M.within_tolerance(a, r)), f"call {call}: {np.abs(a - r).max()}"
        assert np.isfinite(a).all()


def test_noalloc_rejects_layers_beyond_its_array(lib):
    fake = 0x7F0000000000
    qw = lambda base: B.moe_qweight(base, base + 0x100000, base + 0x200000)
    big = B.moe_layer(16384, 8192, 1024, 16, B.MOE_FMT_NVFP4, fake, None, qw(fake + 0x1000000),
                      qw(fake + 0x2000000), qw(fake + 0x3000000), 0, 0, qw(0), qw(0), qw(0))
    assert lib.moe_workspace_size(ctypes.byref(big), 8, None) > 32 << 20
    st = lib.moe_decode_forward_noalloc(ctypes.byref(big), fake, 8, fake, None, None)
    assert st == B.MOE_ERR_WORKSPACE, B.status_string(st)
