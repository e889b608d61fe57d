"""moe_decode_forward_noalloc: the decode forward for callers that cannot
allocate device memory (a host framework that owns every device buffer and
gives plugins no allocator, or a serving loop that forbids allocation once it
runs).  It uses the library's fixed 32 MiB device array as its workspace.

Checked through the C ABI:
  * two calls in a row give bit for bit the outputs of moe_decode_forward
    with a caller workspace (both run the same deterministic kernels, so any
    difference would be state carried over in the shared array);
  * the first call of a fresh process, made on a non-blocking stream, is
    ordered before its own kernels (its counter clearing runs on that stream);
  * the device-side error word of the array reads clean through
    moe_check(NULL, 0, stream);
  * a layer whose workspace would exceed the fixed array is rejected.
Runs last (file name) so a failure here cannot stop the rest of a -x run; it
also passes alone in a fresh process.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import synth
from quantized_moe_decode_router_gb300 import _binding as B
from quantized_moe_decode_router_gb300 import build as qbuild
from quantized_moe_decode_router_gb300.device import to_device

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return B.load()


@pytest.mark.parametrize("name,T", [("tiny_nvfp4", 1), ("decode_nvfp4", 8), ("decode_nvfp4", 3),
                                    ("decode_mxfp4", 8)])
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
        y_na = torch.full((T, cfg.H), -1, dtype=torch.int16, device="cuda")
        B.moe_decode_forward(dev, x, T, y_ref, ws)
        B.moe_decode_forward_noalloc(dev, x, T, y_na)
        torch.cuda.synchronize()
        assert torch.equal(y_na, y_ref), f"call {call}: {int((y_na != y_ref).sum())} outputs differ"
    assert B.moe_check(ws) == 0
    assert B.moe_check_noalloc() == 0


_FRESH = r"""
import numpy as np, torch, synth
from quantized_moe_decode_router_gb300 import _binding as B
from quantized_moe_decode_router_gb300.device import to_device
B.load()
cfg = synth.CONFIGS["decode_nvfp4"]
dev = to_device(synth.make_layer(cfg, seed=4))
T = 8
x = torch.from_numpy(synth.make_tokens(cfg, T, seed=4, batch=1).view(np.int16)).cuda()
ws = torch.empty(B.workspace_size(dev, T), dtype=torch.uint8, device="cuda")
B.workspace_init(ws)
y_ref = torch.zeros((T, cfg.H), dtype=torch.int16, device="cuda")
B.moe_decode_forward(dev, x, T, y_ref, ws)
torch.cuda.synchronize()
s = torch.cuda.Stream()                  # non-blocking with respect to the legacy default stream
outs = []
with torch.cuda.stream(s):
    for i in range(2):
        y = torch.full((T, cfg.H), -1, dtype=torch.int16, device="cuda")
        B.moe_decode_forward_noalloc(dev, x, T, y, stream=s)
        outs.append(y)
s.synchronize()
assert all(torch.equal(y, y_ref) for y in outs), [int((y != y_ref).sum()) for y in outs]
assert B.moe_check_noalloc(s) == 0
print("fresh-process no-alloc ok")
"""


def test_noalloc_first_call_on_a_non_blocking_stream_in_a_fresh_process(lib):
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", _FRESH], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "fresh-process no-alloc ok" in r.stdout


def test_noalloc_rejects_layers_beyond_its_array(lib):
    fake = 0x7F0000000000
    qw = lambda base: B.moe_qweight(base, base + 0x100000, base + 0x200000)
    big = B.moe_layer(16384, 8192, 1024, 16, B.MOE_FMT_NVFP4, fake, None, qw(fake + 0x1000000),
                      qw(fake + 0x2000000), qw(fake + 0x3000000), 0, 0, qw(0), qw(0), qw(0))
    assert lib.moe_workspace_size(ctypes.byref(big), 4, None) > 32 << 20
    st = lib.moe_decode_forward_noalloc(ctypes.byref(big), fake, 4, fake, None, None)
    assert st == B.MOE_ERR_WORKSPACE, B.status_string(st)
