"""C ABI checks that need no GPU: the library builds and loads, exports every
entry point include/moe.h declares, and rejects invalid arguments on the host
before any launch (fake, never-dereferenced device addresses)."""
import ctypes
import os
import re

import pytest

from quantized_moe_decode_router_gb300 import _binding as B
from quantized_moe_decode_router_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return B.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\*?\s+\**(moe_[a-z_0-9]+)\s*\(", src, re.M)))


def test_exports_every_declared_entry_point(lib):
    names = _declared()
    assert len(names) >= 10, names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(B._SIGNATURES), (set(names) ^ set(B._SIGNATURES))


def test_status_strings(lib):
    for st in range(-7, 1):
        assert B.status_string(st).startswith("MOE_")
    assert "unknown" in B.status_string(-99)


FAKE = 0x7F0000000000  # 256-byte aligned, never dereferenced (validation rejects first or we never launch)


def _qw(fmt, base, ts=True):
    return B.moe_qweight(base, base + 0x100000, (base + 0x200000) if ts else None)


def _layer(**kw):
    d = dict(hidden=2048, inter=512, n_experts=512, top_k=10, fmt=B.MOE_FMT_NVFP4)
    d.update(kw)
    L = B.moe_layer(d["hidden"], d["inter"], d["n_experts"], d["top_k"], d["fmt"], FAKE, None,
                    _qw(d["fmt"], FAKE + 0x1000000), _qw(d["fmt"], FAKE + 0x2000000), _qw(d["fmt"], FAKE + 0x3000000),
                    d.get("shared_fmt", 0), d.get("shared_inter", 0),
                    _qw(0, FAKE + 0x4000000), _qw(0, FAKE + 0x5000000), _qw(0, FAKE + 0x6000000))
    return L


def _ws_size(lib, L, T=8):
    return lib.moe_workspace_size(ctypes.byref(L), T, None)


def test_workspace_size_and_layout(lib):
    L = _layer()
    n = _ws_size(lib, L)
    assert n > 8 * 512 * 4
    assert _ws_size(lib, L, 16) > n
    out = B.moe_ws_layout()
    assert lib.moe_workspace_layout(ctypes.byref(L), 8, None, ctypes.byref(out)) == 0
    assert out.total == n
    offs = [out.logits, out.topk_idx, out.topk_w, out.expert_cnt, out.expert_off, out.pair_list]
    assert all(o % 256 == 0 for o in offs) and len(set(offs)) == len(offs)
    bad = _layer(top_k=0)
    assert _ws_size(lib, bad) == 0


@pytest.mark.parametrize("mut,status", [
    (dict(top_k=0), B.MOE_ERR_INVALID_ARG),
    (dict(top_k=17), B.MOE_ERR_UNSUPPORTED),
    (dict(n_experts=4, top_k=5), B.MOE_ERR_UNSUPPORTED),
    (dict(n_experts=2048), B.MOE_ERR_UNSUPPORTED),
    (dict(fmt=9), B.MOE_ERR_INVALID_ARG),
    (dict(hidden=2000), B.MOE_ERR_UNSUPPORTED),
    (dict(inter=100), B.MOE_ERR_UNSUPPORTED),
    (dict(shared_fmt=7, shared_inter=512), B.MOE_ERR_INVALID_ARG),
])
def test_invalid_layers_rejected_before_launch(lib, mut, status):
    L = _layer(**mut)
    ws = FAKE
    st = lib.moe_decode_forward(ctypes.byref(L), FAKE, 1, FAKE, None, ws, 1 << 30, None)
    assert st == status, B.status_string(st)


def test_invalid_calls_rejected_before_launch(lib):
    L = _layer()
    n = _ws_size(lib, L)
    f = lib.moe_decode_forward
    assert f(None, FAKE, 1, FAKE, None, FAKE, n, None) == B.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(L), None, 1, FAKE, None, FAKE, n, None) == B.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(L), FAKE + 8, 1, FAKE, None, FAKE, n, None) == B.MOE_ERR_MISALIGNED
    assert f(ctypes.byref(L), FAKE, 0, FAKE, None, FAKE, n, None) == B.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(L), FAKE, 9, FAKE, None, FAKE, n, None) == B.MOE_ERR_UNSUPPORTED
    assert f(ctypes.byref(L), FAKE, 1, FAKE, None, None, n, None) == B.MOE_ERR_WORKSPACE
    assert f(ctypes.byref(L), FAKE, 8, FAKE, None, FAKE, 1024, None) == B.MOE_ERR_WORKSPACE
    assert f(ctypes.byref(L), FAKE, 1, FAKE, None, FAKE + 16, n, None) == B.MOE_ERR_MISALIGNED
    o = B._opts(act_quant=1)
    assert f(ctypes.byref(L), FAKE, 1, FAKE, ctypes.byref(o), FAKE, n, None) == B.MOE_ERR_UNSUPPORTED
    o = B._opts(fold_scales=1)   # a prefill-only lever: refused by the decode entry points, never ignored
    assert f(ctypes.byref(L), FAKE, 1, FAKE, ctypes.byref(o), FAKE, n, None) == B.MOE_ERR_UNSUPPORTED
    o = B._opts(fp8_act=1)
    assert f(ctypes.byref(L), FAKE, 1, FAKE, ctypes.byref(o), FAKE, n, None) == B.MOE_ERR_UNSUPPORTED
    o = B._opts()
    o.reserved[0] = 1
    assert f(ctypes.byref(L), FAKE, 1, FAKE, ctypes.byref(o), FAKE, n, None) == B.MOE_ERR_INVALID_ARG
    for bad in (dict(bf16_partials=2), dict(wait_limit_us=-1), dict(fold_scales=2), dict(fp8_act=-1)):
        o = B._opts(**bad)
        assert f(ctypes.byref(L), FAKE, 1, FAKE, ctypes.byref(o), FAKE, n, None) == B.MOE_ERR_INVALID_ARG, bad
    # a shared-expert gate without a shared expert, a bias mode outside 0/1
    L4 = _layer()
    L4.shared_expert_gate = FAKE
    assert f(ctypes.byref(L4), FAKE, 1, FAKE, None, FAKE, n, None) == B.MOE_ERR_INVALID_ARG
    L5 = _layer()
    L5.bias_select = 2
    assert f(ctypes.byref(L5), FAKE, 1, FAKE, None, FAKE, n, None) == B.MOE_ERR_INVALID_ARG
    # a missing NVFP4 tensor scale, a misaligned weight pointer
    L2 = _layer()
    L2.gate.tensor_scale = None
    assert f(ctypes.byref(L2), FAKE, 1, FAKE, None, FAKE, n, None) == B.MOE_ERR_INVALID_ARG
    L3 = _layer()
    L3.up.data = FAKE + 0x2000008
    assert f(ctypes.byref(L3), FAKE, 1, FAKE, None, FAKE, n, None) == B.MOE_ERR_MISALIGNED
    # routing entry point: same checks
    r = lib.moe_route
    assert r(ctypes.byref(L), FAKE, 0, None, None, None, None, None, FAKE, n, None) == B.MOE_ERR_INVALID_ARG
    assert r(ctypes.byref(L), FAKE, 1, FAKE + 2, None, None, None, None, FAKE, n, None) == B.MOE_ERR_MISALIGNED
    # dequantize / activation quantizer argument checks
    q = _qw(B.MOE_FMT_NVFP4, FAKE)
    assert lib.moe_dequantize(B.MOE_FMT_NVFP4, ctypes.byref(q), 512, 2048, 0, 500, 20, FAKE, None) == \
        B.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_act_nvfp4(FAKE, 4, 100, FAKE, FAKE, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_init(None, 1024, None) == B.MOE_ERR_WORKSPACE


def test_noalloc_rejects_bad_calls_before_touching_the_device(lib):
    # every host check of moe_decode_forward runs before the allocation-free entry point looks up its
    # device array or clears anything: on a machine without a GPU a call that reached the device would
    # return MOE_ERR_CUDA instead of these codes
    L = _layer()
    f = lib.moe_decode_forward_noalloc
    assert f(ctypes.byref(L), FAKE, 1, None, None, None) == B.MOE_ERR_INVALID_ARG        # null y
    assert f(ctypes.byref(L), None, 1, FAKE, None, None) == B.MOE_ERR_INVALID_ARG        # null x
    assert f(ctypes.byref(L), FAKE, 1, FAKE + 4, None, None) == B.MOE_ERR_MISALIGNED
    assert f(ctypes.byref(L), FAKE, 0, FAKE, None, None) == B.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(L), FAKE, 9, FAKE, None, None) == B.MOE_ERR_UNSUPPORTED        # as moe_decode_forward
    o = B._opts(act_quant=1)
    assert f(ctypes.byref(L), FAKE, 1, FAKE, ctypes.byref(o), None) == B.MOE_ERR_UNSUPPORTED
    assert f(None, FAKE, 1, FAKE, None, None) == B.MOE_ERR_INVALID_ARG
    big = _layer(hidden=16384, inter=8192, n_experts=1024, top_k=16)
    assert lib.moe_workspace_size(ctypes.byref(big), 4, None) > 32 << 20
    assert f(ctypes.byref(big), FAKE, 4, FAKE, None, None) == B.MOE_ERR_WORKSPACE


def test_check_reports_short_workspaces(lib):
    assert lib.moe_check(None, 16, None) == B.MOE_ERR_WORKSPACE
    assert lib.moe_check(FAKE, 4, None) == B.MOE_ERR_WORKSPACE


def test_binding_structs_match_the_header_layout(tmp_path):
    # every struct the binding passes across the boundary has the C header's size and field offsets:
    # a small C program compiled against include/moe.h prints them (gcc, no GPU)
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    header = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")
    structs = {"moe_qweight": B.moe_qweight, "moe_layer": B.moe_layer, "moe_options": B.moe_options,
               "moe_ws_layout": B.moe_ws_layout, "moe_decode_plan_info": B.moe_decode_plan_info}
    lines = [f'#include "{header}"', "#include <stdio.h>", "#include <stddef.h>", "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'  printf("{name} sizeof %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'  printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-std=c11", "-o", str(exe), str(src)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    c_vals = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for name, cls in structs.items():
        assert c_vals[(name, "sizeof")] == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert c_vals[(name, field)] == getattr(cls, field).offset, (name, field)
