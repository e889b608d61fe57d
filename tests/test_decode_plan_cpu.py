"""Host-side launch planning of the decode path (no GPU): for every decode
layer shape the tests and the bench use, each token count and several SM
counts, the plan that moe_decode_forward would launch with must fit in shared
memory, split K only along whole blocks (so the fixed block-order sum is the
same for every split), and store no more block sums than the workspace holds."""
import ctypes

import pytest

from quantized_moe_decode_router_gb300 import _binding as B
from quantized_moe_decode_router_gb300 import build as qbuild
from synth.configs import (CONFIGS, FMT_FP8_B128, FMT_INT4_G64, FMT_INT8_G64, FMT_MXFP4, FMT_NVFP4,
                           LayerConfig)

FAKE = 0x7F0000000000  # 256-byte aligned, never dereferenced: planning reads shapes only


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return B.load()


def _qw(base):
    return B.moe_qweight(base, base + 0x100000, base + 0x200000)


def _layer(cfg: LayerConfig):
    sf = cfg.shared_fmt or 0
    return B.moe_layer(cfg.H, cfg.I, cfg.E, cfg.k, cfg.fmt, FAKE, None,
                       _qw(FAKE + 0x1000000), _qw(FAKE + 0x2000000), _qw(FAKE + 0x3000000),
                       sf, cfg.shared_I if sf else 0,
                       _qw(FAKE + 0x4000000), _qw(FAKE + 0x5000000), _qw(FAKE + 0x6000000))


def _blocks(fmt: int, K: int) -> int:
    """Fixed K blocks of a tile: units of 128 columns (4-bit codes) or 64 (8-bit), two per block when even."""
    unit = 128 if fmt in (FMT_NVFP4, FMT_MXFP4, FMT_INT4_G64) else 64
    units = K // unit
    return units // 2 if units % 2 == 0 else units


def _pow2(v: int) -> bool:
    return v >= 1 and v & (v - 1) == 0


LAYERS = [c for c in CONFIGS.values() if c.name.startswith("decode") or c.name.startswith("tiny")] + [
    LayerConfig("s_nvfp4_fp8", FMT_NVFP4, H=512, E=24, k=5, I=256, shared_fmt=FMT_FP8_B128, shared_I=384),
    LayerConfig("s_mxfp4", FMT_MXFP4, H=640, E=12, k=3, I=384),
    LayerConfig("s_int4_int8", FMT_INT4_G64, H=768, E=16, k=4, I=256, shared_fmt=FMT_INT8_G64, shared_I=512),
    LayerConfig("s_int8", FMT_INT8_G64, H=512, E=9, k=2, I=128, shared_fmt=FMT_NVFP4, shared_I=256),
    LayerConfig("s_fp8", FMT_FP8_B128, H=384, E=6, k=6, I=256, shared_fmt=FMT_MXFP4, shared_I=128),
    LayerConfig("nvfp4_no_shared", FMT_NVFP4, H=2048, E=512, k=10, I=512),
]


@pytest.mark.parametrize("cfg", LAYERS, ids=[c.name for c in LAYERS])
def test_decode_plan_invariants(lib, cfg):
    L = _layer(cfg)
    Br, Brd = _blocks(cfg.fmt, cfg.H), _blocks(cfg.fmt, cfg.I)
    Bs = _blocks(cfg.shared_fmt, cfg.H) if cfg.shared_fmt else None
    for sms in (132, 148, 152, 160):
        for T in range(1, B.MOE_DECODE_MAX_TOKENS + 1):
            p = B.moe_decode_plan_info()
            st = lib.moe_decode_plan(ctypes.byref(L), T, sms, ctypes.byref(p))
            assert st == 0, (cfg.name, T, sms, B.status_string(st))
            assert p.gu_smem <= 227 * 1024 and p.dn_smem <= 227 * 1024
            assert p.gu_ctas_per_sm == (3 if T <= 4 else 2)
            assert 1 <= p.dn_segs <= 4
            for S in (p.gu_slices, p.gu_slices_tail, p.gu_slices_shared, p.dn_slices):
                assert _pow2(S), (cfg.name, T, S)
            assert Br % p.gu_slices == 0 and Br % p.gu_slices_tail == 0
            assert p.gu_slices_tail >= p.gu_slices and p.gu_slices_tail <= 8
            assert Brd % p.dn_slices == 0
            if Bs is not None:
                assert Bs % p.gu_slices_shared == 0
            else:
                assert p.gu_slices_shared == p.gu_slices
            assert p.gu_split_blocks <= p.split_block_capacity
            assert p.dn_split_blocks <= p.split_block_capacity
            assert p.gu_tail_cap >= 0


def test_decode_plan_rejects_bad_arguments(lib):
    L = _layer(CONFIGS["decode_nvfp4"])
    p = B.moe_decode_plan_info()
    for T, sms in ((0, 152), (B.MOE_DECODE_MAX_TOKENS + 1, 152), (1, 0)):
        assert lib.moe_decode_plan(ctypes.byref(L), T, sms, ctypes.byref(p)) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_decode_plan(ctypes.byref(L), 1, 152, None) == B.MOE_ERR_INVALID_ARG
    assert lib.moe_decode_plan(None, 1, 152, ctypes.byref(p)) == B.MOE_ERR_INVALID_ARG


def test_decode_plan_reports_staging_that_does_not_fit(lib):
    # 8 tokens of a 12288-wide hidden state alone take 197 KB of the gate/up CTA's shared memory
    L = _layer(LayerConfig("wide", FMT_NVFP4, H=12288, E=64, k=4, I=512))
    p = B.moe_decode_plan_info()
    assert lib.moe_decode_plan(ctypes.byref(L), 1, 152, ctypes.byref(p)) == 0
    assert lib.moe_decode_plan(ctypes.byref(L), 8, 152, ctypes.byref(p)) == B.MOE_ERR_UNSUPPORTED
