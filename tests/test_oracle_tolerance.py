"""Pins for the parity bar itself: the BF16 unit in the last place, the
per-element tolerance max(2 BF16 ulp, 1e-3) that every layer comparison uses,
and the FP64 -> BF16 encoder's special cases.  The references are the BF16
definition (8 significant bits, binary32 exponent range, subnormal spacing
2^-133), enumerated over every bit pattern, not the functions under test."""
import numpy as np
import pytest

from oracle import formats as F
from oracle import moe as M


def test_bf16_ulp_is_the_spacing_to_the_next_bf16_value_for_every_pattern():
    bits = np.arange(0x0000, 0x7F7F, dtype=np.uint32)  # 0 .. largest finite - 1
    v = F.bf16_to_f64(bits.astype(np.uint16))
    nxt = F.bf16_to_f64((bits + 1).astype(np.uint16))
    spacing = nxt - v
    ulp = M.bf16_ulp(v)
    pos = v > 0
    assert np.array_equal(ulp[pos], spacing[pos])
    assert np.array_equal(M.bf16_ulp(-v[pos]), spacing[pos])  # symmetric in sign


@pytest.mark.parametrize("v,ulp", [
    (1.0, 2.0 ** -7), (1.9921875, 2.0 ** -7), (2.0, 2.0 ** -6), (0.75, 2.0 ** -8), (-3.0, 2.0 ** -6),
    (2.0 ** -126, 2.0 ** -133), (2.0 ** -130, 2.0 ** -133), (0.0, 2.0 ** -133), (448.0, 2.0 ** 1),
])
def test_bf16_ulp_closed_forms(v, ulp):
    assert M.bf16_ulp(np.array([v]))[0] == ulp


def test_tolerance_is_max_of_two_ulp_and_abs():
    ref = np.array([1.0, 1.0, 1e-4, 1e-4, 64.0, 64.0, -2.0])
    got = np.array([1.0 + 2 * 2.0 ** -7,            # exactly 2 ulp: inside (inclusive)
                    1.0 + 2 * 2.0 ** -7 + 1e-9,     # just beyond 2 ulp
                    1e-4 + 1e-3,                    # abs bar dominates near zero: inside
                    1e-4 + 1.001e-3,                # beyond the abs bar
                    64.0 - 1.25,                    # 2 ulp at 64 is 2 * 2**-1 = 1.0: 1.25 is outside
                    64.0 - 0.5,                     # 1 ulp: inside
                    -2.0 - 2 * 2.0 ** -6])          # negative side, exactly 2 ulp
    ok = M.within_tolerance(got, ref)
    assert ok.tolist() == [True, False, True, False, False, True, True]
    assert not M.within_tolerance(np.array([np.nan]), np.array([1.0]))[0]


def test_bf16_encoder_special_cases():
    max_bf16 = F.bf16_to_f64(np.array([0x7F7F], dtype=np.uint16))[0]
    half_ulp_at_max = 2.0 ** (127 - 8)
    enc = F.f64_to_bf16_bits(np.array([max_bf16, max_bf16 + half_ulp_at_max * 0.999,
                                       max_bf16 + half_ulp_at_max, -0.0, np.nan, -np.inf]))
    assert enc[0] == 0x7F7F and enc[1] == 0x7F7F     # rounds down to the largest finite value
    assert enc[2] == 0x7F80                          # the tie rounds to even: the exponent overflows to +Inf
    assert enc[3] == 0x8000                          # -0 keeps its sign
    assert np.isnan(F.bf16_to_f64(enc[4:5]))[0]
    assert enc[5] == 0xFF80
