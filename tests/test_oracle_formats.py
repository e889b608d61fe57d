"""Pins for the oracle's format decoders and the generator's encoders.

Every decoder is checked against something other than itself: torch's CPU
float8 / bfloat16 casts (independent library decoders), hand-built layouts
written from the format definitions, and exact rational rounding.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth
from oracle import formats as F


# ------------------------------------------------------------ code tables ----

def test_e4m3_table_matches_torch_all_256_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(F.E4M3_TABLE))
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan], F.E4M3_TABLE[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(F.E4M3_TABLE[~nan]))


def test_e8m0_table_matches_torch_all_256_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.isnan(ref[255]) and np.isnan(F.E8M0_TABLE[255])
    assert np.array_equal(ref[:255], F.E8M0_TABLE[:255])


def _e2m1_to_e4m3_code(c: int) -> int:
    """Re-encode an E2M1 code as the E4M3 code of the same value, by bit fields.

    E2M1 exponent bias 1, E4M3 bias 7: a normal E2M1 exponent e maps to e + 6
    and its 1-bit mantissa to the top of the 3-bit mantissa; the E2M1
    subnormal 0.5 (e=0, m=1) is the E4M3 normal 2^-1 (exponent 6, mantissa 0).
    """
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    if e == 0:
        body = 0 if m == 0 else (6 << 3)
    else:
        body = ((e + 6) << 3) | (m << 2)
    return (s << 7) | body


def test_e2m1_table_all_16_codes_via_torch_e4m3():
    codes = [_e2m1_to_e4m3_code(c) for c in range(16)]
    ref = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ref, F.E2M1_TABLE)
    assert np.array_equal(np.signbit(ref), np.signbit(F.E2M1_TABLE))
    # magnitudes 0..7 strictly increasing, largest 6: the E2M1 range
    assert np.all(np.diff(F.E2M1_TABLE[:8]) > 0) and F.E2M1_TABLE[7] == 6.0


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 65536, size=20000, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = F.bf16_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def _bf16_round_exact(v: float) -> float:
    """Nearest BF16 to v by exact rational comparison (ties to even mantissa)."""
    if v == 0:
        return v
    a = Fraction(abs(v))
    e = 0
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    while Fraction(2) ** e > a:
        e -= 1
    q = max(e - 7, -133)
    step = Fraction(2) ** q
    lo = (a // step) * step
    hi = lo + step
    if a - lo < hi - a:
        r = lo
    elif hi - a < a - lo:
        r = hi
    else:
        r = lo if (lo / step) % 2 == 0 else hi
    return float(r) if v > 0 else -float(r)


def test_bf16_rounding_single_rounding_from_f64():
    # fp32-representable inputs: single rounding equals torch's fp32 -> bf16 RNE
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.round_bf16(v.astype(np.float64)), ref)
    # inputs that round differently through an fp32 intermediate (double rounding)
    cases = [1 + 2.0 ** -8 + 2.0 ** -30, 1 + 2.0 ** -8 - 2.0 ** -30, 3 * (1 + 2.0 ** -8) + 2.0 ** -40,
             -(1 + 2.0 ** -8 + 2.0 ** -33), 2.0 ** -130 * (1 + 2.0 ** -3) + 2.0 ** -160]
    for c in cases:
        assert F.round_bf16(np.array([c]))[0] == _bf16_round_exact(c), c
    # ties go to even
    assert F.round_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert F.round_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6


# ------------------------------------------------------- checkpoint layout ----

def test_nvfp4_layout_hand_built():
    # row 0: byte 0x21 -> k0 = code 1 (0.5), k1 = code 2 (1.0); byte 0xF9 -> k2 = -0.5, k3 = -6
    data = np.zeros((1, 8), dtype=np.uint8)
    data[0, 0], data[0, 1] = 0x21, 0xF9
    scales = np.array([[0x38]], dtype=np.uint8)          # E4M3 0x38 = 1.0
    W = F.decode(F.FMT_NVFP4, data, scales, 0.5, 1, 16)
    assert list(W[0, :4]) == [0.25, 0.5, -0.25, -3.0]
    assert np.all(W[0, 4:] == 0)


def test_mxfp4_layout_hand_built():
    data = np.zeros((1, 16), dtype=np.uint8)
    data[0, 0] = 0x7B                                     # k0 = code 11 (-1.5), k1 = code 7 (6)
    scales = np.array([[130]], dtype=np.uint8)            # 2^3
    W = F.decode(F.FMT_MXFP4, data, scales, 1.0, 1, 32)
    assert list(W[0, :2]) == [-12.0, 48.0]


def test_int4_int8_layout_hand_built():
    data = np.zeros((1, 32), dtype=np.uint8)
    data[0, 0] = 0xF8                                     # k0 = -8, k1 = -1 (two's complement)
    data[0, 1] = 0x71                                     # k2 = 1, k3 = 7
    sc = np.array([[0x4000]], dtype=np.uint16)            # bf16 2.0
    W = F.decode(F.FMT_INT4_G64, data, sc, 1.0, 1, 64)
    assert list(W[0, :4]) == [-16.0, -2.0, 2.0, 14.0]
    d8 = np.zeros((1, 64), dtype=np.uint8)
    d8[0, :3] = [0x81, 0x7F, 0xFF]                         # -127, 127, -1
    W8 = F.decode(F.FMT_INT8_G64, d8, np.array([[0x3F00]], dtype=np.uint16), 1.0, 1, 64)  # 0.5
    assert list(W8[0, :3]) == [-63.5, 63.5, -0.5]


def test_int4_g128_layout_hand_built():
    # unsigned nibbles with zero point 8: byte 0x80 -> k0 = 0 - 8, k1 = 8 - 8; byte 0xF7 -> k2 = -1, k3 = 7;
    # FP16 scale 0x3C00 = 1.0 for the first 128 columns, 0xC000 = -2.0 for the next 128
    data = np.full((1, 128), 0x88, dtype=np.uint8)
    data[0, 0], data[0, 1] = 0x80, 0xF7
    data[0, 64] = 0x9F                                    # k128 = 15 - 8 = 7, k129 = 9 - 8 = 1
    sc = np.array([[0x3C00, 0xC000]], dtype=np.uint16)
    W = F.decode(F.FMT_INT4_G128, data, sc, 1.0, 1, 256)
    assert list(W[0, :4]) == [-8.0, 0.0, -1.0, 7.0]
    assert list(W[0, 128:130]) == [-14.0, -2.0]
    assert np.all(W[0, 4:128] == 0) and np.all(W[0, 130:] == 0)


def test_fp8_b128_layout_hand_built():
    data = np.zeros((256, 128), dtype=np.uint8)
    data[0, 0] = 0x38                                     # 1.0
    data[200, 5] = 0xC0                                   # -2.0
    sc = np.array([[0.25], [3.0]], dtype=np.float32)     # [N/128, K/128]
    W = F.decode(F.FMT_FP8_B128, data, sc, 1.0, 256, 128)
    assert W[0, 0] == 0.25 and W[200, 5] == -6.0
    assert np.count_nonzero(W) == 2


# ------------------------------------------- generator encoders (round trip) ----

@pytest.mark.parametrize("fmt,N,K", [(F.FMT_NVFP4, 8, 64), (F.FMT_MXFP4, 8, 64), (F.FMT_INT4_G64, 8, 128),
                                     (F.FMT_INT8_G64, 8, 128), (F.FMT_FP8_B128, 128, 256),
                                     (F.FMT_INT4_G128, 8, 256)])
def test_quantize_error_bound(fmt, N, K):
    rng = np.random.default_rng(fmt)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    data, scales, ts = synth.quantize(fmt, W)
    D = F.decode(fmt, data, scales, ts, N, K)
    Wd = W.astype(np.float64)
    if fmt == F.FMT_NVFP4:
        s = np.repeat(F.E4M3_TABLE[scales], 16, axis=1) * ts
        y = np.abs(Wd) / s
        # half the E2M1 spacing at y, or the clamp at 6
        spacing = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0))
        err = np.abs(Wd - D) / s
        assert np.all((err <= spacing / 2 + 1e-12) | (y > 6))
        # the block maximum maps to code 6 up to the E4M3 rounding of its scale
        assert np.all(np.abs(D).max() <= 6 * 448 * ts * (1 + 1e-12))
    elif fmt == F.FMT_MXFP4:
        s = np.repeat(F.E8M0_TABLE[scales], 32, axis=1)
        y = np.abs(Wd) / s
        assert np.all(y <= 6)                             # smallest e with 6*2^e >= amax: no clamping
        spacing = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0))
        assert np.all(np.abs(Wd - D) / s <= spacing / 2 + 1e-12)
        blk = np.abs(Wd).reshape(N, K // 32, 32).max(-1)
        assert np.all(6 * F.E8M0_TABLE[scales] / 2 < blk)  # e is the smallest such exponent
    elif fmt in (F.FMT_INT4_G64, F.FMT_INT8_G64):
        s = np.repeat(F.bf16_to_f64(scales), 64, axis=1)
        qmax = 7 if fmt == F.FMT_INT4_G64 else 127
        y = np.abs(Wd) / s
        ok = (np.abs(Wd - D) <= s / 2 * (1 + 1e-12)) | (y > qmax)
        assert np.all(ok)
    elif fmt == F.FMT_INT4_G128:
        # FP16 scale = torch's float16 of amax / 7 per 128 columns; error within half a step or the clamp
        amax = np.abs(Wd).reshape(N, K // 128, 128).max(-1)
        ref = torch.from_numpy(amax / 7.0).to(torch.float16).numpy().view(np.uint16)
        assert np.array_equal(scales, ref)
        s = np.repeat(scales.view(np.float16).astype(np.float64), 128, axis=1)
        ok = (np.abs(Wd - D) <= s / 2 * (1 + 1e-12)) | (np.abs(Wd) / s > 7)
        assert np.all(ok)
    else:
        s = np.repeat(np.repeat(scales.astype(np.float64), 128, 0), 128, 1)
        y = Wd / s
        ref = torch.from_numpy(y.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        # in-range values: generator's RNE equals torch's e4m3 cast (same value)
        inr = np.abs(y) < 448
        assert np.array_equal(D[inr] / s[inr], ref[inr]) or np.allclose(D[inr] / s[inr], ref[inr], rtol=0, atol=0)


@pytest.mark.parametrize("fmt,N,K", [(F.FMT_NVFP4, 4, 64), (F.FMT_MXFP4, 4, 64), (F.FMT_INT4_G64, 4, 128),
                                     (F.FMT_INT8_G64, 4, 128), (F.FMT_FP8_B128, 128, 128)])
def test_quantize_round_trip_on_grid(fmt, N, K):
    """Decoded values re-quantise to the same codes (they are on the grid)."""
    rng = np.random.default_rng(10 + fmt)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    data, scales, ts = synth.quantize(fmt, W)
    D = F.decode(fmt, data, scales, ts, N, K).astype(np.float32)
    if fmt == F.FMT_NVFP4:
        # e2m1 * e4m3 * ts needs up to 30 significant bits, so the fp32 copy is rounded;
        # blocks whose re-derived scale is unchanged must give back the same codes
        d2, s2, ts2 = synth.quantize(fmt, D)
        assert ts2 == ts
        same = np.repeat(s2 == scales, 16, axis=1)
        assert same.mean() > 0.5
        v1 = F.E2M1_TABLE[F.unpack_nibbles(data)]
        v2 = F.E2M1_TABLE[F.unpack_nibbles(d2)]
        assert np.array_equal(v1[same], v2[same])       # same values (a -0 code may come back as +0)
        return
    if fmt == F.FMT_FP8_B128:
        # e4m3 * fp32 scale needs up to 28 significant bits: compare codes' values where s is unchanged
        d2, s2, _ = synth.quantize(fmt, D)
        assert np.array_equal(s2, scales)
        assert np.array_equal(F.E4M3_TABLE[d2], F.E4M3_TABLE[data])
        return
    assert np.array_equal(D.astype(np.float64), F.decode(fmt, data, scales, ts, N, K))  # exact in fp32
    d2, s2, ts2 = synth.quantize(fmt, D)
    # MXFP4 may pick a smaller exponent for a block whose maximum rounded down; values are kept
    if fmt in (F.FMT_INT4_G64, F.FMT_INT8_G64):
        assert np.array_equal(s2, scales)
    assert np.array_equal(F.decode(fmt, d2, s2, ts2, N, K), D.astype(np.float64))


def test_e2m1_encoder_ties_to_even_code():
    # NVFP4 block with scale 1 and ts such that x/(s*ts) hits every E2M1 midpoint
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    expect = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    W = np.zeros((1, 16), dtype=np.float32)
    W[0, 0] = 6.0                                          # amax 6 -> ts = 6/2688, s = e4m3(448) = 448
    W[0, 1:1 + len(mids)] = mids
    W[0, 8] = -5.0
    data, scales, ts = synth.quantize(F.FMT_NVFP4, W)
    assert scales[0, 0] == 0x7E and ts == np.float32(6.0) / np.float32(2688.0)
    D = F.decode(F.FMT_NVFP4, data, scales, 1.0, 1, 16) / 448.0   # back to E2M1 units
    assert D[0, 0] == 6.0
    step = 448.0 * float(ts)
    y = W[0, 1:1 + len(mids)].astype(np.float64) / step
    # the generator divides by s*ts exactly; values are midpoints only up to fp32(ts) rounding,
    # so compare with the nearest-even rule applied to the exact quotients
    ref = F.E2M1_TABLE[F.e2m1_encode_rne(y)]
    assert np.array_equal(D[0, 1:1 + len(mids)], ref)
    # exact midpoints through a power-of-two MXFP4 scale: ties must go to the even code
    Wm = np.zeros((1, 32), dtype=np.float32)
    Wm[0, 0] = 6.0
    Wm[0, 1:1 + len(mids)] = mids
    d, s, _ = synth.quantize(F.FMT_MXFP4, Wm)
    assert s[0, 0] == 127
    Dm = F.decode(F.FMT_MXFP4, d, s, 1.0, 1, 32)
    assert list(Dm[0, 1:1 + len(mids)]) == expect


def test_oracle_e2m1_encoder_brute_force():
    rng = np.random.default_rng(3)
    y = np.concatenate([rng.uniform(-8, 8, 5000), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 7.0, -0.0]])
    codes = F.e2m1_encode_rne(y)
    for v, c in zip(y, codes):
        a = min(abs(v), 6.0)
        d = [abs(a - g) for g in F.E2M1_GRID]
        best = min(d)
        cands = [i for i in range(8) if d[i] == best]
        exp = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
        assert (c & 7) == exp
        assert bool(c & 8) == bool(np.signbit(v))


def test_oracle_e4m3_encoder_matches_torch():
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.uniform(0, 460, 20000), 2.0 ** rng.uniform(-12, 8, 20000),
                        F.E4M3_TABLE[:126] + np.diff(F.E4M3_TABLE[:127]) / 2]).astype(np.float32)
    codes = F.e4m3_encode_rne_sat(v.astype(np.float64))
    inr = v <= 448
    ref = torch.from_numpy(v[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[inr], ref)
    assert np.all(codes[~inr] == 0x7E)                    # saturation
    # negative values, including ones that round to -0 (code 0x80)
    w = -np.concatenate([v[inr][:5000], 2.0 ** rng.uniform(-14, -9, 2000).astype(np.float32)])
    ref_n = torch.from_numpy(w).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode_rne_sat(w.astype(np.float64)), ref_n)
    assert np.any(ref_n == 0x80)


# ------------------------------------------------------ fold-scales lever ----

def _round_frac(x: Fraction, bits: int) -> Fraction:
    """Nearest binary value with `bits` significant bits to x (ties to even), normal range."""
    if x == 0:
        return x
    a = abs(x)
    e = 0
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    while Fraction(2) ** e > a:
        e -= 1
    step = Fraction(2) ** (e - bits + 1)
    lo = (a // step) * step
    hi = lo + step
    if a - lo < hi - a:
        r = lo
    elif hi - a < a - lo:
        r = hi
    else:
        r = lo if (lo / step) % 2 == 0 else hi
    return r if x > 0 else -r


def _fold_ref(code: float, scale: float) -> float:
    """bf16(fl32(code * scale)) by exact rational rounding: 24 significant bits, then 8."""
    return float(_round_frac(_round_frac(Fraction(code) * Fraction(scale), 24), 8))


def _double_rounding_fp8_cases():
    """(E4M3 value, FP32 scale) pairs whose FP32 product lands on a BF16 midpoint that the exact
    product is not on: rounding through FP32 and rounding directly disagree there."""
    out = []
    for j in range(128):
        m = Fraction(1) + Fraction(j, 128) + Fraction(1, 256)          # a BF16 midpoint in [1, 2)
        for c in (1.125, 1.25, 1.375, 1.625, 1.75, 1.875):
            s0 = float(np.float32(float(m / Fraction(c))))
            for k in range(-3, 4):
                s = float(np.nextafter(np.float32(s0), np.float32(np.inf if k > 0 else -np.inf))) if k else s0
                for _ in range(abs(k) - 1):
                    s = float(np.nextafter(np.float32(s), np.float32(np.inf if k > 0 else -np.inf)))
                p = Fraction(c) * Fraction(s)
                if _round_frac(p, 8) != _round_frac(_round_frac(p, 24), 8):
                    out.append((c, s))
    return out


def _fold_cases():
    rng = np.random.default_rng(11)
    f32 = (rng.standard_normal(40) * 0.02).astype(np.float32)
    bf16_scales = [float(v) for v in torch.from_numpy(f32).to(torch.bfloat16).to(torch.float64).numpy()]
    bf16_scales += [2.0 ** -7, 1.0078125, -3.0 * 2.0 ** -9]
    fp16_scales = [float(v) for v in (rng.standard_normal(40) * 0.01).astype(np.float16)] + [2.0 ** -10]
    fp32_scales = [float(v) for v in (rng.standard_normal(20) * 1e-3).astype(np.float32)] + [2.0 ** -8]
    cases = []
    for s in bf16_scales:
        cases += [(F.FMT_INT8_G64, float(q), s) for q in range(-128, 128)]
    for s in fp16_scales:
        cases += [(F.FMT_INT4_G128, float(q), s) for q in range(-8, 8)]
    e4m3 = [float(v) for v in F.E4M3_TABLE if np.isfinite(v)]
    for s in fp32_scales:
        cases += [(F.FMT_FP8_B128, q, s) for q in e4m3]
    cases += [(F.FMT_FP8_B128, c, s) for c, s in _double_rounding_fp8_cases()]
    return cases


_FOLD_CASES = None


def _fold_mismatches(fold_fn) -> int:
    global _FOLD_CASES
    if _FOLD_CASES is None:
        _FOLD_CASES = _fold_cases()
    bad = 0
    for fmt, c, s in _FOLD_CASES:
        got = float(fold_fn(fmt, np.array([c * s]))[0])  # c * s is exact in FP64 for every format here
        bad += got != _fold_ref(c, s)
    return bad


def test_fold_scales_weights_exact_rationals():
    # every code of int8 g64 / int4 g128 / FP8 b128 times sampled scales of the format's scale type,
    # plus constructed FP8 cases where rounding through FP32 and rounding directly disagree
    assert len(_double_rounding_fp8_cases()) > 0
    assert _fold_mismatches(F.fold_scales_weights) == 0


def test_fold_scales_hand_example_and_identity_cases():
    # q = 3 times the BF16 scale 1 + 2^-7: 3.0234375 = 1.1000001|1 x 2^1 rounds up to 3.03125
    assert F.fold_scales_weights(F.FMT_INT8_G64, np.array([3 * 1.0078125]))[0] == 3.03125
    # power-of-two scales: an int8 code has at most 7 significant bits, so the fold is exact
    q = np.arange(-128, 128, dtype=np.float64)
    assert np.array_equal(F.fold_scales_weights(F.FMT_INT8_G64, q * 2.0 ** -7), q * 2.0 ** -7)
    # formats the exact chain already folds exactly are left as decoded
    W = np.array([0.1234567, -3.3e-5, 7.0])
    for fmt in (F.FMT_NVFP4, F.FMT_MXFP4, F.FMT_INT4_G64):
        assert np.array_equal(F.fold_scales_weights(fmt, W), W)


def _fold_truncating(fmt, W):
    if fmt not in F.FOLD_LEVER_FORMATS:
        return W
    b = np.asarray(W, dtype=np.float64).astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    return b.view(np.float32).astype(np.float64)


def _fold_direct(fmt, W):
    return F.round_bf16(W) if fmt in F.FOLD_LEVER_FORMATS else W


def _fold_to_f16(fmt, W):
    # wrong: the folded weight rounded to FP16 (the exact chain's operand type) instead of BF16
    if fmt not in F.FOLD_LEVER_FORMATS:
        return W
    return np.asarray(W, dtype=np.float64).astype(np.float32).astype(np.float16).astype(np.float64)


@pytest.mark.parametrize("planted", [_fold_truncating, _fold_direct, _fold_to_f16])
def test_fold_scales_pin_catches_planted_mistakes(planted):
    assert _fold_mismatches(planted) > 0
