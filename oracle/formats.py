"""Exact decoders of the checkpoint weight formats (oracle; test infrastructure).

Each decoder maps stored codes to their exact real values in FP64.  The code
tables are written from the format definitions:

* E2M1 (FP4): 1 sign, 2 exponent bits with bias 1, 1 mantissa bit, with a
  subnormal at exponent 0; no Inf or NaN (OCP Microscaling Formats v1.0).
* E4M3 (FP8, "fn" variant): 1 sign, 4 exponent bits with bias 7, 3 mantissa
  bits, subnormals m * 2^-9, the all-ones pattern S.1111.111 is NaN, no Inf
  (OCP 8-bit Floating Point Specification).
* E8M0: unsigned power of two 2^(c - 127); 255 is NaN (OCP MX v1.0).
* BF16: the top 16 bits of an IEEE binary32.

Checkpoint layouts (the DGPP pages serve these formats as published, page 1
README intro "Serves checkpoints as published"; page 4 forum post 1
quantisation table):

* NVFP4:    data [N, K/2] u8, two E2M1 codes per byte, low nibble = even k;
            scales [N, K/16] E4M3 (one per 16-element block); FP32 tensor scale.
            W = e2m1 * e4m3 * ts.
* MXFP4:    data as NVFP4; scales [N, K/32] E8M0.  W = e2m1 * 2^(c-127).
* INT4 g64: data as NVFP4 but two's-complement nibbles; scales [N, K/64]
            BF16.  W = q * s.
* INT8 g64: data [N, K] i8; scales [N, K/64] BF16.  W = q * s.
* FP8 b128: data [N, K] E4M3; scales [N/128, K/128] FP32.  W = q * s.
"""
from __future__ import annotations

import numpy as np

FMT_NVFP4, FMT_MXFP4, FMT_INT4_G64, FMT_INT8_G64, FMT_FP8_B128, FMT_INT4_G128 = 1, 2, 3, 4, 5, 6


def e2m1_value(code: int) -> float:
    """Exact value of one E2M1 code 0..15."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return -mag if s else mag


def e4m3_value(code: int) -> float:
    """Exact value of one E4M3 ("fn") code 0..255; NaN for S.1111.111."""
    s = (code >> 7) & 1
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return float("nan")
    mag = m * 2.0 ** -9 if e == 0 else 2.0 ** (e - 7) * (1.0 + m / 8.0)
    return -mag if s else mag


def e8m0_value(code: int) -> float:
    """Exact value of one E8M0 code 0..255; NaN for 255."""
    if code == 255:
        return float("nan")
    return 2.0 ** (code - 127)


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
E8M0_TABLE = np.array([e8m0_value(c) for c in range(256)], dtype=np.float64)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) -> exact FP64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """FP64 -> BF16 bit patterns with ONE round-to-nearest-even (no double rounding).

    BF16 keeps 8 significant bits and the binary32 exponent range; results
    above the largest finite BF16 after rounding become Inf.
    """
    a = np.asarray(a, dtype=np.float64)
    out = np.zeros(a.shape, dtype=np.uint16)
    sign = np.signbit(a)
    mag = np.abs(a)
    nan = np.isnan(a)
    fin = np.isfinite(a) & (mag > 0)
    m, e = np.frexp(np.where(fin, mag, 1.0))          # mag = m * 2^e, m in [0.5, 1)
    q = e - 8                                          # spacing of 8 significant bits
    q = np.where(e - 1 < -126, -133, q)                # subnormal spacing 2^-133
    r = np.rint(np.ldexp(np.where(fin, mag, 0.0), -q))  # ties to even
    v = np.ldexp(r, q)
    big = v > float(np.float32(3.3895313892515355e38))  # largest finite bf16
    v32 = v.astype(np.float32)                         # exact for representable values
    bits = (v32.view(np.uint32) >> 16).astype(np.uint16)
    out = np.where(fin & ~big, bits, out)
    out = np.where(fin & big, np.uint16(0x7F80), out)
    out = np.where(np.isinf(a), np.uint16(0x7F80), out)
    out = np.where(sign & ~nan, out | np.uint16(0x8000), out)
    out = np.where(nan, np.uint16(0x7FC0), out)
    return out.astype(np.uint16)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """FP64 -> nearest BF16 value (single RNE), returned as FP64."""
    return bf16_to_f64(f64_to_bf16_bits(a))


def unpack_nibbles(data: np.ndarray) -> np.ndarray:
    """[.., K/2] u8 -> [.., K] codes 0..15; the low nibble holds the even k."""
    d = np.asarray(data, dtype=np.uint8)
    out = np.empty(d.shape[:-1] + (d.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = d & 0x0F
    out[..., 1::2] = d >> 4
    return out


def decode(fmt: int, data: np.ndarray, scales: np.ndarray, ts: float, N: int, K: int) -> np.ndarray:
    """Decode one matrix W[N, K] to exact FP64 values."""
    if fmt == FMT_NVFP4:
        v = E2M1_TABLE[unpack_nibbles(data).reshape(N, K)]
        s = E4M3_TABLE[np.asarray(scales, dtype=np.uint8).reshape(N, K // 16)]
        return v * np.repeat(s, 16, axis=1) * float(ts)
    if fmt == FMT_MXFP4:
        v = E2M1_TABLE[unpack_nibbles(data).reshape(N, K)]
        s = E8M0_TABLE[np.asarray(scales, dtype=np.uint8).reshape(N, K // 32)]
        return v * np.repeat(s, 32, axis=1)
    if fmt == FMT_INT4_G64:
        nib = unpack_nibbles(data).reshape(N, K).astype(np.int16)
        q = np.where(nib >= 8, nib - 16, nib).astype(np.float64)
        s = bf16_to_f64(np.asarray(scales, dtype=np.uint16).reshape(N, K // 64))
        return q * np.repeat(s, 64, axis=1)
    if fmt == FMT_INT8_G64:
        q = np.asarray(data, dtype=np.uint8).reshape(N, K).view(np.int8).astype(np.float64)
        s = bf16_to_f64(np.asarray(scales, dtype=np.uint16).reshape(N, K // 64))
        return q * np.repeat(s, 64, axis=1)
    if fmt == FMT_INT4_G128:
        # AutoRound / GPTQ layout (page 2 README "Highlights": int4 group-128 experts served in their
        # packed form): unsigned nibble u with zero point 8, q = u - 8; FP16 scale per 128 columns
        q = unpack_nibbles(data).reshape(N, K).astype(np.float64) - 8.0
        s = np.asarray(scales, dtype=np.uint16).reshape(N, K // 128).view(np.float16).astype(np.float64)
        return q * np.repeat(s, 128, axis=1)
    if fmt == FMT_FP8_B128:
        q = E4M3_TABLE[np.asarray(data, dtype=np.uint8).reshape(N, K)]
        s = np.asarray(scales, dtype=np.float32).reshape(N // 128, K // 128).astype(np.float64)
        return q * np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)
    raise ValueError(f"unknown format {fmt}")


def decode_qmat(qm, e: int = 0) -> np.ndarray:
    """Decode expert e of a synth.QMat stack."""
    return decode(qm.fmt, qm.data[e], qm.scales[e], float(qm.ts[e]), qm.N, qm.K)


# Formats whose group scale the fold-scales lever folds into BF16 weights.
FOLD_LEVER_FORMATS = (FMT_INT8_G64, FMT_FP8_B128, FMT_INT4_G128)


def fold_scales_weights(fmt: int, W: np.ndarray) -> np.ndarray:
    """The fold-scales lever's weight values from the exact decode W = code * scale.

    DGPP README "Execution and performance" table, row engine.prefill_fold_scales:
    each group's scale is folded into the BF16 weight values, and one FP32
    accumulator runs across K (Marlin's form, no per-group FMA).  Reading:
    the product is taken in FP32, as a kernel computes code * scale, and is
    then rounded to BF16 (nearest, ties to even).  For int8 g64 and int4 g128
    the FP32 product is exact (at most 8 + 11 significant bits); for FP8 b128
    (E4M3 times an FP32 scale) it is the FP32 rounding of the exact product.
    The other formats (NVFP4, MXFP4, int4 g64) already reach the exact
    chain's MMA with their scales folded exactly, so the lever leaves them as
    decoded.
    """
    if fmt not in FOLD_LEVER_FORMATS:
        return W
    return round_bf16(np.asarray(W, dtype=np.float64).astype(np.float32).astype(np.float64))


def decode_qmat_fold(qm, e: int = 0) -> np.ndarray:
    """Expert e of a synth.QMat stack as the fold-scales lever's weights."""
    return fold_scales_weights(qm.fmt, decode_qmat(qm, e))


# ---- encoders used by the W4A4 activation quantizer (the layer's own arithmetic) ----

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_encode_rne(y: np.ndarray) -> np.ndarray:
    """Nearest E2M1 code, ties to the even code, saturating at +-6.

    The sign bit is the sign bit of y (IEEE signbit), so values that round to
    zero keep their sign as the -0 code 8.
    """
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), 6.0)
    d = np.abs(a[..., None] - E2M1_GRID)              # distance to each grid point
    best = d.min(axis=-1, keepdims=True)
    cand = d == best                                   # one or two nearest codes
    even = cand & (np.arange(8) % 2 == 0)
    code = np.where(even.any(axis=-1), even.argmax(axis=-1), cand.argmax(axis=-1)).astype(np.uint8)
    return np.where(np.signbit(y), code | 8, code).astype(np.uint8)


def e4m3_encode_rne_sat(y: np.ndarray) -> np.ndarray:
    """Nearest E4M3 code (ties to even mantissa), saturating at +-448.

    The sign bit is the sign bit of y (IEEE signbit), so a negative value that
    rounds to zero is the -0 code 0x80, as in the IEEE conversions.
    """
    y = np.asarray(y, dtype=np.float64)
    pos = E4M3_TABLE[:127]                             # codes 0..126: 0 .. 448, increasing
    a = np.minimum(np.abs(y), 448.0)
    idx = np.searchsorted(pos, a)                      # pos[idx-1] < a <= pos[idx]
    idx = np.clip(idx, 1, 126)
    lo, hi = pos[idx - 1], pos[idx]
    pick_hi = (hi - a < a - lo) | ((hi - a == a - lo) & (idx % 2 == 0))
    code = np.where(a == hi, idx, np.where(pick_hi, idx, idx - 1)).astype(np.uint8)
    code = np.where(a == 0.0, 0, code).astype(np.uint8)
    return np.where(np.signbit(y), code | 0x80, code).astype(np.uint8)
