"""MX (OCP Microscaling) element and scale rules in fp64 -- oracle, test infrastructure only.

Source of the format: [S2.1] "FP8 Quantization Strategy" names the mxfp8 recipe
as 1x32 blocks with OCP UE8M0 shared exponents (32-element shared exponents,
the OCP MX standard) and E4M3 elements; the steps the pages leave open follow
the OCP MX v1.0 specification:

1. per block of 32 consecutive elements along K: amax = max |v_i|;
2. shared exponent s = floor(log2(amax)) - emax(E4M3), emax(E4M3) = 8,
   clamped to the UE8M0 range [-127, 127]; the scale byte is s + 127;
3. elements q_i = E4M3(v_i / 2^s), round to nearest even, values above the
   largest finite E4M3 (448) saturate to +-448 (never NaN).

Readings where the spec leaves room:
* all-zero block -> s = -127 (scale byte 0x00), elements 0x00 / 0x80 by sign;
* the sign of zero is kept (-0 and negative values rounding to 0 give 0x80);
* E4M3 subnormals are m * 2^-9, m = 1..7, reached by the same RNE rule;
* NaN/Inf inputs are outside the tested domain.

Scaling by 2^-s is exact in fp64, so each element is rounded exactly once.
"""
from __future__ import annotations

import numpy as np

BLOCK = 32
E4M3_MAX = 448.0
E4M3_EMAX = 8      # 448 = 1.75 * 2^8
E4M3_EMIN = -6     # smallest normal exponent; below it the spacing stays 2^-9
E4M3_MBITS = 3
UE8M0_BIAS = 127


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(v) -> np.ndarray:
    """fp64 -> bf16 bit patterns, one rounding: nearest, ties to even.

    bf16 keeps 8 significant bits; its smallest normal exponent is -126 and its
    subnormal spacing 2^-133. Magnitudes that round to 2^128 or above become inf.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)
    e = np.maximum(ex - 1, -126)
    quantum = np.ldexp(1.0, e - 7)
    r = np.rint(a / quantum) * quantum
    r = np.where(r >= 2.0 ** 128, np.inf, r)
    r = np.copysign(r, v).astype(np.float32)          # exact: r has <= 8 significant bits
    out = (r.view(np.uint32) >> 16).astype(np.uint16)
    return np.where(np.isnan(v), np.uint16(0x7FC0), out)


def e4m3_value(code) -> np.ndarray:
    """Closed-form value of an E4M3 byte: sign bit, 4-bit exponent (bias 7),
    3-bit mantissa; exponent field 0 is subnormal (m * 2^-9); 0x7F/0xFF are NaN."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(v) -> np.ndarray:
    """fp64 -> E4M3 byte, round to nearest (ties to even), saturating at +-448."""
    v = np.asarray(v, dtype=np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    _, ex = np.frexp(a)
    e = np.maximum(ex - 1, E4M3_EMIN)
    quantum = np.ldexp(1.0, e - E4M3_MBITS)
    r = np.rint(a / quantum) * quantum              # a / quantum is exact (power of two)
    r = np.minimum(r, E4M3_MAX)
    # encode the representable magnitude r
    _, rex = np.frexp(np.where(r > 0, r, 1.0))
    re = rex - 1
    sub = r < 2.0 ** E4M3_EMIN
    mant_sub = np.rint(r / 2.0 ** -9)
    mant_norm = np.rint(r / np.ldexp(1.0, re - E4M3_MBITS)) - 8
    code = np.where(sub, mant_sub, (re + 7) * 8 + mant_norm)
    code = code.astype(np.int64) | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)


def shared_exponent(amax) -> np.ndarray:
    """UE8M0 shared exponent s (unbiased) of a block with the given amax."""
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)                         # amax = f * 2^ex, f in [0.5, 1)
    s = np.clip(ex - 1 - E4M3_EMAX, -UE8M0_BIAS, UE8M0_BIAS)
    return np.where(amax == 0, -UE8M0_BIAS, s).astype(np.int64)


def mx_quantize(x):
    """MX-quantise along the last axis (blocks of 32). Returns (q uint8 [..., K],
    scale bytes uint8 [..., K/32])."""
    x = np.asarray(x, dtype=np.float64)
    K = x.shape[-1]
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    blk = x.reshape(*x.shape[:-1], K // BLOCK, BLOCK)
    amax = np.max(np.abs(blk), axis=-1)
    s = shared_exponent(amax)
    q = e4m3_encode(blk * np.exp2(-s.astype(np.float64))[..., None])
    return q.reshape(x.shape), (s + UE8M0_BIAS).astype(np.uint8)


def scale_value(sbyte) -> np.ndarray:
    """UE8M0 byte -> 2^(b - 127) (0xFF is NaN)."""
    b = np.asarray(sbyte, dtype=np.int64)
    return np.where(b == 255, np.nan, np.exp2(b - 127.0))


def mx_dequantize(q, sbytes) -> np.ndarray:
    """Exact fp64 values E4M3(q_i) * 2^s of an MX tensor."""
    q = np.asarray(q, dtype=np.uint8)
    K = q.shape[-1]
    v = e4m3_value(q).reshape(*q.shape[:-1], K // BLOCK, BLOCK)
    return (v * scale_value(sbytes)[..., None]).reshape(q.shape)
