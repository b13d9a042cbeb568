"""FP8 (E4M3) storage of cached keys and values for the H2O oracle.

TEST INFRASTRUCTURE, like the rest of this package: only the tests, the smoke
check and the benchmark's CPU leg use it, and it shares no code with the CUDA
path.

The pages say that H2O combines with quantisation of the KV cache and that the
combination beats either alone ([H2O] section 5), but fix no scheme. The
reading used here, for a cache whose slots hold single tokens:

  * every cached token's key vector and value vector are stored separately as
    E4M3 codes with one fp32 scale each;
  * scale = amax / 448 with amax = max_i |x_i| (448 is E4M3's largest finite
    value), and code_i = E4M3(x_i * (448 / amax)), rounded to the nearest
    representable value with ties to even and saturated to +-448; a zero
    vector has scale 0 and zero codes;
  * the stored token is the dequantised vector E4M3^-1(code_i) * scale, and it
    is what every later step attends to -- the new token of a decode step
    included, because it is appended to the cache before the attention;
  * prefill attention runs on the full-precision prompt; the retained tokens
    are quantised when they enter the cache.

The scale arithmetic is fp32 with IEEE round-to-nearest, one rounding per
operation (448 / amax, x * that, amax / 448), as the kernel does, so the codes
and scales are identical on both sides. E4M3 (OCP 8-bit Floating Point
Specification, OFP8, v1.0): 1 sign bit, 4 exponent bits with bias 7, 3
mantissa bits; exponent field 0 holds subnormals m * 2^-9; S.1111.111 is NaN
and there are no infinities, so the largest finite value is 1.75 * 2^8 = 448.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Values (float64) of E4M3 codes (uint8); NaN for the two NaN codes."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """E4M3 codes (uint8) of fp32 values: round to nearest, ties to even,
    saturating to +-448. The sign of zero is kept."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    sign = np.signbit(x).astype(np.uint8) << 7
    a = np.abs(x)
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6  # subnormal range: steps of 2^-9
    m_sub = np.rint(a / 2.0 ** -9)  # 0 .. 8; 8 is the smallest normal (code 8)
    code = np.where(sub, m_sub.astype(np.int64), code)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(sub, 1.0, a)))
    e = np.clip(e, -6, 8)
    q = np.rint(a / np.exp2(e - 3))  # 8 .. 16 for normal values
    carry = q >= 16
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 8, q)
    normal = ((e + 7).astype(np.int64) << 3) | (q.astype(np.int64) - 8)
    code = np.where(sub, code, normal)
    code = np.where(a >= E4M3_MAX, 0x7E, code)  # saturate (also covers 448 < a)
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def quantize_vector(x):
    """(codes uint8 [d], scale float32) of one token vector (bf16 values)."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0)
    if amax == 0:
        return np.zeros(x32.shape, dtype=np.uint8), np.float32(0)
    inv = np.float32(E4M3_MAX) / amax           # one fp32 rounding
    y = (x32 * inv).astype(np.float32)          # one fp32 rounding per element
    scale = amax / np.float32(E4M3_MAX)         # one fp32 rounding
    return e4m3_encode(y), np.float32(scale)


def dequantize_vector(codes, scale) -> np.ndarray:
    """The stored token: code values times the scale (exact in float64)."""
    return e4m3_decode(codes) * np.float64(scale)


def roundtrip(x) -> np.ndarray:
    """x quantised and dequantised (float64)."""
    codes, scale = quantize_vector(x)
    return dequantize_vector(codes, scale)
