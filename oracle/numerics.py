"""Bit-level number formats used by the decoder, written from their definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources
-------
* tinyllm L10.1 "Candle model runner (Llama + bigram, int4), Rust KV cache,
  sampler and PCG32", section 2.3 "The model directory": bf16 widens by
  placing the 16 bits above 16 zero bits; f16 decodes as
  (-1)^s 2^(e-15) (1 + m/1024) for 0 < e < 31 and (-1)^s 2^-14 m/1024 for
  e = 0; f32 -> f16 keeps the top 10 mantissa bits and rounds to nearest,
  ties to even.
* same page, section 3 "Worked example by hand", f16 rounding: 1 + 2^-11
  rounds to 0x3C00 and 1 + 3*2^-11 to 0x3C02.

Everything here works on integers so that no library rounding routine is
involved; the tests compare the results against numpy's and torch's own
conversions as an independent check.
"""

from __future__ import annotations

import numpy as np


def bf16_round(x) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); return float32.

    bfloat16 is the upper half of a float32.  Rounding to nearest-even adds
    0x7FFF plus the lowest kept bit, then clears the 16 dropped bits.  NaNs
    keep their sign and become a quiet NaN; infinities pass through.
    """
    shape = np.shape(x)
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).reshape(-1)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = ((u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)).astype(np.uint32)
    is_nan = np.isnan(a)
    rounded = np.where(is_nan, (a.view(np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x00400000), rounded)
    return rounded.astype(np.uint32).view(np.float32).reshape(shape)


def bf16_bits(x) -> np.ndarray:
    """The 16-bit bfloat16 pattern of ``bf16_round(x)``."""
    return (bf16_round(x).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def f32_to_f16_bits(x) -> np.ndarray:
    """float32 -> IEEE binary16 bit pattern, round to nearest, ties to even.

    Handles normal results, gradual underflow into subnormals, overflow to
    infinity and NaN.  Written on the integer fields: the float32 value is
    sign s, biased exponent E (bias 127) and 23-bit fraction F.
    """
    shape = np.shape(x)
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).reshape(-1)
    u = a.view(np.uint32).astype(np.int64)
    sign = ((u >> 31) & 1) << 15
    exp = (u >> 23) & 0xFF
    frac = u & 0x7FFFFF
    out = np.zeros(u.shape, dtype=np.int64)

    nan = (exp == 0xFF) & (frac != 0)
    inf = (exp == 0xFF) & (frac == 0)
    finite = exp != 0xFF

    # Unbiased exponent of the float32 value; float32 subnormals (exp == 0)
    # are far below the smallest f16 subnormal and round to signed zero.
    e = exp - 127
    mant = frac | (1 << 23)  # 24-bit significand with the hidden one

    # Normal f16 range: e in [-14, 15].  Keep 10 fraction bits, drop 13.
    normal = finite & (exp != 0) & (e >= -14)
    drop = 13
    kept = mant >> drop
    rem = mant & ((1 << drop) - 1)
    half = 1 << (drop - 1)
    up = (rem > half) | ((rem == half) & ((kept & 1) == 1))
    kept_r = kept + up.astype(np.int64)
    # kept_r is in [1024, 2048]; 2048 means the significand carried over.
    carry = kept_r >> 11
    e_r = e + carry
    kept_r = np.where(carry == 1, kept_r >> 1, kept_r)
    biased = e_r + 15
    normal_bits = (biased << 10) | (kept_r & 0x3FF)
    normal_bits = np.where(biased >= 31, 0x7C00, normal_bits)  # overflow -> inf
    out = np.where(normal, normal_bits, out)

    # Subnormal f16 range: value = k * 2^-24 with k in [0, 1024]. The float32
    # significand is mant * 2^(e-23), so k = mant * 2^(e+1); shift right by
    # -(e+1) and round to nearest even.  k == 1024 is the smallest normal.
    sub = finite & (exp != 0) & (e < -14)
    shift = np.clip(-(e + 1), 0, 63)
    big = shift >= 25  # everything is dropped and the remainder < half
    sh = np.where(big, 0, shift)
    k = mant >> sh
    rem_s = mant - (k << sh)
    half_s = np.where(sh > 0, 1 << np.maximum(sh - 1, 0), 0)
    up_s = (sh > 0) & ((rem_s > half_s) | ((rem_s == half_s) & ((k & 1) == 1)))
    k = k + up_s.astype(np.int64)
    k = np.where(big, 0, k)
    out = np.where(sub, k, out)  # k == 1024 encodes 0x0400, the smallest normal

    out = np.where(inf, 0x7C00, out)
    out = np.where(nan, 0x7E00 | ((frac >> 13) & 0x1FF), out)
    out = out | sign
    return out.astype(np.uint16).reshape(shape)


def f16_bits_to_f32(h) -> np.ndarray:
    """IEEE binary16 bit pattern -> float32, exactly, from the decoding formula."""
    b = np.asarray(h, dtype=np.uint16).astype(np.int64)
    s = (b >> 15) & 1
    e = (b >> 10) & 0x1F
    m = b & 0x3FF
    sgn = np.where(s == 1, -1.0, 1.0)
    with np.errstate(over="ignore", invalid="ignore"):
        normal = sgn * np.ldexp(1.0 + m / 1024.0, (e - 15).astype(np.int32))
        sub = sgn * np.ldexp(m / 1024.0, -14)
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 31) & (m == 0), sgn * np.inf, val)
    val = np.where((e == 31) & (m != 0), np.nan, val)
    return val.astype(np.float32)


def f16_round(x) -> np.ndarray:
    """float32 -> nearest f16 value, widened back to float32."""
    return f16_bits_to_f32(f32_to_f16_bits(x))
