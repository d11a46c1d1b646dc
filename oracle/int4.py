"""Int4 group-symmetric weights, written out from their definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: tinyllm L10.1 "Candle model runner (Llama + bigram, int4), Rust KV
cache, sampler and PCG32", section 2.5 "Int4 weights": a linear weight W
(out x in) with groups of g consecutive input columns stores, per group, one
f16 scale s = f16(max|W_group| / 7) and g four-bit integers
q = clamp(rint(W / s), -8, 7), rint rounding half to even and s being the
f16 value actually stored, so |W - q s| <= s / 2; the effective weight is
q s.  Two values share a byte: column 2b in the low nibble, column 2b + 1 in
the high nibble, each in 4-bit two's complement.  Section 3 works one group
by hand (int4_hand_example).

Readings where the pages leave a step open:
* The quantizer runs in float32, as the runner quantizes f32 weights at
  load: max|W|/7 is an f32 division rounded once to f16 (nearest, ties to
  even), W/s an f32 division, then rint.
* A group whose weights are all zero has s = 0; its codes are 0 (0/0 is
  read as 0).
"""

from __future__ import annotations

import numpy as np

from .numerics import f16_bits_to_f32, f32_to_f16_bits

GROUP = 32


def quantize(W, group: int = GROUP):
    """(codes int8 [out, in], scale bits uint16 [out, in/group]) of a float32 matrix."""
    W = np.asarray(W, dtype=np.float32)
    out, inn = W.shape
    if inn % group:
        raise ValueError("in-features must be a multiple of the group")
    Wg = W.reshape(out, inn // group, group)
    amax = np.abs(Wg).max(axis=2)                         # float32, exact
    s_bits = f32_to_f16_bits(amax / np.float32(7.0))       # f32 division, one rounding to f16
    s = f16_bits_to_f32(s_bits).astype(np.float32)         # the stored value
    with np.errstate(invalid="ignore", divide="ignore"):
        r = Wg / s[:, :, None]                             # f32 division
    r = np.where(s[:, :, None] == 0, np.float32(0.0), r)
    q = np.clip(np.rint(r), -8, 7).astype(np.int8)         # numpy rint: half to even
    return q.reshape(out, inn), s_bits


def dequantize(q, s_bits, group: int = GROUP) -> np.ndarray:
    """The effective weight q * s, float64 (exact: a 4-bit integer times an f16)."""
    q = np.asarray(q, dtype=np.float64)
    out, inn = q.shape
    s = f16_bits_to_f32(np.asarray(s_bits)).astype(np.float64)
    return (q.reshape(out, inn // group, group) * s[:, :, None]).reshape(out, inn)


def pack(q) -> np.ndarray:
    """Two codes per byte: column 2b in the low nibble, 2b + 1 in the high one."""
    q = np.asarray(q, dtype=np.int8)
    lo = q[:, 0::2].astype(np.uint8) & 0x0F
    hi = q[:, 1::2].astype(np.uint8) & 0x0F
    return (lo | (hi << 4)).astype(np.uint8)


def unpack(b) -> np.ndarray:
    """Codes back from packed bytes (4-bit two's complement)."""
    b = np.asarray(b, dtype=np.uint8)
    lo = (b & 0x0F).astype(np.int8)
    hi = (b >> 4).astype(np.int8)
    lo = np.where(lo > 7, lo - 16, lo).astype(np.int8)
    hi = np.where(hi > 7, hi - 16, hi).astype(np.int8)
    out = np.empty((b.shape[0], b.shape[1] * 2), dtype=np.int8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def effective(W, group: int = GROUP) -> np.ndarray:
    """The weight an int4 model computes with: dequantize(quantize(W))."""
    q, s = quantize(W, group)
    return dequantize(q, s, group)
