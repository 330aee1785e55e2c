"""Scalar number formats of the compressed FP4 KV cache, written from their definitions.

TEST INFRASTRUCTURE. This package is the CPU oracle that the CUDA path is checked
against. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and its ``--impl reference`` arm) may import it. The product
path never does, and this package imports nothing from the product.

Formats named by the pages ("DeepSeek-V4.1-Flash: le cache KV en FP4",
sections "Cache principal" and "Cles d'indexeur"):

* E2M1 (FP4): 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit, no
  infinity and no NaN. Magnitudes by 3-bit code: 0, 0.5, 1, 1.5, 2, 3, 4, 6.
  Bit 3 of a code is the sign.
* E4M3 ("float8_e4m3fn", the ``scale_dtype`` of the quantiser call on the same
  page): 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinity,
  NaN = S.1111.111, largest finite value 448, smallest subnormal 2**-9.
* E8M0 (the MX block-scale format): 8-bit biased exponent, value 2**(e-127),
  0xFF is NaN.

Readings where the pages are silent:
* Rounding is round-to-nearest, ties to the code with an even mantissa bit
  (IEEE round-half-even applied to the target grid), saturating to the largest
  finite magnitude ("satfinite").
* The sign of an input that rounds to zero is kept (a small negative value
  encodes as E2M1 code 0x8), as an IEEE conversion would do.

Every function here works on numpy arrays and is vectorised only over
independent elements; each element follows the definition directly.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------- E2M1 (FP4)
#: magnitude of each 3-bit E2M1 code 0..7 (sign is bit 3 of the 4-bit code)
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def e2m1_value(exp_bits: int, man_bit: int) -> float:
    """Value of an E2M1 magnitude from its fields (bias 1; exponent 0 is subnormal)."""
    if exp_bits == 0:
        return man_bit * 0.5
    return 2.0 ** (exp_bits - 1) * (1.0 + man_bit / 2.0)


def e2m1_decode(codes) -> np.ndarray:
    """4-bit E2M1 codes (0..15, any integer dtype) -> float64 values."""
    c = np.asarray(codes).astype(np.int64)
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where((c & 8) != 0, -mag, mag)


def e2m1_encode(v) -> np.ndarray:
    """Round each value to the nearest E2M1 number, ties to even mantissa, saturating.

    ``v`` holds finite float32 or float64 values; the comparison against the eight
    magnitudes is done in float64, where the differences are exact for these inputs.
    Returns uint8 codes 0..15.
    """
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("E2M1 encode: non-finite input")
    a = np.minimum(np.abs(v), 6.0)                        # satfinite: clamp, then round
    d = np.abs(a[..., None] - E2M1_MAGNITUDES)          # distance to each magnitude
    dmin = d.min(axis=-1, keepdims=True)
    nearest = d == dmin                                   # one or two candidates
    # among the nearest candidates prefer an even mantissa bit (code & 1 == 0)
    even = (np.arange(8) & 1) == 0
    pick_even = nearest & even
    has_even = pick_even.any(axis=-1, keepdims=True)
    choice = np.where(has_even, pick_even, nearest)
    mag_code = np.argmax(choice, axis=-1).astype(np.uint8)
    sign = np.signbit(v).astype(np.uint8) << 3
    return (mag_code | sign).astype(np.uint8)


# ---------------------------------------------------------------- E4M3 (fn)
def e4m3_decode(codes) -> np.ndarray:
    """8-bit float8_e4m3fn codes -> float64 (NaN for S.1111.111)."""
    c = np.asarray(codes).astype(np.int64)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where((c & 0x80) != 0, -mag, mag)


#: the 127 non-negative finite E4M3 values, indexed by code 0x00..0x7E
_E4M3_POS = e4m3_decode(np.arange(0x7F))


def e4m3_encode(v) -> np.ndarray:
    """Round to the nearest finite E4M3 value, ties to even mantissa, saturating at 448.

    Inputs are finite float32/float64 values; distances are computed in float64,
    exact for float32 inputs against these 4-significant-bit grid points.
    """
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("E4M3 encode: non-finite input")
    a = np.minimum(np.abs(v), 448.0)                     # satfinite
    d = np.abs(a[..., None] - _E4M3_POS)
    dmin = d.min(axis=-1, keepdims=True)
    nearest = d == dmin
    even = (np.arange(0x7F) & 1) == 0
    pick_even = nearest & even
    has_even = pick_even.any(axis=-1, keepdims=True)
    choice = np.where(has_even, pick_even, nearest)
    code = np.argmax(choice, axis=-1).astype(np.uint8)
    sign = np.signbit(v).astype(np.uint8) << 7
    return (code | sign).astype(np.uint8)


# ---------------------------------------------------------------- E8M0
def e8m0_decode(codes) -> np.ndarray:
    """8-bit E8M0 codes -> float64 powers of two (NaN for 0xFF)."""
    c = np.asarray(codes).astype(np.int64)
    return np.where(c == 255, np.nan, np.exp2(c - 127.0))


def floor_log2(a) -> np.ndarray:
    """floor(log2(a)) for positive finite a, from the exact binary exponent (frexp)."""
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)                                    # a = m * 2**e, m in [0.5, 1)
    return e.astype(np.int64) - 1


# ---------------------------------------------------------------- bf16 helper
def bf16_bits_to_float(bits) -> np.ndarray:
    """Raw bfloat16 bit patterns (uint16) -> float64, exactly."""
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
