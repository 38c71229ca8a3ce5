"""16-bit storage formats decoded to float64 (oracle; test infrastructure only).

Both decoders are written from the formats' definitions, not through a
library's float16/bfloat16 type, so that the test that compares them with
library conversions is an independent check.

* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
  e = 0 is zero/subnormal (value 2^-14 * f/1024), e = 31 is inf/NaN,
  otherwise 2^(e-15) * (1 + f/1024).
* bfloat16: the upper 16 bits of an IEEE 754 binary32 encoding
  (1 sign, 8 exponent bits with bias 127, 7 fraction bits).

Every binary16 and bfloat16 value is exactly representable in float64, so
decoding is exact.
"""

import numpy as np


def decode_f16(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = (b & 0x3FF).astype(np.float64)
    normal = np.ldexp(1.0 + f / 1024.0, (e - 15).astype(np.int64))
    sub = np.ldexp(f / 1024.0, -14)
    special = np.where(f == 0.0, np.inf, np.nan)
    mag = np.where(e == 0, sub, np.where(e == 31, special, normal))
    return sign * mag


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    e = (b >> 7) & 0xFF
    f = (b & 0x7F).astype(np.float64)
    normal = np.ldexp(1.0 + f / 128.0, (e - 127).astype(np.int64))
    sub = np.ldexp(f / 128.0, -126)
    special = np.where(f == 0.0, np.inf, np.nan)
    mag = np.where(e == 0, sub, np.where(e == 255, special, normal))
    return sign * mag


def decode_bits(bits: np.ndarray, dtype: str) -> np.ndarray:
    """uint16 bit patterns of ``dtype`` ("f16" or "bf16") -> float64, same shape."""
    if dtype == "f16":
        return decode_f16(bits)
    if dtype == "bf16":
        return decode_bf16(bits)
    raise ValueError(f"unknown dtype {dtype!r}")
