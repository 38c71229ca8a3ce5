"""Pins of the oracle's 16-bit decoders against library conversions and known
encodings (binary16 / bfloat16 definitions)."""

import numpy as np
import torch

from oracle.formats import decode_bits
from workloads import round_to_storage

ALL = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def _same(a, b):
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])


def test_f16_all_patterns_match_numpy():
    ours = decode_bits(ALL, "f16")
    lib = ALL.view(np.float16).astype(np.float64)
    assert _same(ours, lib)


def test_bf16_all_patterns_match_torch():
    ours = decode_bits(ALL, "bf16")
    lib = torch.from_numpy(ALL.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    assert _same(ours, lib)


def test_known_encodings():
    f16 = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0001: 2.0 ** -24, 0x0400: 2.0 ** -14,
           0x3555: 0.333251953125, 0x8000: -0.0}
    bf16 = {0x3F80: 1.0, 0xC040: -3.0, 0x0001: 2.0 ** -133, 0x0080: 2.0 ** -126,
            0x7F7F: 3.3895313892515355e38, 0x3EAB: 0.333984375}
    for bits, val in f16.items():
        assert decode_bits(np.array([bits], np.uint16), "f16")[0] == val
    for bits, val in bf16.items():
        assert decode_bits(np.array([bits], np.uint16), "bf16")[0] == val
    assert np.isinf(decode_bits(np.array([0x7C00], np.uint16), "f16")[0])
    assert np.isnan(decode_bits(np.array([0x7E00], np.uint16), "f16")[0])
    assert np.isnan(decode_bits(np.array([0x7FC0], np.uint16), "bf16")[0])


def test_generator_rounding_is_nearest_even():
    """The input generator's bf16 rounding agrees with torch's float32->bfloat16
    conversion (round-to-nearest-even) on random and tie values."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(100000).astype(np.float32)
    ties = (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, -ties])
    ours = round_to_storage(x, "bf16")
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, lib)
    ours16 = round_to_storage(x[:100000], "f16")
    lib16 = torch.from_numpy(x[:100000]).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours16, lib16)
