"""Pins for the oracle's E4M3 (FP8) KV quantisation."""
import os

import numpy as np
import pytest
import torch

from oracle import fp8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp8_e4m3.txt")


def _fixture():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            c, v = line.split()
            rows.append((int(c, 16), float(v)))
    return rows


def test_worked_codes():
    for code, val in _fixture():
        assert fp8.decode(np.uint8(code)) == val
        assert fp8.encode(val) == code or val == 0.0


def test_nan_codes():
    assert np.isnan(fp8.decode(np.uint8(0x7F))) and np.isnan(fp8.decode(np.uint8(0xFF)))
    assert fp8.encode(float("nan")) & 0x7F == 0x7F


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    vals = fp8.decode(codes)
    back = fp8.encode(vals)
    # +0 and -0 both decode to a zero; everything else maps back to itself
    nz = vals != 0
    np.testing.assert_array_equal(back[nz], codes[nz])


def test_value_grid_is_monotone_and_spaced_by_format():
    v = fp8.decode(np.arange(0, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)
    # within a binade the spacing is 2^(e-10); subnormal spacing 2^-9
    assert np.allclose(np.diff(v[:9]), 2.0 ** -9)
    assert np.allclose(np.diff(v[0x38:0x40]), 2.0 ** -3)


def test_round_to_nearest_ties_to_even_and_saturation():
    assert fp8.encode(1.0625) == 0x38          # halfway 1.0 / 1.125 -> even mantissa
    assert fp8.encode(1.1875) == 0x3A          # halfway 1.125 / 1.25 -> 1.25 (even)
    assert fp8.encode(1.07) == 0x39
    assert fp8.encode(2.0 ** -10) == 0x00      # halfway 0 / 2^-9 -> 0 (even)
    assert fp8.encode(3 * 2.0 ** -10) == 0x02  # halfway 2^-9 / 2^-8 -> 2^-8
    assert fp8.encode(460.0) == 0x7E and fp8.encode(1e30) == 0x7E
    assert fp8.encode(-1e30) == 0xFE


def test_matches_torch_float8_cast_in_range():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 3)
    x = x.clamp(-440, 440)
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = fp8.encode(x.numpy().astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_quantize_divides_in_float32():
    x = np.array([1.0, 3.0, -7.5], np.float32)
    s = 0.1
    want = fp8.encode((x / np.float32(s)).astype(np.float64))
    np.testing.assert_array_equal(fp8.quantize(x, s), want)


def test_cache_write_fp8_slots():
    rng = np.random.default_rng(2)
    k = rng.standard_normal((3, 2, 8)).astype(np.float32)
    v = rng.standard_normal((3, 2, 8)).astype(np.float32)
    kc0 = np.zeros((2, 16, 2, 8), np.uint8)
    kc, vc = fp8.cache_write_fp8(k, v, [5, -1, 20], kc0, kc0, 0.05, 0.02)
    np.testing.assert_array_equal(kc[0, 5], fp8.quantize(k[0], 0.05))
    np.testing.assert_array_equal(vc[1, 4], fp8.quantize(v[2], 0.02))
    assert not kc[0, 6:].any() and not kc[1, :4].any()
    np.testing.assert_allclose(fp8.dequantize(kc[0, 5], 0.05), k[0], rtol=0.07, atol=0.05 * 2 ** -9)
