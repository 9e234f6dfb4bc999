"""FP8 (E4M3) KV-cache quantisation for the oracle.  TEST INFRASTRUCTURE ONLY.

"Serving models at scale with vLLM", section Your model is too big: KV data
can be stored at lower precision (8-bit instead of 16-bit).  The pages name
no format; the reading used here is the common 8-bit float E4M3:
  1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
  encodes subnormals m * 2^-9; no infinities; S.1111.111 is NaN; the largest
  finite magnitude is 1.75 * 2^8 = 448.
A cache element holds code = E4M3(x / scale), the division done in float32
and the rounding to nearest with ties to the even code, saturating to +-448
(NaN stays NaN).  Its value is decode(code) * scale.  The scale is one float
per cache tensor (one for K, one for V).

Written from that definition with float64 arithmetic, apart from the CUDA
path.
"""
from __future__ import annotations

import numpy as np

MAX_FINITE = 448.0


def _all_finite_values() -> np.ndarray:
    """Value of every non-negative finite code 0x00..0x7E, in code order."""
    vals = np.empty(127, dtype=np.float64)
    for code in range(127):
        e, m = code >> 3, code & 7
        vals[code] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_POS = _all_finite_values()


def decode(codes) -> np.ndarray:
    """float64 value of each E4M3 code (uint8)."""
    c = np.asarray(codes, dtype=np.uint8)
    mag = c & 0x7F
    out = _POS[np.minimum(mag, 126)]
    out = np.where(mag == 0x7F, np.nan, out)
    return np.where(c & 0x80, -out, out)


def encode(x) -> np.ndarray:
    """E4M3 code of each value: nearest representable magnitude, ties to the
    even code, magnitudes past 448 saturate to 448, NaN -> 0x7F (sign kept)."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.minimum(a, MAX_FINITE))
    # index of the largest representable value <= a, and the next one up
    lo = np.searchsorted(_POS, a, side="right") - 1
    lo = np.clip(lo, 0, 126)
    hi = np.minimum(lo + 1, 126)
    d_lo = a - _POS[lo]
    d_hi = _POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (lo % 2 == 1) & (hi != lo))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(nan, np.uint8(0x7F), code)
    return np.where(sign, code | np.uint8(0x80), code).astype(np.uint8)


def quantize(x, scale: float) -> np.ndarray:
    """Codes of x / scale, the division in float32 (x widened exactly first)."""
    xf = np.asarray(x, dtype=np.float32)
    return encode(xf / np.float32(scale))


def cache_write_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale: float, v_scale: float,
                    block_size: int = 16):
    """Slot write into FP8 caches: token t's K and V (float, e.g. widened bf16)
    are quantised with the tensors' scales and stored in slot
    slot_mapping[t]; negative slots are skipped.  Returns new uint8 caches."""
    kc = np.array(k_cache, dtype=np.uint8, copy=True)
    vc = np.array(v_cache, dtype=np.uint8, copy=True)
    kq = quantize(k, k_scale)
    vq = quantize(v, v_scale)
    for t, s in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if s < 0:
            continue
        kc[s // block_size, s % block_size] = kq[t]
        vc[s // block_size, s % block_size] = vq[t]
    return kc, vc


def dequantize(cache_codes, scale: float) -> np.ndarray:
    """float64 values of a whole FP8 cache."""
    return decode(cache_codes) * float(scale)
