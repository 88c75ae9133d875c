"""Plain CPU oracle of FP8 K/V rows: the E4M3 code, and per-row quantisation.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module; the product path never does.  It
shares no code with the CUDA library.

Passage: "DwarfStar 4 (DS4) - DeepSeek V4 Flash Inference Engine", sections
"GPU Backend Architecture" (the GPU op list includes DS4-specific FP8 KV
quantization) and "Whole-Model Graph Execution" (K/V rows are quantised to FP8
before they are stored).  The pages do not define the format.  Readings
(each pinned by a test):

* the FP8 format is E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa
  bits; exponent field 0 holds subnormals of 2^-6 * m/8; no infinities; the
  code S.1111.111 is NaN, so the largest finite magnitude is 448);
* one fp32 scale per row: ``scale = absmax / 448`` and code = E4M3 of
  ``x * (448 / absmax)``, both quotients and the product in fp32 with
  round-to-nearest-even, the code rounded to nearest even and saturated to
  +-448; an all-zero row has scale 0 and codes 0;
* a row's value is ``decode(code) * scale``.

The code is built here from its definition (enumerating the 256 bit patterns),
not from any library conversion.
"""

from __future__ import annotations

import numpy as np


def decode_table() -> np.ndarray:
    """float64 value of each of the 256 codes (NaN for the two NaN codes)."""
    out = np.empty(256, dtype=np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            out[c] = np.nan
        elif e == 0:
            out[c] = sign * (m / 8.0) * 2.0 ** -6
        else:
            out[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_TABLE = decode_table()
# finite non-negative codes in increasing value order (0x00 .. 0x7E)
_POS_CODES = np.arange(0x7F)
_POS_VALUES = _TABLE[_POS_CODES]


def encode(y) -> np.ndarray:
    """E4M3 code of each value: nearest finite code, ties to the even code
    (even mantissa), magnitudes of 448 and above saturate to 448; NaN -> 0x7F."""
    y = np.asarray(y, dtype=np.float64)
    nan = np.isnan(y)
    a = np.where(nan, 0.0, np.abs(y))
    v = _POS_VALUES
    j = np.searchsorted(v, a, side="left")          # first code whose value >= a
    hi = np.clip(j, 0, len(v) - 1)
    lo = np.clip(j - 1, 0, len(v) - 1)
    exact = v[hi] == a
    d_lo, d_hi = a - v[lo], v[hi] - a
    code = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    code = np.where(exact, hi, code)
    code = np.where(a >= 448.0, 0x7E, code)
    code = np.where(nan, 0x7F, code).astype(np.uint8)
    return code | (np.signbit(y).astype(np.uint8) << 7)


def quantize_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Per-row E4M3 quantisation of fp16 rows: (codes uint8 [rows, dim], scale fp32 [rows])."""
    x = np.asarray(x)
    rows = x.shape[0]
    codes = np.zeros(x.shape, dtype=np.uint8)
    scales = np.zeros(rows, dtype=np.float32)
    for r in range(rows):
        xr = x[r].astype(np.float32)
        amax = np.float32(np.max(np.abs(xr))) if xr.size else np.float32(0)
        if amax == 0:
            continue
        inv = np.float32(448.0) / amax               # fp32 quotient, round to nearest even
        scales[r] = amax / np.float32(448.0)
        y = (xr * inv).astype(np.float32)            # fp32 product, round to nearest even
        codes[r] = encode(y)
    return codes, scales


def dequantize_rows(codes, scales) -> np.ndarray:
    """float64 value of each element: decode(code) * scale."""
    return _TABLE[np.asarray(codes)] * np.asarray(scales, dtype=np.float64)[:, None]
