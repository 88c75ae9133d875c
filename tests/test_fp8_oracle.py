"""The FP8 oracle against its pins, and planted mistakes against the pins (CPU only)."""

import numpy as np
import pytest

import oracle.fp8 as f8

from fp8_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_fp8_pin(pin):
    pin(f8)


def _table_variant(kind):
    def t():
        out = np.empty(256)
        for c in range(256):
            sign = -1.0 if c & 0x80 else 1.0
            e, m = (c >> 3) & 0xF, c & 7
            bias = 8 if kind == "bias8" else 7
            if e == 0xF and m == 7 and kind != "no_nan":
                out[c] = np.nan
            elif e == 0:
                out[c] = sign * (m / 8.0) * 2.0 ** (1 - bias) if kind != "no_subnormal" else 0.0
            else:
                out[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - bias)
        return out
    return t


def _encode_variant(kind):
    orig = f8.encode

    def enc(y):
        y = np.asarray(y, dtype=np.float64)
        if kind == "ties_away":
            a = np.abs(y)
            v = f8._POS_VALUES
            j = np.clip(np.searchsorted(v, a), 1, len(v) - 1)
            lo, hi = j - 1, j
            code = np.where(a - v[lo] < v[hi] - a, lo, hi)
            code = np.where(v[np.clip(np.searchsorted(v, a), 0, len(v) - 1)] == a,
                            np.clip(np.searchsorted(v, a), 0, len(v) - 1), code)
            code = np.where(a >= 448, 0x7E, code).astype(np.uint8)
            return code | (np.signbit(y).astype(np.uint8) << 7)
        if kind == "truncate":
            a = np.abs(y)
            j = np.clip(np.searchsorted(f8._POS_VALUES, a, side="right") - 1, 0, 0x7E).astype(np.uint8)
            return j | (np.signbit(y).astype(np.uint8) << 7)
        if kind == "saturate_nan":
            c = orig(y)
            return np.where(np.abs(y) > 448, (c & 0x80) | 0x7F, c).astype(np.uint8)
        return orig(y)
    return enc


def _quant_variant(kind):
    def q(x):
        x = np.asarray(x)
        codes = np.zeros(x.shape, np.uint8)
        scales = np.zeros(x.shape[0], np.float32)
        for r in range(x.shape[0]):
            xr = x[r].astype(np.float32)
            amax = np.float32(np.abs(xr).max())
            if amax == 0:
                continue
            lim = np.float32(240.0 if kind == "limit_240" else 448.0)
            scales[r] = amax / lim
            codes[r] = f8.encode((xr * (lim / amax)).astype(np.float32))
        return codes, scales
    return q


MUTATIONS = {
    "exponent bias 8": ("decode_table", _table_variant("bias8")),
    "subnormals flushed": ("decode_table", _table_variant("no_subnormal")),
    "no NaN code": ("decode_table", _table_variant("no_nan")),
    "ties away from zero": ("encode", _encode_variant("ties_away")),
    "truncation": ("encode", _encode_variant("truncate")),
    "overflow to NaN": ("encode", _encode_variant("saturate_nan")),
    "scale to 240": ("quantize_rows", _quant_variant("limit_240")),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_fp8_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(f8, attr, fn)
    if attr == "decode_table":  # the cached table and value list follow the planted table
        monkeypatch.setattr(f8, "_TABLE", fn())
        monkeypatch.setattr(f8, "_POS_VALUES", fn()[f8._POS_CODES])
    failed = []
    for pin in ALL_PINS:
        try:
            pin(f8)
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches: {name}"
