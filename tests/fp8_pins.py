"""Pins of the FP8 (E4M3) oracle: hand-derived codes, the format's own
properties, brute-force nearest rounding and a worked row quantisation."""

from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append(line.split())
    return out


def pin_codes_golden(f8):
    for val, code in _rows("e4m3.txt"):
        got = int(f8.encode(np.array([float(val)]))[0])
        assert got == int(code, 16), (val, hex(got), code)


def pin_decode_values(f8):
    t = f8.decode_table()
    assert t[0x38] == 1.0 and t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert t[0x01] == 2.0 ** -9 and t[0x08] == 2.0 ** -6 and t[0x77] == 240.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    fin = t[:0x7F]
    assert (np.diff(fin) > 0).all(), "finite non-negative codes must increase"
    assert np.array_equal(t[0x80:0xFF], -fin[:0x7F])


def pin_round_trip(f8):
    t = f8.decode_table()
    codes = np.array([c for c in range(256) if not np.isnan(t[c]) and c != 0x80], dtype=np.uint8)
    assert np.array_equal(f8.encode(t[codes]), codes)


def pin_nearest_bruteforce(f8):
    t = f8.decode_table()
    fin = np.array([c for c in range(256) if not np.isnan(t[c])])
    rng = np.random.default_rng(10)
    y = np.concatenate([rng.uniform(-460, 460, 2000), rng.uniform(-0.03, 0.03, 2000),
                        (t[fin][:-1] + t[fin][1:]) / 2])           # midpoints: ties
    y = y[np.abs(y) <= 448]
    got = f8.encode(y)
    for yi, c in zip(y, got):
        d = np.abs(t[fin] - yi)
        best = d.min()
        assert abs(t[c] - yi) == best, (yi, hex(c))
        cands = fin[d == best]
        if len(cands) > 1:  # tie: the even mantissa
            assert (c & 1) == 0, (yi, hex(c), cands)


def pin_saturation(f8):
    assert (f8.encode(np.array([449.0, 1e6, 480.0])) == 0x7E).all()
    assert (f8.encode(np.array([-449.0, -1e6])) == 0xFE).all()


def pin_quantize_worked_row(f8):
    # absmax 4: the multiplier is 448/4 = 112, so 1 -> 112 (0x6E), -2 -> -224 (0xF6),
    # 0.5 -> 56 (0x66), 4 -> 448 (0x7E); scale 4/448 in fp32
    x = np.zeros((1, 512), np.float16)
    x[0, :4] = [1.0, -2.0, 0.5, 4.0]
    codes, scale = f8.quantize_rows(x)
    assert list(codes[0, :4]) == [0x6E, 0xF6, 0x66, 0x7E] and (codes[0, 4:] == 0).all()
    assert scale[0] == np.float32(4.0) / np.float32(448.0)


def pin_quantize_properties(f8):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((64, 512)) * rng.uniform(0.01, 50, (64, 1))).astype(np.float16)
    x[3] = 0
    codes, scale = f8.quantize_rows(x)
    t = f8.decode_table()
    assert scale[3] == 0 and (codes[3] == 0).all()
    d = f8.dequantize_rows(codes, scale)
    xf = x.astype(np.float64)
    for r in range(64):
        if r == 3:
            continue
        amax = np.abs(xf[r]).max()
        assert np.isclose(scale[r], amax / 448, rtol=1e-6)
        assert np.abs(t[codes[r]]).max() == 448.0          # the absmax element lands on 448
        # error within half a code step (relative 1/16 above the subnormals) plus fp32 slack
        step = np.maximum(np.abs(xf[r]) / 8.0, 2.0 ** -9 * scale[r])
        assert (np.abs(d[r] - xf[r]) <= step / 2 * (1 + 1e-5) + 1e-12).all(), r


ALL_PINS = [pin_codes_golden, pin_decode_values, pin_round_trip, pin_nearest_bruteforce, pin_saturation,
            pin_quantize_worked_row, pin_quantize_properties]
