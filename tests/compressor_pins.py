"""Pins of the compressor oracle: a hand-derived pooling, closed forms,
invariants and the streaming property."""

from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden():
    out = {}
    with open(os.path.join(GOLDEN, "compressor_pool.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, *v = line.split()
                out[k] = [float(x) for x in v]
    return out


def pin_golden(cm):
    g = _golden()
    r2 = cm.pool(np.array([[1.0, 2.0], [3.0, 4.0]]), np.array([[0.0, 0.0], [math.log(3.0), 0.0]]), 2)
    assert np.allclose(r2[0], g["r2"], rtol=0, atol=1e-12), r2
    r3 = cm.pool(np.array([[2.0], [4.0], [8.0]]), np.log(np.array([[1.0], [2.0], [5.0]])), 3)
    assert np.allclose(r3[0], g["r3"], rtol=0, atol=1e-12), r3


def pin_equal_scores_mean(cm):
    rng = np.random.default_rng(50)
    kv = rng.standard_normal((12, 16))
    s = np.tile(rng.standard_normal((1, 16)), (12, 1))  # the same score at every position, per dim
    got = cm.pool(kv, s, 4)
    assert np.allclose(got, kv.reshape(3, 4, 16).mean(axis=1), rtol=0, atol=1e-12)


def pin_dominant_position(cm):
    kv = np.arange(24, dtype=np.float64).reshape(8, 3)
    s = np.zeros((8, 3))
    s[2, 0] = 60.0   # span 0, dim 0: row 2 wins
    s[5, 2] = 60.0   # span 1, dim 2: row 5 wins
    got = cm.pool(kv, s, 4)
    assert abs(got[0, 0] - kv[2, 0]) < 1e-12 and abs(got[1, 2] - kv[5, 2]) < 1e-12
    assert np.isclose(got[0, 1], kv[:4, 1].mean()) and np.isclose(got[1, 0], kv[4:, 0].mean())


def pin_shift_invariance(cm):
    rng = np.random.default_rng(51)
    kv = rng.standard_normal((8, 5))
    s = rng.standard_normal((8, 5))
    shift = np.repeat(rng.standard_normal((2, 5)) * 30, 4, axis=0)  # one shift per (span, dim)
    assert np.allclose(cm.pool(kv, s, 4), cm.pool(kv, s + shift, 4), rtol=0, atol=1e-10)


def pin_ratio_one_identity(cm):
    rng = np.random.default_rng(52)
    kv = rng.standard_normal((7, 9))
    assert np.allclose(cm.pool(kv, rng.standard_normal((7, 9)), 1), kv, rtol=0, atol=0)


def pin_counts(cm):
    w = 3
    for ratio in (1, 4, 128):
        for have in range(min(ratio, 5)):
            for n_new in (0, 1, ratio - 1, ratio, 3 * ratio + 2):
                rows, sk, ss = cm.append(np.zeros((have, w)), np.zeros((have, w)), np.ones((n_new, w)),
                                         np.zeros((n_new, w)), ratio)
                assert rows.shape[0] == (have + n_new) // ratio
                assert sk.shape[0] == (have + n_new) % ratio == ss.shape[0]


def pin_streaming_equals_one_call(cm):
    rng = np.random.default_rng(53)
    for ratio in (4, 7):
        kv = rng.standard_normal((61, 6))
        s = rng.standard_normal((61, 6)) * 3
        whole, tail_kv, tail_s = cm.append(np.zeros((0, 6)), np.zeros((0, 6)), kv, s, ratio)
        sk, ss, rows, i = np.zeros((0, 6)), np.zeros((0, 6)), [], 0
        for step in (1, 2, 9, 0, 5, 13, 3, 28):
            r, sk, ss = cm.append(sk, ss, kv[i:i + step], s[i:i + step], ratio)
            rows.append(r)
            i += step
            # the state after each call is the incomplete span, oldest row first
            assert np.array_equal(sk, kv[(i // ratio) * ratio:i]) and np.array_equal(ss, s[(i // ratio) * ratio:i])
        assert i == 61
        assert np.allclose(np.concatenate(rows), whole, rtol=0, atol=1e-12)
        assert np.array_equal(sk, tail_kv) and np.array_equal(ss, tail_s)
        assert np.array_equal(tail_kv, kv[(61 // ratio) * ratio:])  # the state is the incomplete span, in order


ALL_PINS = [pin_golden, pin_equal_scores_mean, pin_dominant_position, pin_shift_invariance, pin_ratio_one_identity,
            pin_counts, pin_streaming_equals_one_call]
