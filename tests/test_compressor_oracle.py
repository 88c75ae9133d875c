"""The compressor oracle against its pins, and planted mistakes against the pins (CPU only)."""

import numpy as np
import pytest

import oracle.compressor as cm

from compressor_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_compressor_pin(pin):
    pin(cm)


def _pool_variant(kind):
    def pool(kv, s, ratio):
        kv = np.asarray(kv, dtype=np.float64)
        s = np.asarray(s, dtype=np.float64)
        n = kv.shape[0] // ratio
        out = np.empty((n, kv.shape[1]))
        for c in range(n):
            lo = c * ratio + (1 if kind == "span_shift" and c * ratio + ratio < kv.shape[0] else 0)
            sk, vk = s[lo:lo + ratio], kv[lo:lo + ratio]
            if kind == "softmax_over_dims":
                w = np.exp(sk - sk.max(axis=1, keepdims=True))
                w = w / w.sum(axis=1, keepdims=True)
                out[c] = (w * vk).sum(axis=0)
                continue
            w = np.exp(sk - sk.max(axis=0, keepdims=True))
            if kind == "unnormalised":
                out[c] = (w * vk).sum(axis=0)
            elif kind == "mean_only":
                out[c] = vk.mean(axis=0)
            elif kind == "last_row":
                out[c] = vk[-1]
            else:
                out[c] = (w * vk).sum(axis=0) / w.sum(axis=0)
        return out
    return pool


def _append_variant(kind):
    orig = cm.append

    def append(state_kv, state_s, kv_new, s_new, ratio):
        if kind == "state_dropped":
            return orig(np.zeros((0, np.asarray(kv_new).shape[1])), np.zeros((0, np.asarray(kv_new).shape[1])),
                        kv_new, s_new, ratio)
        if kind == "state_reversed":
            return orig(np.asarray(state_kv)[::-1], np.asarray(state_s)[::-1], kv_new, s_new, ratio)
        return orig(state_kv, state_s, kv_new, s_new, ratio)
    return append


MUTATIONS = {
    "softmax over dimensions": ("pool", _pool_variant("softmax_over_dims")),
    "weights not normalised": ("pool", _pool_variant("unnormalised")),
    "plain mean": ("pool", _pool_variant("mean_only")),
    "last row of the span": ("pool", _pool_variant("last_row")),
    "span off by one": ("pool", _pool_variant("span_shift")),
    "state dropped between calls": ("append", _append_variant("state_dropped")),
    "state reversed": ("append", _append_variant("state_reversed")),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_compressor_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(cm, attr, fn)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(cm)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches: {name}"
