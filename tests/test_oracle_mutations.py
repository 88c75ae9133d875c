"""Planted mistakes in the oracle must each fail at least one pin (CPU only).

Every mutation below is a plausible slip (a window off by one, a dropped scale,
K and V swapped, a bias ignored, a transposed reduction ...).  It is planted in
the oracle module with ``monkeypatch`` and the whole pin set is run; the test
passes only if some pin catches it.  This is what makes the pins a check on the
oracle rather than a restatement of it.
"""

import numpy as np
import pytest

import oracle.mqa as om

from oracle_pins import ALL_PINS

_orig_softmax = om._softmax_weighted
_orig_pairs = om.pair_visibility


def _window_129(layout, p):
    pos = layout["raw_pos0"] + np.arange(layout["n_raw"], dtype=np.int64)
    return (pos >= p - layout["window"]) & (pos <= p)


def _window_no_self(layout, p):
    pos = layout["raw_pos0"] + np.arange(layout["n_raw"], dtype=np.int64)
    return (pos >= p - layout["window"] + 1) & (pos < p)


def _window_rows_not_positions(layout, p):
    pos = np.arange(layout["n_raw"], dtype=np.int64)
    return (pos >= p - layout["window"] + 1) & (pos <= p)


def _comp_strict(layout, p):
    c = np.arange(layout["n_comp"], dtype=np.int64)
    return (c + 1) * layout["ratio"] <= p


def _comp_span_start(layout, p):
    c = np.arange(layout["n_comp"], dtype=np.int64)
    return c * layout["ratio"] <= p


def _softmax_variant(kind):
    def f(q_t, keys, vals, bias, scale):
        if keys.shape[0] == 0:
            return np.zeros((64, 512)), np.full(64, -np.inf)
        if kind == "kv_swapped":
            keys, vals = vals, keys
        if kind == "no_scale":
            scale = 1.0
        if kind == "bias_ignored":
            bias = np.zeros_like(bias)
        if kind == "bias_negated":
            bias = -bias
        if kind == "head0_only":
            q_t = np.broadcast_to(q_t[0], q_t.shape)
        s = scale * (q_t @ keys.T) + bias[None, :]
        if kind == "max_over_heads":
            m = s.max(axis=0, keepdims=True)
            w = np.exp(s - m)
            den = w.sum(axis=0, keepdims=True)
            return (w / den) @ vals, np.log(den[0, :64] if den.shape[1] >= 64 else np.ones(64))
        m = s.max(axis=1, keepdims=True)
        w = np.exp(s - m)
        den = w.sum(axis=1, keepdims=True)
        if kind == "no_normalise":
            o = w @ vals
        else:
            o = (w @ vals) / den
        lse = m[:, 0] + np.log(den[:, 0])
        if kind == "lse_without_max":
            lse = np.log(den[:, 0])
        return o, lse
    return f


def _unique_rows(lst, n_comp):
    lst = np.asarray(lst, dtype=np.int64)
    return np.unique(lst[(lst >= 0) & (lst < n_comp)])


def _rows_past_the_end_kept(lst, n_comp):
    lst = np.asarray(lst, dtype=np.int64)
    return lst[lst >= 0]


def _rows_wrapped(lst, n_comp):
    lst = np.asarray(lst, dtype=np.int64)
    return lst[lst >= 0] % max(n_comp, 1)


def _pairs_pad_visible(layout, mask=None):
    vis, bias = _orig_pairs(layout, mask)
    npr = -(-layout["n_raw"] // 32) * 32
    if mask is None:
        vis[:, layout["n_raw"]: npr] = vis[:, max(layout["n_raw"] - 1, 0): max(layout["n_raw"], 1)]
    return vis, bias


def _pairs_bias_ignored_in_status(layout, mask=None):
    vis, bias = _orig_pairs(layout, mask)
    return vis, np.zeros_like(bias)


def _status_any_all_swapped(layout, q_tile, mask=None):
    st = _orig_status(layout, q_tile, mask)
    return np.where(st == 2, 1, np.where(st == 1, 2, 0)).astype(np.uint8)


def _pad_keeps_garbage(src, n_rows):
    out = np.array(src[: -(-n_rows // 32) * 32], copy=True)
    return out


_orig_status = om.block_status

MUTATIONS = {
    "window_129_positions": ("raw_visible", _window_129),
    "window_excludes_self": ("raw_visible", _window_no_self),
    "window_ignores_raw_pos0": ("raw_visible", _window_rows_not_positions),
    "comp_strict_inequality": ("comp_visible", _comp_strict),
    "comp_visible_at_span_start": ("comp_visible", _comp_span_start),
    "kv_swapped": ("_softmax_weighted", _softmax_variant("kv_swapped")),
    "scale_dropped": ("_softmax_weighted", _softmax_variant("no_scale")),
    "bias_ignored": ("_softmax_weighted", _softmax_variant("bias_ignored")),
    "bias_negated": ("_softmax_weighted", _softmax_variant("bias_negated")),
    "head0_query_for_all_heads": ("_softmax_weighted", _softmax_variant("head0_only")),
    "softmax_over_heads": ("_softmax_weighted", _softmax_variant("max_over_heads")),
    "no_normalisation": ("_softmax_weighted", _softmax_variant("no_normalise")),
    "lse_without_max": ("_softmax_weighted", _softmax_variant("lse_without_max")),
    "index_duplicates_collapsed": ("listed_rows", _unique_rows),
    "index_entries_past_the_rows_kept": ("listed_rows", _rows_past_the_end_kept),
    "index_entries_wrapped_modulo_rows": ("listed_rows", _rows_wrapped),
    "status_pad_rows_visible": ("pair_visibility", _pairs_pad_visible),
    "status_bias_ignored": ("pair_visibility", _pairs_bias_ignored_in_status),
    "status_partial_full_swapped": ("block_status", _status_any_all_swapped),
    "pad_tail_not_zeroed": ("pad_rows", _pad_keeps_garbage),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(om, attr, fn)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(om)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name!r}"
