"""The indexer oracle against its pins, and planted mistakes against the pins (CPU only)."""

import numpy as np
import pytest

import oracle.indexer as ix

from indexer_pins import ALL_PINS

_orig_candidates = ix.candidates
_orig_scores = ix.scores
_orig_topk = ix.topk


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_indexer_pin(pin):
    pin(ix)


def _cand_strict(layout, p, n_rows):
    c = np.arange(n_rows, dtype=np.int64)
    return (c + 1) * int(layout["ratio"]) <= p


def _cand_span_start(layout, p, n_rows):
    c = np.arange(n_rows, dtype=np.int64)
    return c * int(layout["ratio"]) <= p


def _scores_variant(kind):
    def f(layout, q_idx, k_idx, w, scale, relu, tokens=None):
        q = np.asarray(q_idx)
        k = np.asarray(k_idx).astype(np.float64)
        w = np.asarray(w, dtype=np.float64)
        toks = range(q.shape[0]) if tokens is None else tokens
        out = np.full((len(toks), k.shape[0]), -np.inf)
        for i, t in enumerate(toks):
            p = int(layout["q_pos0"]) + int(t)
            cand = ix.candidates(layout, p, k.shape[0])
            if not cand.any():
                continue
            dots = (1.0 if kind == "no_scale" else scale) * (q[t].astype(np.float64) @ k[cand].T)
            if kind == "relu_after_weights":
                s = w[t] @ dots
                out[i, cand] = np.maximum(s, 0.0) if relu else s
                continue
            if relu and kind != "relu_ignored":
                dots = np.maximum(dots, 0.0)
            if kind == "weights_ignored":
                out[i, cand] = dots.sum(axis=0)
            elif kind == "head_zero_only":
                out[i, cand] = w[t, 0] * dots[0]
            elif kind == "abs_instead_of_relu" and relu:
                out[i, cand] = w[t] @ np.abs(q[t].astype(np.float64) @ k[cand].T * scale)
            else:
                out[i, cand] = w[t] @ dots
        return out
    return f


def _topk_variant(kind):
    def f(layout, s, top_k, tokens=None):
        s = np.asarray(s)
        toks = range(s.shape[0]) if tokens is None else tokens
        out = np.full((len(toks), top_k), -1, dtype=np.int32)
        for i, t in enumerate(toks):
            p = int(layout["q_pos0"]) + int(t)
            cand = np.nonzero(ix.candidates(layout, p, s.shape[1]))[0]
            if cand.size == 0:
                continue
            v = s[t, cand].astype(np.float64)
            v = np.where(np.isnan(v), np.inf if kind == "nan_high" else -np.inf, v)
            if kind == "ties_high_index":
                order = np.lexsort((-cand, -v))
            elif kind == "ascending_scores":
                order = np.lexsort((cand, v))
            else:
                order = np.lexsort((cand, -v))
            k = top_k - 1 if kind == "k_minus_one" else top_k
            chosen = cand[order[:k]]
            if kind != "score_order":
                chosen = np.sort(chosen)
            out[i, :chosen.size] = chosen
            if kind == "pad_zero":
                out[i, chosen.size:] = 0
        return out
    return f


MUTATIONS = {
    "candidates: span must end before p": ("candidates", _cand_strict),
    "candidates: span start instead of end": ("candidates", _cand_span_start),
    "scores: scale dropped": ("scores", _scores_variant("no_scale")),
    "scores: relu ignored": ("scores", _scores_variant("relu_ignored")),
    "scores: relu after the head sum": ("scores", _scores_variant("relu_after_weights")),
    "scores: head weights ignored": ("scores", _scores_variant("weights_ignored")),
    "scores: head 0 only": ("scores", _scores_variant("head_zero_only")),
    "scores: |x| instead of max(0, x)": ("scores", _scores_variant("abs_instead_of_relu")),
    "topk: ties to the higher index": ("topk", _topk_variant("ties_high_index")),
    "topk: smallest scores": ("topk", _topk_variant("ascending_scores")),
    "topk: output in score order": ("topk", _topk_variant("score_order")),
    "topk: one row short": ("topk", _topk_variant("k_minus_one")),
    "topk: pad with row 0": ("topk", _topk_variant("pad_zero")),
    "topk: NaN ranks first": ("topk", _topk_variant("nan_high")),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_indexer_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(ix, attr, fn)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(ix)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin catches: {name}"
