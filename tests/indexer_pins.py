"""Pins that tie the indexer oracle to hand-derived values, closed forms,
invariants and brute force.

Each ``pin_*`` takes the indexer oracle module and raises ``AssertionError``
when it disagrees.  ``test_indexer_oracle.py`` runs them on the oracle as it is
and on copies with a planted mistake (each mistake must fail some pin).
"""

from __future__ import annotations

import itertools
import os

import numpy as np

from mqa_flash_attention_gb300.workloads import make_layout

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append(line.split())
    return out


def _layout(q_pos0, T=1, ratio=4, n_comp=8):
    # the indexer reads only T, q_pos0 and ratio from the layout
    return make_layout(T=T, q_pos0=q_pos0, n_raw=1, raw_pos0=q_pos0, n_comp=n_comp, ratio=ratio)


def _golden_case():
    q = np.array([[[1, 0, 2, 0], [0, 1, 0, -1]]], dtype=np.float16)
    k = np.array([[1, 1, 1, 1], [2, 0, 0, 0], [0, 0, 0, 3], [1, 0, 0, 0]], dtype=np.float16)
    w = np.array([[1.0, 0.5]], dtype=np.float32)
    return _layout(11, n_comp=4), q, k, w


def pin_scores_golden(ix):
    L, q, k, w = _golden_case()
    for f, *vals in _rows("indexer_scores.txt"):
        want = np.array([float(v) for v in vals])
        got = ix.scores(L, q, k, w, 0.5, f == "relu")[0]
        assert np.array_equal(got, want), (f, got, want)


_TOPK_SCORES = np.array([0.5, 2.0, -1.0, 2.0, 0.25, 3.0, 9.0, 9.0], dtype=np.float32)


def pin_topk_golden(ix):
    for row in _rows("indexer_topk.txt"):
        p, k = int(row[0]), int(row[1])
        want = np.array([int(v) for v in row[3:]], dtype=np.int32)
        got = ix.topk(_layout(p), _TOPK_SCORES[None, :], k)[0]
        assert np.array_equal(got, want), (p, k, got, want)


def pin_candidate_count(ix):
    # the attention's hand-derived compressed-row counts (same pooled-span rule)
    for ratio, n_comp, p, count in _rows("comp_visible.txt"):
        ratio, n_comp, p, count = int(ratio), int(n_comp), int(p), int(count)
        L = _layout(p, ratio=ratio, n_comp=n_comp)
        q = np.ones((1, 1, 8), np.float16)
        k = np.ones((n_comp, 8), np.float16)
        s = ix.scores(L, q, k, np.ones((1, 1), np.float32), 1.0, False)[0]
        assert int(np.isfinite(s).sum()) == count, (ratio, n_comp, p)
        assert np.isfinite(s[:count]).all()


def pin_one_hot_dot_product(ix):
    # one head, w = 1, identity: q = a e_i, k_c = b e_j  ->  s = scale * a * b if i == j else 0
    L = _layout(1000, n_comp=6)
    q = np.zeros((1, 1, 16), np.float16)
    q[0, 0, 3] = 3.0
    k = np.zeros((6, 16), np.float16)
    for c in range(6):
        k[c, c] = c + 1.0
    s = ix.scores(L, q, k, np.ones((1, 1), np.float32), 0.25, False)[0]
    want = np.zeros(6)
    want[3] = 0.25 * 3.0 * 4.0
    assert np.array_equal(s, want), s


def pin_heads_weighted_sum(ix):
    # w = e_h picks head h alone; scores are linear in w; heads permute with w
    rng = np.random.default_rng(5)
    L = _layout(200, T=2, n_comp=20)
    q = rng.standard_normal((2, 4, 32)).astype(np.float16)
    k = rng.standard_normal((20, 32)).astype(np.float16)
    w = rng.standard_normal((2, 4)).astype(np.float32)
    for relu in (False, True):
        full = ix.scores(L, q, k, w, 0.125, relu)
        parts = []
        for h in range(4):
            e = np.zeros((2, 4), np.float32)
            e[:, h] = 1.0
            ph = ix.scores(L, q, k, e, 0.125, relu)
            one = ix.scores(L, q[:, h:h + 1], k, np.ones((2, 1), np.float32), 0.125, relu)
            assert np.allclose(ph, one, rtol=0, atol=1e-12)
            parts.append(ph)
        fin = np.isfinite(full)
        comb = sum(w[:, h:h + 1] * np.where(fin, parts[h], 0.0) for h in range(4))
        assert np.allclose(full[fin], comb[fin], rtol=1e-12, atol=1e-12)
        perm = [2, 0, 3, 1]
        assert np.allclose(ix.scores(L, q[:, perm], k, w[:, perm], 0.125, relu)[fin], full[fin], rtol=1e-12)


def pin_relu(ix):
    # with w >= 0: relu scores >= identity scores; a row with every dot < 0 scores 0 under relu
    rng = np.random.default_rng(6)
    L = _layout(100, n_comp=10)
    q = rng.standard_normal((1, 3, 16)).astype(np.float16)
    k = rng.standard_normal((10, 16)).astype(np.float16)
    q_pos = np.abs(q)
    k_neg = -np.abs(k)
    w = np.abs(rng.standard_normal((1, 3))).astype(np.float32) + 0.1
    a = ix.scores(L, q, k, w, 0.5, False)
    b = ix.scores(L, q, k, w, 0.5, True)
    fin = np.isfinite(a)
    assert (b[fin] >= a[fin] - 1e-12).all()
    z = ix.scores(L, q_pos, k_neg, w, 0.5, True)
    assert np.array_equal(z[np.isfinite(z)], np.zeros(int(np.isfinite(z).sum())))
    assert (ix.scores(L, q_pos, k_neg, w, 0.5, False)[np.isfinite(z)] < 0).all()


def pin_scale_linear(ix):
    rng = np.random.default_rng(7)
    L = _layout(60, n_comp=16)
    q = rng.standard_normal((1, 2, 8)).astype(np.float16)
    k = rng.standard_normal((16, 8)).astype(np.float16)
    w = rng.standard_normal((1, 2)).astype(np.float32)
    a = ix.scores(L, q, k, w, 1.0, False)
    b = ix.scores(L, q, k, w, 0.25, False)
    fin = np.isfinite(a)
    assert np.allclose(b[fin], 0.25 * a[fin], rtol=1e-12, atol=0)


def _valid_selection(scores, cand, chosen):
    """Definition check: every chosen row beats every candidate left out
    (larger score, or equal score and lower index)."""
    v = np.where(np.isnan(scores), -np.inf, scores)
    left = [j for j in cand if j not in chosen]
    return all(v[i] > v[j] or (v[i] == v[j] and i < j) for i in chosen for j in left)


def pin_topk_bruteforce(ix):
    rng = np.random.default_rng(8)
    for trial in range(120):
        n = int(rng.integers(1, 9))
        ratio = int(rng.choice([1, 2, 4]))
        p = int(rng.integers(0, 10 * ratio))
        k = int(rng.integers(1, 7))
        s = rng.integers(-3, 4, size=n).astype(np.float32)  # small integers: many ties
        s[rng.random(n) < 0.15] = -np.inf
        s[rng.random(n) < 0.1] = np.nan
        L = _layout(p, ratio=ratio, n_comp=n)
        cand = [c for c in range(n) if (c + 1) * ratio <= p + 1]
        m = min(k, len(cand))
        valid = [set(S) for S in itertools.combinations(cand, m) if _valid_selection(s, cand, set(S))]
        assert len(valid) == 1, (trial, s, cand, k)
        want = sorted(valid[0]) + [-1] * (k - m)
        got = ix.topk(L, s[None, :], k)[0]
        assert list(got) == want, (trial, s, p, ratio, k, got, want)


def pin_topk_invariants(ix):
    # larger random case: ascending, distinct, candidates only, definition holds, -1 only at the tail
    rng = np.random.default_rng(9)
    n, k = 300, 64
    L = _layout(700, T=3, ratio=4, n_comp=n)
    s = np.round(rng.standard_normal((3, n)) * 4).astype(np.float32)
    out = ix.topk(L, s, k)
    for t in range(3):
        p = 700 + t
        cand = [c for c in range(n) if (c + 1) * 4 <= p + 1]
        sel = [int(x) for x in out[t] if x >= 0]
        assert len(sel) == min(k, len(cand))
        assert sel == sorted(set(sel)) and all(c in cand for c in sel)
        assert (out[t][len(sel):] == -1).all()
        assert _valid_selection(s[t], cand, set(sel))


ALL_PINS = [pin_scores_golden, pin_topk_golden, pin_candidate_count, pin_one_hot_dot_product,
            pin_heads_weighted_sum, pin_relu, pin_scale_linear, pin_topk_bruteforce, pin_topk_invariants]
