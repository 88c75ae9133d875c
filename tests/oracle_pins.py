"""Pins that tie the oracle to facts fixed by the pages and by mathematics.

Each ``pin_*`` takes the oracle module and raises ``AssertionError`` when the
oracle disagrees with something it must reproduce: a hand-derived golden value
(``tests/golden``), a closed form, an invariant of softmax attention or a
brute-force evaluation on a tiny case.  ``test_oracle_pins.py`` runs them on the
oracle as it is; ``test_oracle_mutations.py`` runs them on copies of the oracle
with a planted mistake and checks that some pin fails.
"""

from __future__ import annotations

import math
import os

import numpy as np

from mqa_flash_attention_gb300 import synth
from mqa_flash_attention_gb300.workloads import make_layout

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
H, D = 64, 512
SCALE = 1.0 / math.sqrt(512)


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _normal(seed, stream, shape):
    return synth.normal_f16(seed, stream, shape)


def _tiny_layout(**kw):
    base = dict(T=16, q_pos0=144, n_raw=160, raw_pos0=0)
    base.update(kw)
    return make_layout(**base)


# ---------------------------------------------------------------- golden values

def pin_window_golden(o):
    """Q = 0 makes every visible score equal, so o is the mean of the visible V
    rows; with V row i one-hot at column i the mean reveals the visible set,
    which must be the hand-derived window ``tests/golden/window_tiny.txt``."""
    L = _tiny_layout()
    q = np.zeros((16, H, D), np.float16)
    k = _normal(11, 2, (160, D))
    v = np.zeros((160, D), np.float16)
    v[np.arange(160), np.arange(160)] = 1.0
    out, lse = o.attention(L, q, k, v)
    for t, p, first, last, count in (map(int, r) for r in _golden_rows("window_tiny.txt")):
        assert p == 144 + t
        want = np.zeros(D)
        want[first: last + 1] = 1.0 / count
        for h in (0, 17, 63):
            np.testing.assert_allclose(out[t, h], want, rtol=0, atol=1e-14)
            assert abs(lse[t, h] - math.log(count)) < 1e-12


def pin_comp_golden(o):
    """Same mean-of-V probe over compressed rows only (no raw rows): the visible
    compressed rows must be ``0 .. count-1`` of ``tests/golden/comp_visible.txt``."""
    for ratio, n_comp, p, count in (map(int, r) for r in _golden_rows("comp_visible.txt")):
        L = make_layout(T=1, q_pos0=p, n_raw=0, raw_pos0=0, n_comp=n_comp, ratio=ratio)
        q = np.zeros((1, H, D), np.float16)
        kc = _normal(12, 4, (n_comp, D))
        vc = np.zeros((n_comp, D), np.float16)
        vc[np.arange(n_comp), np.arange(n_comp)] = 1.0
        out, lse = o.attention(L, q, np.zeros((0, D), np.float16), np.zeros((0, D), np.float16), kc, vc)
        want = np.zeros(D)
        if count:
            want[:count] = 1.0 / count
            assert abs(lse[0, 5] - math.log(count)) < 1e-12
        else:
            assert lse[0, 5] == -np.inf
        np.testing.assert_allclose(out[0, 5], want, rtol=0, atol=1e-14)


def parse_block_status_golden():
    cases, cur = [], None
    for r in _golden_rows("block_status.txt"):
        if r[0] == "layout":
            T, q0, nr, rp0, nc, ratio, win, qt = map(int, r[1:])
            cur = (make_layout(T=T, q_pos0=q0, n_raw=nr, raw_pos0=rp0, n_comp=nc, ratio=ratio,
                               window=win), qt, [])
        elif r[0] == "end":
            cases.append((cur[0], cur[1], np.array(cur[2], dtype=np.uint8)))
            cur = None
        else:
            cur[2].append([int(x) for x in r])
    return cases


def pin_block_status_golden(o):
    """Block status bytes equal the hand-derived ``tests/golden/block_status.txt``."""
    for L, qt, want in parse_block_status_golden():
        got = o.block_status(L, qt)
        assert got.shape == want.shape, (got.shape, want.shape)
        assert np.array_equal(got, want), (L, qt, got, want)


# ---------------------------------------------------------------- closed forms

def pin_one_hot(o):
    """q = 32 e_0 on every head and one K row equal to 32 e_0 (the others zero):
    that row scores 32*32/sqrt(512) ~ 45.25 above the rest, so o equals its V
    row up to e^-45."""
    L = _tiny_layout()
    q = np.zeros((16, H, D), np.float16)
    q[:, :, 0] = 32.0
    k = np.zeros((160, D), np.float16)
    k[100, 0] = 32.0
    v = _normal(13, 3, (160, D))
    out, _ = o.attention(L, q, k, v)
    want = v[100].astype(np.float64)
    for t in range(16):
        np.testing.assert_allclose(out[t], np.broadcast_to(want, (H, D)), rtol=0, atol=1e-12)


def pin_constant_v(o):
    """Every V row equal to u gives o = u for any scores."""
    L = _tiny_layout()
    q = _normal(14, 1, (16, H, D))
    k = _normal(14, 2, (160, D))
    u = _normal(14, 3, (1, D))
    v = np.repeat(u, 160, axis=0)
    out, _ = o.attention(L, q, k, v)
    np.testing.assert_allclose(out, np.broadcast_to(u[0].astype(np.float64), out.shape), rtol=1e-13, atol=1e-13)


def pin_single_row(o):
    """A window of one position leaves only the token's own row: o = v_self."""
    L = _tiny_layout(window=1)
    q = _normal(15, 1, (16, H, D))
    k = _normal(15, 2, (160, D))
    v = _normal(15, 3, (160, D))
    out, _ = o.attention(L, q, k, v)
    for t in range(16):
        want = v[144 + t].astype(np.float64)
        np.testing.assert_allclose(out[t], np.broadcast_to(want, (H, D)), rtol=0, atol=1e-15)


def pin_two_rows_logistic(o):
    """A window of two positions leaves rows a = p-1 and b = p; softmax over two
    values is the logistic function, so o = sig(d) v_b + (1 - sig(d)) v_a with
    d = (q.k_b - q.k_a) / sqrt(512), head by head."""
    L = _tiny_layout(window=2)
    q = _normal(16, 1, (16, H, D))
    k = _normal(16, 2, (160, D))
    v = _normal(16, 3, (160, D))
    out, _ = o.attention(L, q, k, v)
    for t in (0, 7, 15):
        a, b = 143 + t, 144 + t
        for h in (0, 31, 63):
            qh = q[t, h].astype(np.float64)
            d = (math.fsum(qh * k[b]) - math.fsum(qh * k[a])) / math.sqrt(512.0)
            sig = 1.0 / (1.0 + math.exp(-d))
            want = sig * v[b].astype(np.float64) + (1.0 - sig) * v[a].astype(np.float64)
            np.testing.assert_allclose(out[t, h], want, rtol=1e-12, atol=1e-12)


def pin_lse_two_rows(o):
    """With two visible rows, lse = log(e^{s_a} + e^{s_b})."""
    L = _tiny_layout(window=2)
    q = _normal(17, 1, (16, H, D))
    k = _normal(17, 2, (160, D))
    v = _normal(17, 3, (160, D))
    _, lse = o.attention(L, q, k, v)
    t, h = 4, 9
    qh = q[t, h].astype(np.float64)
    sa = math.fsum(qh * k[147]) / math.sqrt(512.0)
    sb = math.fsum(qh * k[148]) / math.sqrt(512.0)
    assert abs(lse[t, h] - math.log(math.exp(sa) + math.exp(sb))) < 1e-12


# ---------------------------------------------------------------- invariants

def pin_invisible_rows_no_effect(o):
    """Rows outside a token's window can hold anything finite (here +-65504, the
    fp16 extremes) without changing that token's output at all."""
    L = _tiny_layout()
    q = _normal(18, 1, (16, H, D))
    k = _normal(18, 2, (160, D))
    v = _normal(18, 3, (160, D))
    base, _ = o.attention(L, q, k, v)
    for t, _, first, last, _ in (map(int, r) for r in _golden_rows("window_tiny.txt")):
        if t not in (0, 9, 15):
            continue
        k2, v2 = k.copy(), v.copy()
        outside = np.ones(160, bool)
        outside[first: last + 1] = False
        k2[outside] = 65504.0
        v2[outside] = -65504.0
        got, _ = o.attention(L, q, k2, v2, tokens=[t])
        assert np.array_equal(got[0], base[t])


def pin_scale_equivalence(o):
    """Scaling q by 2 is the same as doubling the softmax scale."""
    L1 = _tiny_layout()
    L2 = _tiny_layout(scale=2.0 * SCALE)
    q = _normal(19, 1, (16, H, D))
    k = _normal(19, 2, (160, D))
    v = _normal(19, 3, (160, D))
    a, _ = o.attention(L1, (q.astype(np.float32) * 2).astype(np.float16), k, v)
    b, _ = o.attention(L2, q, k, v)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def _structural_mask(L):
    """A dense mask that is 0 exactly on the hand-derived tiny windows."""
    npr = -(-L["n_raw"] // 32) * 32
    m = np.full((L["T"], npr), -np.inf, np.float16)
    for t, _, first, last, _ in (map(int, r) for r in _golden_rows("window_tiny.txt")):
        m[t, first: last + 1] = 0.0
    return m


def pin_dense_mask_matches_structure(o):
    """A dense mask that is 0 on the window and -inf elsewhere reproduces the
    structural result, and permuting the rows together with the mask columns
    changes nothing (softmax attention is a sum over a set)."""
    L = _tiny_layout()
    q = _normal(20, 1, (16, H, D))
    k = _normal(20, 2, (160, D))
    v = _normal(20, 3, (160, D))
    base, _ = o.attention(L, q, k, v)
    m = _structural_mask(L)
    got, _ = o.attention(L, q, k, v, mask=m)
    np.testing.assert_allclose(got, base, rtol=1e-13, atol=1e-13)
    perm = np.argsort(synth.uniform(20, 9, 160))
    mp = m.copy()
    mp[:, :160] = m[:, perm]
    got2, _ = o.attention(L, q, k[perm], v[perm], mask=mp)
    np.testing.assert_allclose(got2, base, rtol=1e-12, atol=1e-12)


def pin_bias_is_log_multiplicity(o):
    """Adding log 2 to one row's bias weighs it exactly like listing it twice:
    the dense-mask bias is added to the scaled score in natural-log units, and
    an index list counts repeated entries once per occurrence."""
    L = make_layout(T=1, q_pos0=99, n_raw=0, raw_pos0=0, n_comp=24, ratio=4)
    q = _normal(21, 1, (1, H, D))
    kc = _normal(21, 4, (24, D))
    vc = _normal(21, 5, (24, D))
    empty = np.zeros((0, D), np.float16)
    idx = np.array([[3, 3, 5, 7, -1, -1]], np.int32)
    a, la = o.attention(L, q, empty, empty, kc, vc, idx=idx)
    m = np.full((1, 32), -np.inf, np.float64)
    m[0, [3, 5, 7]] = 0.0
    m[0, 3] = math.log(2.0)
    b, lb = o.attention(L, q, empty, empty, kc, vc, mask=m)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(la, lb, rtol=1e-12, atol=1e-12)


def pin_indexed_all_rows_equals_dense(o):
    """An index list that names every available compressed row, once, gives the
    dense (all pooled rows) result."""
    L = make_layout(T=3, q_pos0=57, n_raw=60, raw_pos0=0, n_comp=20, ratio=4, window=16)
    q = _normal(22, 1, (3, H, D))
    kr, vr = _normal(22, 2, (60, D)), _normal(22, 3, (60, D))
    kc, vc = _normal(22, 4, (20, D)), _normal(22, 5, (20, D))
    idx = np.full((3, 20), -1, np.int32)
    for t in range(3):
        n = (57 + t + 1) // 4           # pooled spans ended by p (comp_visible.txt)
        idx[t, 20 - n:] = np.arange(n)[::-1]   # order and -1 placement must not matter
    a, _ = o.attention(L, q, kr, vr, kc, vc, idx=idx)
    b, _ = o.attention(L, q, kr, vr, kc, vc)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


def pin_index_entries_past_the_rows_are_empty(o):
    """An index entry that names no stored row (>= n_comp, as well as < 0) is
    an empty slot, as the library's interface declares: a list whose only
    stored row is 5 gives exactly v_5 (one visible row has weight 1), and a
    list of out-of-range entries alone gives o = 0, lse = -inf."""
    L = make_layout(T=2, q_pos0=99, n_raw=0, raw_pos0=0, n_comp=24, ratio=4)
    q = _normal(27, 1, (2, H, D))
    kc, vc = _normal(27, 4, (24, D)), _normal(27, 5, (24, D))
    empty = np.zeros((0, D), np.float16)
    idx = np.array([[24, 5, 1000, -1, 2 ** 31 - 1],
                    [24, 25, 2 ** 31 - 1, -7, 47]], np.int32)
    out, lse = o.attention(L, q, empty, empty, kc, vc, idx=idx)
    assert np.array_equal(out[0], np.broadcast_to(vc[5].astype(np.float64), (H, D)))
    assert np.all(np.isfinite(lse[0]))
    assert np.all(out[1] == 0.0) and np.all(lse[1] == -np.inf)


def pin_no_visible_rows(o):
    """A token whose rows are all masked gets o = 0 and lse = -inf."""
    L = _tiny_layout(T=1)
    q = _normal(23, 1, (1, H, D))
    k = _normal(23, 2, (160, D))
    v = _normal(23, 3, (160, D))
    m = np.full((1, 160), -np.inf, np.float16)
    out, lse = o.attention(L, q, k, v, mask=m)
    assert np.all(out == 0.0) and np.all(lse == -np.inf)


# ---------------------------------------------------------------- brute force

def pin_bruteforce_tiny(o):
    """Scalar loops over (token, head, row, dim) on a tiny layout with raw and
    compressed rows; visibility decided pair by pair from positions."""
    L = make_layout(T=2, q_pos0=9, n_raw=7, raw_pos0=4, n_comp=3, ratio=3, window=4)
    q = _normal(24, 1, (2, H, D)).astype(np.float64)
    kr, vr = _normal(24, 2, (7, D)).astype(np.float64), _normal(24, 3, (7, D)).astype(np.float64)
    kc, vc = _normal(24, 4, (3, D)).astype(np.float64), _normal(24, 5, (3, D)).astype(np.float64)
    got, _ = o.attention(L, q.astype(np.float16), kr.astype(np.float16), vr.astype(np.float16),
                         kc.astype(np.float16), vc.astype(np.float16))
    for t in range(2):
        p = 9 + t
        rows = []
        for i in range(7):                 # raw row i at position 4 + i
            if p - 4 < 4 + i <= p:
                rows.append((kr[i], vr[i]))
        for c in range(3):                 # pooled positions 3c .. 3c+2 all <= p
            if 3 * c + 2 <= p:
                rows.append((kc[c], vc[c]))
        for h in (0, 1, 40, 63):
            sc = [math.fsum(q[t, h, d] * kk[d] for d in range(D)) / math.sqrt(512.0) for kk, _ in rows]
            mx = max(sc)
            w = [math.exp(s - mx) for s in sc]
            den = math.fsum(w)
            for d in (0, 1, 255, 511):
                num = math.fsum(wi * vv[d] for wi, (_, vv) in zip(w, rows))
                assert abs(got[t, h, d] - num / den) < 1e-12


def closed_form_status(L, q_tile):
    """Block status of a structural mask from interval arithmetic, no pair loop.

    A raw row at position x is seen by positions x .. x+W-1; a pooled row c by
    positions >= (c+1)*ratio - 1.  A q-tile covers positions P0..P1."""
    T, W = L["T"], L["window"]
    npr = -(-L["n_raw"] // 32)
    npc = -(-L["n_comp"] // 32)
    out = np.zeros((-(-T // q_tile), npr + npc), np.uint8)
    for b in range(out.shape[0]):
        P0 = L["q_pos0"] + b * q_tile
        P1 = L["q_pos0"] + min(T, (b + 1) * q_tile) - 1
        for k in range(npr):
            lo, hi = 32 * k, min(32 * k + 31, L["n_raw"] - 1)
            x0, x1 = L["raw_pos0"] + lo, L["raw_pos0"] + hi
            some = x0 <= P1 and x1 + W - 1 >= P0
            every = (hi - lo == 31) and x1 <= P0 and x0 + W - 1 >= P1
            out[b, k] = 2 if every else (1 if some else 0)
        for k in range(npc):
            lo, hi = 32 * k, min(32 * k + 31, L["n_comp"] - 1)
            some = (lo + 1) * L["ratio"] - 1 <= P1
            every = (hi - lo == 31) and (hi + 1) * L["ratio"] - 1 <= P0
            out[b, npr + k] = 2 if every else (1 if some else 0)
    return out


def pin_block_status_closed_form(o):
    """Brute-force status equals the interval rule on many random layouts."""
    rng_u = synth.uniform(25, 1, 4096)
    it = iter(rng_u)

    def ri(lo, hi):
        return lo + int(next(it) * (hi - lo + 1))

    for _ in range(60):
        T = ri(1, 40)
        W = ri(1, 150)
        n_raw = ri(0, 200)
        raw_pos0 = ri(0, 300)
        n_comp = ri(0, 90)
        ratio = (4, 128, 3)[ri(0, 2)]
        q_pos0 = ri(0, 400)
        L = make_layout(T=T, q_pos0=q_pos0, n_raw=n_raw, raw_pos0=raw_pos0, n_comp=n_comp,
                        ratio=ratio, window=W)
        for qt in (1, 2, 4, 16, 64):
            assert np.array_equal(o.block_status(L, qt), closed_form_status(L, qt)), (L, qt)


def pin_block_status_dense_mask(o):
    """Status from a dense mask: all -inf -> 0; all 0 on 32 real rows -> 2; a
    single nonzero bias or a single -inf in an otherwise open block -> 1; a
    block with pad rows is never 2."""
    L = make_layout(T=4, q_pos0=200, n_raw=100, raw_pos0=0, n_comp=0)
    m = np.zeros((4, 128), np.float16)
    m[:, 0:32] = -np.inf          # block 0: closed
    m[2, 40] = 0.5                # block 1: one biased pair
    m[1, 70] = -np.inf            # block 2: one closed pair
    st = o.block_status(L, 4, mask=m)
    assert st.tolist() == [[0, 1, 1, 1]], st
    st1 = o.block_status(L, 1, mask=m)
    assert st1.tolist() == [[0, 2, 2, 1], [0, 2, 1, 1], [0, 1, 2, 1], [0, 2, 2, 1]], st1


def pin_pad(o):
    """Padding keeps the rows and appends +0.0 rows up to a multiple of 32."""
    src = _normal(26, 2, (70, D))
    out = o.pad_rows(src, 45)
    assert out.shape == (64, D) and out.dtype == np.float16
    assert np.array_equal(out[:45].view(np.uint16), src[:45].view(np.uint16))
    assert np.all(out[45:].view(np.uint16) == 0)
    assert o.pad_rows(src, 64).shape == (64, D)
    assert o.pad_rows(src, 0).shape == (0, D)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
