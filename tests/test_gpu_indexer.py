"""Indexer kernels against the indexer oracle (needs a GB300).

* Top-k selection: bit-exact.  Both sides select on the same fp32 scores, so
  the decision is taken in the same precision.
* Scores: fp16 inputs, fp32 tensor-core accumulation.  Per element the error is
  bounded by (head_dim + n_heads + 3) roundings of fp32 against the sum of the
  absolute terms, B = sum_h |w_h| * scale * sum_d |q_hd * k_cd|; the test
  allows 4 * (head_dim + n_heads + 3) * 2^-24 * B.  Non-candidate rows must be
  -inf exactly.
"""

import dataclasses

import numpy as np
import pytest

import oracle
from oracle import indexer as ix
from mqa_flash_attention_gb300 import workloads as W
from mqa_flash_attention_gb300.workloads import make_layout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as _torch
    from mqa_flash_attention_gb300 import build
    build.build()
    assert _torch.cuda.is_available()
    return _torch


@pytest.fixture(scope="module")
def ds4a(torch):
    from mqa_flash_attention_gb300 import ds4a as _ds4a
    _ds4a.lib()
    return _ds4a


@pytest.fixture(autouse=True)
def device_error_word_stays_clear(ds4a):
    ds4a.device_error_word(clear=True)
    yield
    w = ds4a.device_error_word(clear=True)
    assert w == 0, f"a device wait ran out during this test: error word {w:#010x}"


def dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def _layout(T, q_pos0, n_comp, ratio):
    return make_layout(T=T, q_pos0=q_pos0, n_raw=1, raw_pos0=q_pos0, n_comp=n_comp, ratio=ratio)


# ------------------------------------------------------------------ top-k

def _tie_heavy_scores(rng, T, n):
    s = np.round(rng.standard_normal((T, n)) * 3).astype(np.float32)   # integers: many ties
    s[rng.random((T, n)) < 0.05] = -np.inf
    s[rng.random((T, n)) < 0.02] = np.nan
    s[rng.random((T, n)) < 0.02] = np.float32(-0.0)
    s[rng.random((T, n)) < 0.01] = np.inf
    return s


@pytest.mark.parametrize("T,q_pos0,n_comp,ratio,top_k", [
    (5, 0, 40, 4, 3),            # first tokens: 0 or few candidates
    (16, 100, 37, 4, 512),       # fewer candidates than top_k: all of them, then -1
    (33, 2000, 600, 4, 7),
    (9, 30000, 8192, 4, 512),    # cached keys, the model's list length
    (4, 2 ** 20, 40000, 4, 512), # more candidates than the shared-memory cache
    (3, 5000, 300, 1, 1),
    (6, 131071, 1025, 128, 64),  # ratio 128
])
def test_topk_bitexact(torch, ds4a, T, q_pos0, n_comp, ratio, top_k):
    rng = np.random.default_rng(T * 1000 + n_comp)
    L = _layout(T, q_pos0, n_comp, ratio)
    s = _tie_heavy_scores(rng, T, n_comp)
    got = host(ds4a.indexer_topk(L, dev(torch, s), top_k))
    want = ix.topk(L, s, top_k)
    assert np.array_equal(got, want)


def test_topk_distinct_scores(torch, ds4a):
    rng = np.random.default_rng(3)
    L = _layout(64, 30720, 8192, 4)
    s = rng.standard_normal((64, 8192)).astype(np.float32)
    assert np.array_equal(host(ds4a.indexer_topk(L, dev(torch, s), 512)), ix.topk(L, s, 512))


def test_topk_all_equal(torch, ds4a):
    L = _layout(3, 30720, 8192, 4)
    s = np.full((3, 8192), 1.5, np.float32)
    got = host(ds4a.indexer_topk(L, dev(torch, s), 512))
    assert np.array_equal(got, np.tile(np.arange(512, dtype=np.int32), (3, 1)))


def test_topk_strided_rows(torch, ds4a):
    rng = np.random.default_rng(4)
    L = _layout(8, 900, 200, 4)
    s = _tie_heavy_scores(rng, 8, 256)              # row stride 256 > n_comp
    out = torch.full((8, 44), 7, dtype=torch.int32, device="cuda")
    ds4a.indexer_topk(L, dev(torch, s), 33, out=out[:, 4:37])   # 16-byte aligned rows
    o = host(out)
    assert np.array_equal(o[:, 4:37], ix.topk(L, s[:, :200], 33))
    assert (o[:, :4] == 7).all() and (o[:, 37:] == 7).all()


# ------------------------------------------------------------------ scores

def _check_scores(got, wl, tokens=None):
    L = wl.layout
    want = ix.scores(L, wl.q_idx, wl.k_idx, wl.w, wl.scale, wl.relu, tokens=tokens)
    bound = ix.scores(L, np.abs(wl.q_idx), np.abs(wl.k_idx), np.abs(wl.w), abs(wl.scale), False, tokens=tokens)
    g = np.asarray(got, np.float64)
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(g), fin), "-inf pattern differs"
    assert (g[~fin] == -np.inf).all()
    n_heads, head_dim = wl.q_idx.shape[1], wl.q_idx.shape[2]
    tol = 4.0 * (head_dim + n_heads + 3) * 2.0 ** -24 * bound[fin] + 1e-30
    err = np.abs(g[fin] - want[fin])
    assert (err <= tol).all(), f"max err {err.max():.3e}, worst ratio {(err / tol).max():.2f}"


def _indexer_case(T, q_pos0, n_comp, ratio, n_heads, head_dim, relu, seed):
    L = _layout(T, q_pos0, n_comp, ratio)
    return W.draw_indexer(f"ix_{n_heads}x{head_dim}", seed, L, n_heads, head_dim, 8, relu)


def _run_scores(torch, ds4a, wl):
    return host(ds4a.indexer_scores(wl.layout, dev(torch, wl.q_idx), dev(torch, wl.k_idx), dev(torch, wl.w),
                                    scale=wl.scale, relu=wl.relu))


@pytest.mark.parametrize("n_heads", [1, 2, 4, 8, 16, 32, 64, 128])
def test_scores_every_head_count(torch, ds4a, n_heads):
    # ragged: T not a multiple of the token group, n_comp not a multiple of 128,
    # early tokens with no candidate, a partial last tile
    wl = _indexer_case(T=2 * (256 // n_heads) + 3, q_pos0=5, n_comp=333, ratio=4, n_heads=n_heads, head_dim=64,
                       relu=n_heads % 2 == 0, seed=20 + n_heads)
    _check_scores(_run_scores(torch, ds4a, wl), wl)


@pytest.mark.parametrize("head_dim", [64, 128, 256])
@pytest.mark.parametrize("relu", [False, True])
def test_scores_head_dims(torch, ds4a, head_dim, relu):
    wl = _indexer_case(T=19, q_pos0=1200, n_comp=700, ratio=4, n_heads=64, head_dim=head_dim, relu=relu,
                       seed=40 + head_dim)
    _check_scores(_run_scores(torch, ds4a, wl), wl)


@pytest.mark.parametrize("relu", [False, True])
@pytest.mark.parametrize("n_heads", [8, 64])
def test_scores_negative_scale(torch, ds4a, relu, n_heads):
    # max(0, scale x) with scale < 0: the kernel folds |scale| into the weights and negates x
    wl = _indexer_case(T=9, q_pos0=800, n_comp=300, ratio=4, n_heads=n_heads, head_dim=128, relu=relu, seed=55)
    wl = dataclasses.replace(wl, scale=-0.3)
    _check_scores(_run_scores(torch, ds4a, wl), wl)


def test_scores_full_size_sampled(torch, ds4a):
    wl = W.indexer_r4_2048()
    got = _run_scores(torch, ds4a, wl)
    toks = [0, 1, 2, 3, 777, 1024, 2044, 2045, 2046, 2047]
    _check_scores(got[toks], wl, tokens=toks)


def test_scores_strided_output(torch, ds4a):
    wl = _indexer_case(T=7, q_pos0=400, n_comp=150, ratio=4, n_heads=16, head_dim=128, relu=True, seed=50)
    out = torch.full((7, 168), 3.0, dtype=torch.float32, device="cuda")   # 672-byte rows
    ds4a.indexer_scores(wl.layout, dev(torch, wl.q_idx), dev(torch, wl.k_idx), dev(torch, wl.w), scale=wl.scale,
                        relu=True, out=out[:, 4:154])                        # 16-byte aligned start
    o = host(out)
    _check_scores(o[:, 4:154], wl)
    assert (o[:, :4] == 3.0).all() and (o[:, 154:] == 3.0).all()


# ------------------------------------------------------------------ indexer -> attention

def test_indexer_feeds_indexed_attention(torch, ds4a):
    """Scores -> top-k on the GPU, then ds4a_attn_indexed with those lists; the
    lists equal the oracle's selection on the GPU's own scores, and the
    attention output matches the fp64 oracle."""
    L = make_layout(T=24, q_pos0=3000, n_raw=300, raw_pos0=2800, n_comp=750, ratio=4)
    wl = W.draw_indexer("ix_e2e", 60, L, 64, 128, 128)
    att = W.draw("att_e2e", 61, L)
    s = ds4a.indexer_scores(L, dev(torch, wl.q_idx), dev(torch, wl.k_idx), dev(torch, wl.w), scale=wl.scale,
                            relu=True)
    idx = ds4a.indexer_topk(L, s, 128)
    assert np.array_equal(host(idx), ix.topk(L, host(s), 128))
    o = ds4a.attn_indexed(L, dev(torch, att.q), dev(torch, att.k_raw), dev(torch, att.v_raw), dev(torch, att.k_comp),
                          dev(torch, att.v_comp), idx.contiguous())
    want, _ = oracle.attention(L, att.q, att.k_raw, att.v_raw, att.k_comp, att.v_comp, idx=host(idx))
    err = np.abs(host(o).astype(np.float64) - want)
    assert err.max() <= 5e-3 and err.mean() <= 5e-4
