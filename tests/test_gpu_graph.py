"""Recorded call sequences (ds4a_graph_begin / _end / _launch) on a GB300.

A recording captures the kernels of the library calls made on one stream;
each replay runs them on the recorded buffers with whatever those buffers hold
then.  The tests replay recordings on fresh input contents and compare every
result with the fp64 oracle on those inputs (max abs 5e-3, mean abs 5e-4,
log-sum-exp within 1e-3) and, bit for bit, with an eager call of the same
entry point on the same buffers.  Outputs are pre-filled with NaN before each
replay, so a replay that skipped a kernel cannot pass on stale values.
"""

import ctypes

import numpy as np
import pytest

import oracle
from mqa_flash_attention_gb300 import workloads as W
from mqa_flash_attention_gb300.workloads import make_layout

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 5e-3, 5e-4, 1e-3


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


def _close(got, want, what):
    got = np.asarray(got.detach().cpu().numpy(), dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - want)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, f"{what}: max {err.max():.2e} mean {err.mean():.2e}"


def _lse_close(got, want, what):
    got = got.detach().cpu().numpy().astype(np.float64)
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: lse finiteness"
    assert np.abs(got[fin] - want[fin]).max() <= LSE_ABS, what


def _fill(torch, bufs, wl, names, stream):
    with torch.cuda.stream(stream):
        for b, nm in zip(bufs, names):
            b.copy_(torch.from_numpy(np.ascontiguousarray(getattr(wl, nm))))


DECODE = ("q", "k_raw", "v_raw", "k_comp", "v_comp")


def test_recorded_decode_replays_on_new_contents(torch, ds4a):
    """The 32K-context decode step (split-KV partials and merge) recorded once
    on a side stream, then replayed for three input sets copied into the
    recorded buffers.  Recording runs nothing."""
    wls = [W.decode_r128_32k(), W.draw("graph_decode_b", 81, dict(W.decode_r128_32k().layout))]
    wls.append(wls[0])
    L = wls[0].layout
    s = torch.cuda.Stream()
    bufs = [torch.empty(getattr(wls[0], nm).shape, dtype=torch.float16, device="cuda") for nm in DECODE]
    ns = ds4a.decode_default_splits(L)
    ws = torch.empty(ds4a.decode_workspace_bytes(L, ns), dtype=torch.uint8, device="cuda")
    out = torch.full(bufs[0].shape, float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((L["T"], 64), float("nan"), dtype=torch.float32, device="cuda")
    eager = torch.empty_like(out)
    torch.cuda.synchronize()
    g = ds4a.Graph(s)
    with g:
        ds4a.attn_decode(L, *bufs, n_splits=ns, workspace=ws, out=out, lse=lse, stream=s)
    s.synchronize()
    assert torch.isnan(out).all() and torch.isnan(lse).all(), "recording ran kernels"
    for i, wl in enumerate(wls):
        _fill(torch, bufs, wl, DECODE, s)
        with torch.cuda.stream(s):
            out.fill_(float("nan"))
            lse.fill_(float("nan"))
        g()
        s.synchronize()
        want, wlse = oracle.attention(L, wl.q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp)
        _close(out, want, f"replay {i}")
        _lse_close(lse, wlse, f"replay {i}")
        ds4a.attn_decode(L, *bufs, n_splits=ns, workspace=ws, out=eager, stream=s)
        s.synchronize()
        assert torch.equal(eager, out), f"replay {i} differs from an eager call"
    g.close()
    g.close()  # a second close is a no-op


def test_recorded_sequence_skips_a_refused_call(torch, ds4a):
    """A raw-row prefill (the two-token kernel) and a decode recorded in one
    graph, with a call the library refuses between them (no layout): the
    refused call returns its status and records nothing; each replay gives
    both results.  The graph is replayed on a second stream too."""
    wp = W.draw("graph_prefill", 82, make_layout(T=37, q_pos0=700, n_raw=300, raw_pos0=500))
    wd = W.draw("graph_decode_c", 83, make_layout(T=3, q_pos0=9000, n_raw=131, raw_pos0=8873, n_comp=70,
                                                   ratio=128))
    s, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    pb = [torch.empty(getattr(wp, nm).shape, dtype=torch.float16, device="cuda") for nm in DECODE[:3]]
    db = [torch.empty(getattr(wd, nm).shape, dtype=torch.float16, device="cuda") for nm in DECODE]
    po = torch.empty(pb[0].shape, dtype=torch.float16, device="cuda")
    plse = torch.empty((wp.layout["T"], 64), dtype=torch.float32, device="cuda")
    do = torch.empty(db[0].shape, dtype=torch.float16, device="cuda")
    ns = 5
    ws = torch.empty(ds4a.decode_workspace_bytes(wd.layout, ns), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    g = ds4a.Graph(s)
    with g:
        ds4a.attn_prefill(wp.layout, *pb, out=po, lse=plse, stream=s)
        st = ds4a.lib().ds4a_attn_decode(None, None, 0, None, 0, ctypes.c_void_p(s.cuda_stream))
        assert st == ds4a.ERR_INVALID_ARG
        ds4a.attn_decode(wd.layout, *db, n_splits=ns, workspace=ws, out=do, stream=s)
    want_p, wlse_p = oracle.attention(wp.layout, wp.q, wp.k_raw, wp.v_raw, None, None)
    want_d, _ = oracle.attention(wd.layout, wd.q, wd.k_raw, wd.v_raw, wd.k_comp, wd.v_comp)
    _fill(torch, pb, wp, DECODE[:3], s)
    _fill(torch, db, wd, DECODE, s)
    for rs in (s, s2):
        with torch.cuda.stream(s):
            for t in (po, plse, do):
                t.fill_(float("nan"))
        s.synchronize()
        g(rs)
        rs.synchronize()
        _close(po, want_p, "recorded prefill")
        _lse_close(plse, wlse_p, "recorded prefill")
        _close(do, want_d, "recorded decode")
    g.close()


def test_recording_needs_a_created_stream(torch, ds4a):
    """The legacy default stream cannot be recorded; the binding refuses None."""
    lib = ds4a.lib()
    assert lib.ds4a_graph_begin(None) == ds4a.ERR_INVALID_ARG
    with pytest.raises(ValueError):
        ds4a.Graph(None)
