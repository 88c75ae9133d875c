"""Compressor kernel against the compressor oracle (needs a GB300).

* The state after each call is compared bit for bit (the kernel copies fp32
  rows).
* Pooled rows: fp32 arithmetic, rounded to fp16.  With B = sum_i p_i |kv_i|
  (the pooling of |kv| with the same weights) and Delta the spread of the
  span's scores, each weight carries at most (Delta + 3) roundings of fp32 and
  each sum at most (ratio + 8); the test allows
      2^-11 |want| + 2^-25 + 4 (ratio + 8 + Delta) 2^-24 B,
  the first two terms being the fp16 rounding of the result.
"""

import numpy as np
import pytest

from oracle import compressor as cm
from mqa_flash_attention_gb300 import workloads as W

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


def dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def check_rows(got, kv, s, ratio):
    """got: fp16 [n_out, width]; kv, s: the rows of the completed spans."""
    want = cm.pool(kv, s, ratio)
    bound = cm.pool(np.abs(np.asarray(kv, np.float64)), s, ratio)
    assert got.shape == want.shape
    spread = float(np.max(s) - np.min(s)) if len(s) else 0.0
    tol = 2.0 ** -11 * np.abs(want) + 2.0 ** -25 + 4 * (ratio + 8 + spread) * 2.0 ** -24 * bound
    err = np.abs(got.astype(np.float64) - want)
    assert (err <= tol).all(), f"max err {err.max():.3e}, worst ratio {(err / tol).max():.2f}"
    return err


class GpuState:
    def __init__(self, torch, ratio, width, rows=None):
        rows = max(ratio - 1, 1) if rows is None else rows
        # a recognisable fill: rows past the state's count must never be read
        self.kv = torch.full((rows, width), float("nan"), dtype=torch.float32, device="cuda")
        self.s = torch.full((rows, width), float("nan"), dtype=torch.float32, device="cuda")
        self.n = 0


def run_stream(torch, ds4a, wl, steps, width):
    """Feeds wl's rows in chunks of the given sizes through one GPU state and
    the oracle's; compares every call."""
    ratio = wl.ratio
    st = GpuState(torch, ratio, width)
    o_kv, o_s = np.zeros((0, width)), np.zeros((0, width))
    i = 0
    for n in steps:
        kv, s = wl.kv[i:i + n], wl.score[i:i + n]
        got, st.n = ds4a.compress_append(dev(torch, kv), dev(torch, s), st.kv, st.s, st.n, ratio)
        want_n = (len(o_kv) + n) // ratio
        span_kv = np.concatenate([o_kv, kv])[:want_n * ratio]
        span_s = np.concatenate([o_s, s])[:want_n * ratio]
        check_rows(host(got), span_kv, span_s, ratio)
        _, o_kv, o_s = cm.append(o_kv, o_s, kv, s, ratio)
        assert st.n == len(o_kv)
        assert np.array_equal(host(st.kv[:st.n]).astype(np.float64), o_kv)
        assert np.array_equal(host(st.s[:st.n]).astype(np.float64), o_s)
        i += n
    return i


@pytest.mark.parametrize("ratio,width", [(4, 512), (128, 512), (4, 128), (1, 512), (7, 132), (16, 64), (1000, 36)])
def test_one_call_from_empty_state(torch, ds4a, ratio, width):
    n = 2048 if ratio <= 128 else 2 * ratio + 5
    wl = W.draw_compressor(f"c{ratio}_{width}", 70 + ratio, n, width, ratio)
    run_stream(torch, ds4a, wl, [n], width)


def test_full_size_prefill_ratio4(torch, ds4a):
    wl = W.compressor_prefill(4)
    run_stream(torch, ds4a, wl, [2048], 512)


def test_full_size_prefill_ratio128(torch, ds4a):
    wl = W.compressor_prefill(128)
    run_stream(torch, ds4a, wl, [2048], 512)


@pytest.mark.parametrize("ratio", [4, 128, 5])
def test_streaming_calls(torch, ds4a, ratio):
    # prefill chunks of ragged sizes, then one-token decode steps across several boundaries
    steps = [3, 0, 130, 1, 257, ratio - 1, 1] + [1] * (2 * ratio + 3) + [ratio, 2 * ratio + 1]
    wl = W.draw_compressor(f"stream{ratio}", 80 + ratio, sum(steps), 512, ratio)
    run_stream(torch, ds4a, wl, steps, 512)


def test_state_nearly_full_then_one_token(torch, ds4a):
    # decode: 127 positions wait in the state, the 128th completes the span
    wl = W.draw_compressor("nearly_full", 90, 128, 512, 128)
    run_stream(torch, ds4a, wl, [127, 1], 512)


def test_score_extremes(torch, ds4a):
    # wide score spread: one position dominates most dimensions; equal scores in others
    wl = W.draw_compressor("extremes", 91, 512, 256, 8, score_std=40.0)
    wl.score[:, :16] = 0.5
    run_stream(torch, ds4a, wl, [512], 256)


def test_strided_rows_and_output(torch, ds4a):
    ratio, width = 4, 128
    wl = W.draw_compressor("strided", 92, 70, width, ratio)
    big_kv = torch.zeros((70, width + 12), dtype=torch.float32, device="cuda")
    big_s = torch.zeros((70, width + 12), dtype=torch.float32, device="cuda")
    big_kv[:, 4:4 + width] = dev(torch, wl.kv)
    big_s[:, 4:4 + width] = dev(torch, wl.score)
    st_kv = torch.zeros((ratio - 1, width + 8), dtype=torch.float32, device="cuda")
    st_s = torch.zeros((ratio - 1, width + 8), dtype=torch.float32, device="cuda")
    out = torch.full((20, width + 24), 9.0, dtype=torch.float16, device="cuda")
    got, n = ds4a.compress_append(big_kv[:, 4:4 + width], big_s[:, 4:4 + width], st_kv[:, :width], st_s[:, :width],
                                  0, ratio, out=out[:, 8:8 + width])
    assert n == 2
    o = host(out)
    check_rows(o[:17, 8:8 + width], wl.kv[:68], wl.score[:68], ratio)
    assert (o[:, :8] == 9.0).all() and (o[:, 8 + width:] == 9.0).all() and (o[17:] == 9.0).all()
    assert np.array_equal(host(st_kv[:2, :width]), wl.kv[68:])
    assert (host(st_kv[:, width:]) == 0).all() and (host(st_kv[2:]) == 0).all()


def test_arguments_are_checked(torch, ds4a):
    lib = ds4a.lib()
    assert lib.ds4a_compress_rows(3, 6, 4) == 2
    assert lib.ds4a_compress_rows(4, 1, 4) == -1
    kv = torch.zeros((8, 64), dtype=torch.float32, device="cuda")
    st = torch.zeros((3, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        ds4a.compress_append(kv, kv, st, st, 4, 4)       # n_state must be < ratio
    with pytest.raises(ds4a.Ds4aError):
        ds4a.compress_append(kv[:, :62], kv[:, :62], st[:, :62], st[:, :62], 0, 4)   # width % 4
