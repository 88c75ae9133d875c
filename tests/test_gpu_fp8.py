"""FP8 (E4M3) K/V rows on the GPU (needs a GB300).

* ds4a_quantize_kv_fp8: codes and scales bit for bit against the oracle (the
  fp32 quotients, product and E4M3 rounding are the same operations).
* ds4a_attn_decode_fp8: against the fp64 attention oracle run on the rows'
  values decode(code) * scale, within max abs 5e-3 and mean abs 5e-4.
"""

import numpy as np
import pytest

import oracle
from oracle import fp8 as f8
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


def test_quantize_bitexact(torch, ds4a):
    rng = np.random.default_rng(30)
    x = rng.standard_normal((300, 512)) * rng.uniform(1e-4, 300, (300, 1))
    x[7] = 0.0
    x[8, :] = 0.0
    x[8, 100] = -0.0
    x[8, 5] = 6e-8                     # a lone fp16 subnormal
    x[9] = np.linspace(-65504, 65504, 512)
    x[10, ::3] = -0.0
    x = x.astype(np.float16)
    codes, scales = ds4a.quantize_kv_fp8(dev(torch, x))
    want_c, want_s = f8.quantize_rows(x)
    assert np.array_equal(host(codes), want_c)
    assert np.array_equal(host(scales).view(np.uint32), want_s.view(np.uint32))


def test_quantize_strided(torch, ds4a):
    rng = np.random.default_rng(31)
    x = rng.standard_normal((40, 600)).astype(np.float16)      # row stride 1200 bytes
    xs = dev(torch, x)[:, :512]
    codes = torch.full((40, 528), 9, dtype=torch.uint8, device="cuda")
    ds4a.quantize_kv_fp8(xs, codes=codes[:, :512])
    c = host(codes)
    assert np.array_equal(c[:, :512], f8.quantize_rows(x[:, :512])[0])
    assert (c[:, 512:] == 9).all()


def _fp8_case(torch, ds4a, wl):
    kc, ks = ds4a.quantize_kv_fp8(dev(torch, wl.k_comp))
    vc, vs = ds4a.quantize_kv_fp8(dev(torch, wl.v_comp))
    kd = f8.dequantize_rows(host(kc), host(ks))
    vd = f8.dequantize_rows(host(vc), host(vs))
    want, wlse = oracle.attention(wl.layout, wl.q, wl.k_raw, wl.v_raw, kd, vd)
    return (kc, ks, vc, vs), want, wlse


def _check(got, want, what):
    err = np.abs(np.asarray(got, np.float64) - want)
    assert np.isfinite(got).all(), what
    assert err.max() <= 5e-3 and err.mean() <= 5e-4, f"{what}: max {err.max():.2e} mean {err.mean():.2e}"


@pytest.mark.parametrize("name", ["decode_r128_32k", "long_1024", "ragged"])
def test_decode_fp8_matches_oracle(torch, ds4a, name):
    if name == "decode_r128_32k":
        wl = W.decode_r128_32k()
    elif name == "long_1024":
        wl = W.decode_long(1024)
    else:  # a compressed tail shorter than a tile, several tokens
        wl = W.draw("fp8_ragged", 32, make_layout(T=3, q_pos0=40000, n_raw=150, raw_pos0=39853, n_comp=311,
                                                   ratio=128))
    (kc, ks, vc, vs), want, wlse = _fp8_case(torch, ds4a, wl)
    q, kr, vr = dev(torch, wl.q), dev(torch, wl.k_raw), dev(torch, wl.v_raw)
    for splits in (0, 1, 3):
        o, lse = ds4a.attn_decode_fp8(wl.layout, q, kr, vr, kc, ks, vc, vs, n_splits=splits, want_lse=True)
        _check(host(o), want, f"{name} splits={splits}")
        fin = np.isfinite(wlse)
        assert np.abs(host(lse)[fin] - wlse[fin]).max() <= 1e-3


def test_decode_fp8_full_size(torch, ds4a):
    wl = W.decode_long(262144)
    (kc, ks, vc, vs), want, _ = _fp8_case(torch, ds4a, wl)
    o = ds4a.attn_decode_fp8(wl.layout, dev(torch, wl.q), dev(torch, wl.k_raw), dev(torch, wl.v_raw), kc, ks, vc, vs)
    _check(host(o), want, "fp8 decode N=262144")
