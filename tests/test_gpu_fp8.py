"""FP8 (E4M3) K/V rows on the GPU (needs a GB300).

* ds4a_quantize_kv_fp8: codes and scales bit for bit against the oracle (the
  fp32 quotients, product and E4M3 rounding are the same operations).
* ds4a_attn_decode_fp8 / _fp8kv, ds4a_attn_prefill_fp8kv and
  ds4a_attn_indexed_fp8kv: against the
  fp64 attention oracle run on the rows' values decode(code) * scale, within
  max abs 5e-3 and mean abs 5e-4.  The codes and scales the GPU reads are the
  oracle's own quantisation of the rows (uploaded), so no expected value
  comes from the CUDA path.
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


def _quantized(torch, rows):
    """The oracle's E4M3 codes and scales of fp16 rows, on the device, and the
    rows' values decode(code) * scale (float64) for the oracle."""
    codes, scales = f8.quantize_rows(rows)
    return dev(torch, codes), dev(torch, scales), f8.dequantize_rows(codes, scales)


def _fp8_case(torch, ds4a, wl):
    kc, ks, kd = _quantized(torch, wl.k_comp)
    vc, vs, vd = _quantized(torch, wl.v_comp)
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


# ------------------------------------------------------------------ E4M3 raw rows too

def _fp8kv_case(torch, wl, raw_fp8=True):
    """Codes and scales of the compressed rows and, with raw_fp8, of the raw
    rows; the oracle's result over the rows' decoded values."""
    L = wl.layout
    ops = {}
    kr, vr = wl.k_raw, wl.v_raw
    if raw_fp8 and L["n_raw"]:
        ops["k_raw"], ops["k_raw_scale"], kr = _quantized(torch, wl.k_raw)
        ops["v_raw"], ops["v_raw_scale"], vr = _quantized(torch, wl.v_raw)
    else:
        ops["k_raw"], ops["v_raw"] = dev(torch, wl.k_raw), dev(torch, wl.v_raw)
    kc = vc = None
    if L["n_comp"]:
        ops["k_comp"], ops["k_comp_scale"], kc = _quantized(torch, wl.k_comp)
        ops["v_comp"], ops["v_comp_scale"], vc = _quantized(torch, wl.v_comp)
    else:
        ops["k_comp"] = ops["v_comp"] = None
    want, wlse = oracle.attention(L, wl.q, kr, vr, kc, vc)
    return ops, want, wlse


def _call(ds4a, fn, wl, q, ops, **kw):
    return fn(wl.layout, q, ops["k_raw"], ops["v_raw"], ops["k_comp"], ops["v_comp"],
              k_comp_scale=ops.get("k_comp_scale"), v_comp_scale=ops.get("v_comp_scale"),
              k_raw_scale=ops.get("k_raw_scale"), v_raw_scale=ops.get("v_raw_scale"), **kw)


@pytest.mark.parametrize("name", ["decode_r128_32k", "long_8192", "ragged_t3", "raw_only"])
def test_decode_fp8kv_raw_rows_too(torch, ds4a, name):
    """Decode with every K/V row in E4M3 (raw and compressed), several split
    counts, against the oracle over the decoded rows; outputs start as NaN."""
    if name == "decode_r128_32k":
        wl = W.decode_r128_32k()
    elif name == "long_8192":
        wl = W.decode_long(8192)
    elif name == "ragged_t3":
        wl = W.draw("fp8kv_ragged", 33, make_layout(T=3, q_pos0=40000, n_raw=150, raw_pos0=39853, n_comp=311,
                                                     ratio=128))
    else:
        wl = W.draw("fp8kv_raw", 34, make_layout(T=2, q_pos0=600, n_raw=300, raw_pos0=400))
    ops, want, wlse = _fp8kv_case(torch, wl)
    q = dev(torch, wl.q)
    for splits in (0, 1, 3):
        out = torch.full_like(q, float("nan"))
        o, lse = _call(ds4a, ds4a.attn_decode_fp8kv, wl, q, ops, n_splits=splits, out=out, want_lse=True)
        _check(host(o), want, f"{name} splits={splits}")
        fin = np.isfinite(wlse)
        assert np.abs(host(lse)[fin] - wlse[fin]).max() <= 1e-3


def test_decode_fp8kv_full_size_raw_fp16(torch, ds4a):
    """256K compressed E4M3 rows with fp16 raw rows, through the fp8kv entry."""
    wl = W.decode_long(262144)
    ops, want, _ = _fp8kv_case(torch, wl, raw_fp8=False)
    o = _call(ds4a, ds4a.attn_decode_fp8kv, wl, dev(torch, wl.q), ops)
    _check(host(o), want, "fp8kv decode N=262144")


@pytest.mark.parametrize("name", ["tiny", "prefill_raw_2048", "ragged_mixed", "comp_fp8_raw_fp16"])
def test_prefill_fp8kv(torch, ds4a, name):
    """Structural prefill over E4M3 rows against the oracle over the decoded
    rows, every token (the 2048-token chunk included)."""
    raw_fp8 = True
    if name == "tiny":
        wl = W.tiny()
    elif name == "prefill_raw_2048":
        wl = W.prefill_raw_2048()
    elif name == "ragged_mixed":
        wl = W.draw("fp8kv_pre", 35, make_layout(T=37, q_pos0=999, n_raw=170, raw_pos0=862, n_comp=250, ratio=4))
    else:
        wl = W.draw("fp8kv_pre2", 36, make_layout(T=9, q_pos0=5000, n_raw=200, raw_pos0=4850, n_comp=39,
                                                   ratio=128))
        raw_fp8 = False
    ops, want, wlse = _fp8kv_case(torch, wl, raw_fp8=raw_fp8)
    q = dev(torch, wl.q)
    out = torch.full_like(q, float("nan"))
    o, lse = _call(ds4a, ds4a.attn_prefill_fp8kv, wl, q, ops, out=out, want_lse=True)
    _check(host(o), want, f"prefill fp8kv {name}")
    fin = np.isfinite(wlse)
    assert np.abs(host(lse)[fin] - wlse[fin]).max() <= 1e-3


# Raw-only layouts with a window of at most 128 and T >= 2 (the shapes the
# fp16 prefill serves two tokens per tile): one pair with and without the
# extra row, the extra row at row 0, tiles below row 0 with odd T, a short
# window, rows ending before the tokens, more pairs than CTAs with an odd last
# token.
_PAIR_LAYOUTS = [
    dict(T=2, q_pos0=500, n_raw=400, raw_pos0=200),
    dict(T=2, q_pos0=127, n_raw=128, raw_pos0=0),
    dict(T=2, q_pos0=127, n_raw=129, raw_pos0=0),
    dict(T=7, q_pos0=60, n_raw=100, raw_pos0=0),
    dict(T=9, q_pos0=400, n_raw=300, raw_pos0=250, window=37),
    dict(T=6, q_pos0=1000, n_raw=40, raw_pos0=950),
    dict(T=311, q_pos0=3000, n_raw=500, raw_pos0=2700),
]


@pytest.mark.parametrize("path", ["pairs", "one_token"])
@pytest.mark.parametrize("case", range(len(_PAIR_LAYOUTS)))
def test_prefill_fp8kv_pairs(torch, ds4a, case, path):
    """E4M3 raw rows on those layouts against the oracle over the decoded
    rows, through the workspace call (rows decoded once, pair kernel) and the
    call without one (one-token kernel); outputs and log-sum-exp start as
    NaN, and the workspace starts as NaN rows."""
    wl = W.draw(f"fp8_pairs{case}", 120 + case, make_layout(**_PAIR_LAYOUTS[case]))
    ops, want, wlse = _fp8kv_case(torch, wl, raw_fp8=True)
    q = dev(torch, wl.q)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((wl.layout["T"], 64), float("nan"), dtype=torch.float32, device="cuda")
    ws = False
    if path == "pairs":
        need = ds4a.prefill_fp8kv_workspace_size(wl.layout)
        assert need > 0
        ws = torch.full((need // 2,), float("nan"), dtype=torch.float16, device="cuda")
    o, lse = _call(ds4a, ds4a.attn_prefill_fp8kv, wl, q, ops, out=out, lse=lse, workspace=ws)
    _check(host(o), want, f"fp8 pairs {case} {path}")
    got = host(lse)
    fin = np.isfinite(wlse)
    assert np.array_equal(np.isfinite(got), fin), f"fp8 pairs {case} {path}: lse finiteness"
    assert np.abs(got[fin] - wlse[fin]).max() <= 1e-3


def test_prefill_fp8kv_padded_code_rows(torch, ds4a):
    """E4M3 raw rows at a 1024-byte row stride (codes in the first 512 bytes,
    the rest 0xFF, an E4M3 NaN code that must never be read) through the
    workspace call, the workspace pre-filled with NaN rows: against the oracle
    over the decoded rows.  A workspace one byte short is refused."""
    wl = W.draw("fp8_padded", 131, make_layout(T=45, q_pos0=900, n_raw=400, raw_pos0=700))
    L = wl.layout
    ops, dec = {}, {}
    for nm in ("k_raw", "v_raw"):
        codes, scales = f8.quantize_rows(getattr(wl, nm))
        padded = np.full((codes.shape[0], 1024), 0xFF, dtype=np.uint8)
        padded[:, :512] = codes
        ops[nm] = dev(torch, padded)[:, :512]
        ops[nm + "_scale"] = dev(torch, scales)
        dec[nm] = f8.dequantize_rows(codes, scales)
    assert ops["k_raw"].stride(0) == 1024
    want, wlse = oracle.attention(L, wl.q, dec["k_raw"], dec["v_raw"], None, None)
    q = dev(torch, wl.q)
    need = ds4a.prefill_fp8kv_workspace_size(L)
    assert need == (945 - 900 + 127) * 2 * 1024  # positions 773 .. 944 are seen
    ws = torch.full((need // 2,), float("nan"), dtype=torch.float16, device="cuda")
    out = torch.full_like(q, float("nan"))
    o, lse = ds4a.attn_prefill_fp8kv(L, q, ops["k_raw"], ops["v_raw"], k_raw_scale=ops["k_raw_scale"],
                                     v_raw_scale=ops["v_raw_scale"], workspace=ws, out=out, want_lse=True)
    _check(host(o), want, "fp8 padded code rows")
    fin = np.isfinite(wlse)
    assert np.abs(host(lse)[fin] - wlse[fin]).max() <= 1e-3
    short = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(ds4a.Ds4aError) as e:
        ds4a.attn_prefill_fp8kv(L, q, ops["k_raw"], ops["v_raw"], k_raw_scale=ops["k_raw_scale"],
                                v_raw_scale=ops["v_raw_scale"], workspace=short, out=out)
    assert e.value.status == ds4a.ERR_WORKSPACE


def _indexed_fp8(torch, ds4a, wl, idx, raw_fp8):
    """E4M3 indexed attention (listed compressed rows as codes; raw rows as
    codes too with raw_fp8) against the oracle over the decoded rows, the
    outputs pre-filled with NaN; returns the GPU output."""
    L = wl.layout
    ops = {}
    kr, vr = wl.k_raw, wl.v_raw
    if raw_fp8:
        ops["k_raw"], ops["k_raw_scale"], kr = _quantized(torch, wl.k_raw)
        ops["v_raw"], ops["v_raw_scale"], vr = _quantized(torch, wl.v_raw)
    else:
        ops["k_raw"], ops["v_raw"] = dev(torch, wl.k_raw), dev(torch, wl.v_raw)
    kc_codes, kcs, kc = _quantized(torch, wl.k_comp)
    vc_codes, vcs, vc = _quantized(torch, wl.v_comp)
    want, wlse = oracle.attention(L, wl.q, kr, vr, kc, vc, idx=idx)
    q = dev(torch, wl.q)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((L["T"], 64), float("nan"), dtype=torch.float32, device="cuda")
    ds4a.attn_indexed_fp8kv(L, q, ops["k_raw"], ops["v_raw"], kc_codes, vc_codes, dev(torch, idx),
                            k_comp_scale=kcs, v_comp_scale=vcs, k_raw_scale=ops.get("k_raw_scale"),
                            v_raw_scale=ops.get("v_raw_scale"), out=out, lse=lse)
    got = host(out)
    _check(got, want, f"indexed fp8 {wl.name}")
    gl = host(lse)
    fin = np.isfinite(wlse)
    assert np.array_equal(np.isfinite(gl), fin), "indexed fp8: lse finiteness"
    assert np.abs(gl[fin] - wlse[fin]).max() <= 1e-3
    return got


@pytest.mark.parametrize("raw_fp8", [False, True])
def test_indexed_fp8kv_all_tokens(torch, ds4a, raw_fp8):
    """The full indexed ratio-4 chunk (2048 tokens, top-512 of 8192 rows) over
    E4M3 compressed rows (and E4M3 raw rows), every token against the oracle."""
    wl = W.indexed_r4_2048()
    _indexed_fp8(torch, ds4a, wl, wl.idx, raw_fp8)


def test_indexed_fp8kv_edge_cases(torch, ds4a):
    """Duplicates, -1 around entries, every row, entries past the last row
    (empty slots), lists with no valid entry; E4M3 raw and compressed rows."""
    L = make_layout(T=7, q_pos0=700, n_raw=140, raw_pos0=600, n_comp=175, ratio=4)
    wl = W.draw("idx_fp8_edge", 69, L)
    idx = np.full((7, 200), -1, np.int32)
    idx[0, :3] = [4, 4, 9]
    idx[1, 50:60] = np.arange(10)
    idx[2, :] = np.arange(200) % 175
    idx[3, 0] = 174
    idx[4, 199] = 0
    idx[5, :6] = [175, 3, 176, 2 ** 31 - 1, 8, 100000]
    idx[6, 10:140] = np.arange(175, 305)
    _indexed_fp8(torch, ds4a, wl, idx, raw_fp8=True)
