"""CUDA path against the fp64 oracle, element by element (needs a GB300).

Tolerance (fp16 inputs and outputs, fp32 accumulation): max |gpu - oracle| <=
5e-3 and mean |gpu - oracle| <= 5e-4 over every output element compared.
Integer and byte results (block status, padding) must match bit for bit.
"""

import math

import numpy as np
import pytest

import oracle
from mqa_flash_attention_gb300 import synth, workloads as W
from mqa_flash_attention_gb300.workloads import make_layout

pytestmark = pytest.mark.gpu

MAX_ABS = 5e-3
MEAN_ABS = 5e-4


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
    """Every GPU test must leave the device error word clear: a bounded wait
    that ran out would otherwise go unnoticed by tests that check values only."""
    ds4a.device_error_word(clear=True)
    yield
    w = ds4a.device_error_word(clear=True)
    assert w == 0, f"a device wait ran out during this test: error word {w:#010x}"


def dev(torch, a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def assert_close(got, want, what):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err.max() <= MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"


def assert_lse_close(got, want, what):
    got = np.asarray(got, dtype=np.float64)
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: lse finiteness differs"
    if fin.any():
        assert np.abs(got[fin] - want[fin]).max() <= 1e-3, what


def upload(torch, wl):
    return dict(q=dev(torch, wl.q), k_raw=dev(torch, wl.k_raw), v_raw=dev(torch, wl.v_raw),
                k_comp=dev(torch, wl.k_comp) if wl.layout["n_comp"] else None,
                v_comp=dev(torch, wl.v_comp) if wl.layout["n_comp"] else None)


def oracle_out(wl, tokens=None, idx=None, mask=None):
    return oracle.attention(wl.layout, wl.q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp, idx=idx, mask=mask,
                            tokens=tokens)


# ------------------------------------------------------------------ pad

@pytest.mark.parametrize("n", [1, 31, 32, 33, 160, 2175])
def test_pad_matches_oracle_bitwise(torch, ds4a, n):
    src = synth.normal_f16(40 + n, 2, (n + 7, 512))
    want = oracle.pad_rows(src, n)
    got = host(ds4a.pad_kv(dev(torch, src), n))
    assert got.shape == want.shape
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))


def test_pad_in_place_and_strided(torch, ds4a):
    n = 45
    buf = synth.normal_f16(41, 2, (64, 512))
    t = dev(torch, buf)
    ds4a.pad_kv(t[:64], n, dst=t[:64])
    want = oracle.pad_rows(buf, n)
    assert np.array_equal(host(t).view(np.uint16), want.view(np.uint16))
    # rows with a 2048-byte stride (every other row of a wider buffer)
    wide = dev(torch, synth.normal_f16(42, 2, (80, 1024)))
    src = wide[:, :512]
    got = host(ds4a.pad_kv(src, 70))
    assert np.array_equal(got.view(np.uint16), oracle.pad_rows(host(src), 70).view(np.uint16))


# ------------------------------------------------------------------ block status

def _status_layouts():
    out = [(W.tiny().layout, q) for q in (1, 2, 4, 16, 64)]
    out += [(W.decode_r128_32k().layout, 1), (W.prefill_raw_2048().layout, 2),
            (W.prefill_raw_2048().layout, 16), (make_layout(T=2048, q_pos0=30720, n_raw=2175, raw_pos0=30593,
                                                            n_comp=8192, ratio=4), 64)]
    u = iter(synth.uniform(43, 1, 2000))

    def ri(lo, hi):
        return lo + int(next(u) * (hi - lo + 1))

    for _ in range(25):
        out.append((make_layout(T=ri(1, 70), q_pos0=ri(0, 500), n_raw=ri(0, 300), raw_pos0=ri(0, 400),
                                n_comp=ri(0, 200), ratio=(4, 128, 7)[ri(0, 2)], window=ri(1, 200)),
                    (1, 2, 3, 16, 64)[ri(0, 4)]))
    return out


def test_block_status_structural_bitwise(torch, ds4a):
    for L, qt in _status_layouts():
        if oracle.padded_lengths(L) == (0, 0) or L["T"] == 0:
            continue
        want = oracle.block_status(L, qt)
        got = host(ds4a.block_mask(L, qt))
        assert np.array_equal(got, want), (L, qt)


def _random_mask(seed, L, p_open=0.6, p_bias=0.1):
    npr, npc = oracle.padded_lengths(L)
    u = synth.uniform(seed, synth.STREAM_MASK, L["T"] * (npr + npc)).reshape(L["T"], npr + npc)
    m = np.where(u < p_open, 0.0, -np.inf)
    m = np.where((u < p_bias), (u - 0.05) * 10, m)      # a few biased entries in (-0.5, 0.5)
    return m.astype(np.float16)


def test_block_status_dense_mask_bitwise(torch, ds4a):
    L = make_layout(T=37, q_pos0=500, n_raw=150, raw_pos0=0, n_comp=70, ratio=4)
    npr, npc = oracle.padded_lengths(L)
    m = _random_mask(44, L)
    m[:, 0:32] = -np.inf                 # a closed block
    m[:, 64:96] = 0.0                    # a fully open block
    m[5:9, 96:128] = -np.inf
    for qt in (1, 4, 37):
        want = oracle.block_status(L, qt, mask=m)
        got = host(ds4a.block_mask(L, qt, mask=dev(torch, m)))
        assert np.array_equal(got, want), qt
        assert (want == 0).any() and (want == 2).any()


# ------------------------------------------------------------------ prefill

def test_prefill_tiny(torch, ds4a):
    wl = W.tiny()
    d = upload(torch, wl)
    o, lse = ds4a.attn_prefill(wl.layout, d["q"], d["k_raw"], d["v_raw"], want_lse=True)
    want, wlse = oracle_out(wl)
    assert_close(host(o), want, "tiny prefill")
    assert_lse_close(host(lse), wlse, "tiny prefill lse")


def test_prefill_raw_2048_all_tokens(torch, ds4a):
    """Full-size 2048-token raw-only chunk, every output element of every
    token against the oracle (output pre-filled with NaN)."""
    wl = W.prefill_raw_2048()
    d = upload(torch, wl)
    out = torch.full_like(d["q"], float("nan"))
    o, lse = ds4a.attn_prefill(wl.layout, d["q"], d["k_raw"], d["v_raw"], out=out, want_lse=True)
    want, wlse = oracle_out(wl)
    assert_close(host(o), want, "prefill 2048")
    assert_lse_close(host(lse), wlse, "prefill 2048 lse")


def _ragged_cases():
    return [
        make_layout(T=3, q_pos0=5, n_raw=9, raw_pos0=0),                       # windows shorter than 128
        make_layout(T=5, q_pos0=300, n_raw=260, raw_pos0=50, window=128),      # window inside, unaligned
        make_layout(T=2, q_pos0=1000, n_raw=40, raw_pos0=990, n_comp=7, ratio=128),
        make_layout(T=4, q_pos0=999, n_raw=128, raw_pos0=872, n_comp=250, ratio=4),   # 2 compressed tiles
        make_layout(T=3, q_pos0=700, n_raw=300, raw_pos0=400, window=200),     # window > 128: two raw tiles
        make_layout(T=1, q_pos0=64, n_raw=1, raw_pos0=64, window=1),           # single row
        make_layout(T=130, q_pos0=200, n_raw=330, raw_pos0=0, n_comp=50, ratio=4),    # > one wave of tokens
    ]


@pytest.mark.parametrize("case", range(7))
def test_prefill_ragged(torch, ds4a, case):
    L = _ragged_cases()[case]
    wl = W.draw(f"ragged{case}", 50 + case, L)
    d = upload(torch, wl)
    o, lse = ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], want_lse=True)
    want, wlse = oracle_out(wl)
    assert_close(host(o), want, f"ragged {case}")
    assert_lse_close(host(lse), wlse, f"ragged {case} lse")


def _pair_cases():
    """Raw-only layouts with a window of at most 128 and T >= 2: the prefill
    path that serves two consecutive tokens per 128-row tile."""
    return [
        make_layout(T=2, q_pos0=500, n_raw=400, raw_pos0=200),                # one pair, extra row present
        make_layout(T=2, q_pos0=127, n_raw=128, raw_pos0=0),                  # token a's window starts at row 0
        make_layout(T=2, q_pos0=127, n_raw=129, raw_pos0=0),                  # the extra row is row 0
        make_layout(T=7, q_pos0=60, n_raw=100, raw_pos0=0),                   # tiles start below row 0, odd T
        make_layout(T=9, q_pos0=400, n_raw=300, raw_pos0=250, window=37),     # short window: no extra row
        make_layout(T=6, q_pos0=1000, n_raw=40, raw_pos0=950),                # rows end before the tokens
        make_layout(T=311, q_pos0=3000, n_raw=500, raw_pos0=2700),            # > one pair per CTA, odd last token
    ]


@pytest.mark.parametrize("case", range(7))
def test_prefill_pairs(torch, ds4a, case):
    L = _pair_cases()[case]
    wl = W.draw(f"pairs{case}", 90 + case, L)
    d = upload(torch, wl)
    o = torch.full_like(d["q"], float("nan"))
    lse = torch.full((L["T"], 64), float("nan"), dtype=torch.float32, device="cuda")
    ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"], out=o, lse=lse)
    want, wlse = oracle_out(wl)
    assert_close(host(o), want, f"pairs {case}")
    assert_lse_close(host(lse), wlse, f"pairs {case} lse")


def test_prefill_pairs_strided(torch, ds4a):
    """The pair path with Q/O token strides and K/V row strides larger than the packed ones."""
    L = make_layout(T=5, q_pos0=300, n_raw=260, raw_pos0=50)
    wl = W.draw("pairs_strided", 99, L)
    qbig = torch.zeros((5, 72, 512), dtype=torch.float16, device="cuda")
    qbig[:, :64] = dev(torch, wl.q)
    kbig = torch.zeros((260, 640), dtype=torch.float16, device="cuda")
    vbig = torch.zeros((260, 640), dtype=torch.float16, device="cuda")
    kbig[:, :512] = dev(torch, wl.k_raw)
    vbig[:, :512] = dev(torch, wl.v_raw)
    obig = torch.full((5, 66, 512), 7.0, dtype=torch.float16, device="cuda")
    ds4a.attn_prefill(L, qbig[:, :64], kbig[:, :512], vbig[:, :512], out=obig[:, :64])
    want, _ = oracle_out(wl)
    assert_close(host(obig[:, :64]), want, "pairs strided")
    assert bool((obig[:, 64:] == 7.0).all()), "a write landed outside the output rows"


def test_prefill_pairs_output_16_byte_aligned(torch, ds4a):
    """The pair path writes o with 32-byte stores when o and its token stride
    allow them, else with 16-byte ones: here o starts 16 bytes past a 32-byte
    boundary and its token stride is an odd multiple of 16 bytes."""
    L = make_layout(T=7, q_pos0=400, n_raw=300, raw_pos0=200)
    wl = W.draw("pairs_o16", 98, L)
    tok = 64 * 512 + 24                      # elements: 65,584 bytes per token
    flat = torch.full((8 + 7 * tok,), 7.0, dtype=torch.float16, device="cuda")
    out = torch.as_strided(flat, (7, 64, 512), (tok, 512, 1), storage_offset=8)
    assert out.data_ptr() % 32 == 16 and (tok * 2) % 32 == 16
    d = upload(torch, wl)
    ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"], out=out)
    want, _ = oracle_out(wl)
    assert_close(host(out.contiguous()), want, "pairs, 16-byte aligned o")
    mask = torch.ones_like(flat, dtype=torch.bool)
    for t in range(7):
        mask[8 + t * tok: 8 + t * tok + 64 * 512] = False
    assert bool((flat[mask] == 7.0).all()), "a write landed outside the output rows"


def test_prefill_strided_tokens_and_rows(torch, ds4a):
    """Q/O token strides and K/V row strides larger than the packed ones."""
    L = make_layout(T=6, q_pos0=150, n_raw=160, raw_pos0=0, n_comp=40, ratio=4)
    wl = W.draw("strided", 60, L)
    qbig = torch.zeros((6, 80, 512), dtype=torch.float16, device="cuda")
    qbig[:, :64] = dev(torch, wl.q)
    kbig = torch.zeros((160, 768), dtype=torch.float16, device="cuda")
    vbig = torch.zeros((160, 768), dtype=torch.float16, device="cuda")
    kbig[:, :512] = dev(torch, wl.k_raw)
    vbig[:, :512] = dev(torch, wl.v_raw)
    obig = torch.full((6, 70, 512), 7.0, dtype=torch.float16, device="cuda")
    ds4a.attn_prefill(L, qbig[:, :64], kbig[:, :512], vbig[:, :512], dev(torch, wl.k_comp), dev(torch, wl.v_comp),
                      out=obig[:, :64])
    want, _ = oracle_out(wl)
    assert_close(host(obig[:, :64]), want, "strided")
    assert np.all(host(obig[:, 64:]) == 7.0), "wrote outside the output rows"


def test_invisible_rows_do_not_change_output_bitwise(torch, ds4a):
    """Rows outside every window set to +-65504 (finite): bit-identical output."""
    L = make_layout(T=8, q_pos0=400, n_raw=500, raw_pos0=0, n_comp=0)
    wl = W.draw("invis", 61, L)
    d = upload(torch, wl)
    base = host(ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"]))
    k2, v2 = wl.k_raw.copy(), wl.v_raw.copy()
    k2[:400 - 127] = 65504.0           # before the first window
    v2[:400 - 127] = -65504.0
    k2[408:] = -65504.0                # after the last token
    v2[408:] = 65504.0
    got = host(ds4a.attn_prefill(L, d["q"], dev(torch, k2), dev(torch, v2)))
    assert np.array_equal(got.view(np.uint16), base.view(np.uint16))


def test_aliased_k_and_v(torch, ds4a):
    L = make_layout(T=4, q_pos0=300, n_raw=310, raw_pos0=0)
    wl = W.draw("alias", 62, L)
    kv = dev(torch, wl.k_raw)
    got = host(ds4a.attn_prefill(L, dev(torch, wl.q), kv, kv))
    want, _ = oracle.attention(L, wl.q, wl.k_raw, wl.k_raw)
    assert_close(got, want, "k == v")


@pytest.mark.parametrize("name", ["decode_r128_32k", "prefill_raw_2048", "indexed_r4_2048", "decode_long_65536",
                                  "mixed_segments"])
def test_aliased_k_and_v_configs(torch, ds4a, name):
    """One row serving as K and V (the pointers alias, as in an engine that
    stores one KV row): each tile part is loaded once and used by both
    products.  Against the oracle on the same rows used as K and V, on the
    decode, prefill, indexed and long-decode workloads; "mixed_segments"
    aliases the raw rows only (compressed K and V stay distinct)."""
    if name == "decode_r128_32k":
        wl = W.decode_r128_32k()
    elif name == "prefill_raw_2048":
        wl = W.prefill_raw_2048()
    elif name == "indexed_r4_2048":
        wl = W.indexed_r4_2048()
    elif name == "decode_long_65536":
        wl = W.decode_long(65536)
    else:
        wl = W.draw("alias_mixed", 75, make_layout(T=5, q_pos0=40000, n_raw=200, raw_pos0=39873, n_comp=312,
                                                    ratio=128))
    wl.v_raw = wl.k_raw
    if name != "mixed_segments":
        wl.v_comp = wl.k_comp
    L = wl.layout
    kr = dev(torch, wl.k_raw)
    kc = dev(torch, wl.k_comp) if L["n_comp"] else None
    vc = kc if name != "mixed_segments" else dev(torch, wl.v_comp)
    q = dev(torch, wl.q)
    idx = wl.idx if name == "indexed_r4_2048" else None
    want, wlse = oracle_out(wl, idx=idx)
    out = torch.full_like(q, float("nan"))
    if idx is not None:
        o, lse = ds4a.attn_indexed(L, q, kr, kr, kc, vc, dev(torch, idx), out=out, want_lse=True)
    elif L["T"] > 8:
        o, lse = ds4a.attn_prefill(L, q, kr, kr, kc, vc, out=out, want_lse=True)
    else:
        o, lse = ds4a.attn_decode(L, q, kr, kr, kc, vc, out=out, want_lse=True)
    assert_close(host(o), want, f"aliased {name}")
    assert_lse_close(host(lse), wlse, f"aliased {name} lse")
    if L["T"] <= 8:   # the prefill kernel on the same aliased rows
        o2 = ds4a.attn_prefill(L, q, kr, kr, kc, vc)
        assert_close(host(o2), want, f"aliased {name} prefill")


def test_aliased_decode_batch(torch, ds4a):
    """Batched decode with K and V of both segments aliased."""
    from mqa_flash_attention_gb300 import synth
    geo = [(32767, 128, 32640, 256), (5000, 200, 4801, 39), (1000, 60, 941, 7)]
    B, R, C = len(geo), 200, 300
    q = synth.normal_f16(76, synth.STREAM_Q, (B, 64, 512))
    kr = synth.normal_f16(76, synth.STREAM_K_RAW, (B, R, 512))
    kc = synth.normal_f16(76, synth.STREAM_K_COMP, (B, C, 512))
    g = dev(torch, np.array(geo, dtype=np.int32))
    shape = make_layout(T=1, q_pos0=0, n_raw=0, raw_pos0=0, n_comp=0, ratio=128)
    dkr, dkc = dev(torch, kr), dev(torch, kc)
    o = host(ds4a.attn_decode_batch(shape, g, dev(torch, q), dkr, dkr, dkc, dkc))
    for b, (qp, nr, rp, nc) in enumerate(geo):
        L = make_layout(T=1, q_pos0=qp, n_raw=nr, raw_pos0=rp, n_comp=nc, ratio=128)
        want, _ = oracle.attention(L, q[b:b + 1], kr[b, :nr], kr[b, :nr], kc[b, :nc], kc[b, :nc])
        assert_close(o[b:b + 1], want, f"aliased batch seq {b}")


def test_large_score_rescale_path(torch, ds4a):
    """Rows whose scores jump far above the running max in later tiles force
    the lazy reference to move and O to be rescaled (twice for token 0)."""
    L = make_layout(T=2, q_pos0=900, n_raw=129, raw_pos0=772, n_comp=225, ratio=4, window=129)
    wl = W.draw("rescale", 63, L)
    qsum = wl.q[0].astype(np.float32).sum(0)           # scores ~ c * 22.6 for every head of token 0
    k_comp = wl.k_comp.copy()
    k_comp[10] = (0.4 * qsum).astype(np.float16)       # 3rd tile: jump of ~9 (natural log units)
    k_comp[200] = (1.0 * qsum).astype(np.float16)      # 4th tile: jump of ~13 more
    wl.k_comp = k_comp
    d = upload(torch, wl)
    o, lse = ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], want_lse=True)
    want, wlse = oracle_out(wl)
    assert_close(host(o), want, "rescale")
    assert_lse_close(host(lse), wlse, "rescale lse")


# ------------------------------------------------------------------ dense mask

def test_prefill_dense_mask(torch, ds4a):
    L = make_layout(T=40, q_pos0=600, n_raw=300, raw_pos0=0, n_comp=90, ratio=4)
    wl = W.draw("mask", 64, L)
    m = _random_mask(65, L)
    m[3] = -np.inf                     # a token that sees nothing
    d = upload(torch, wl)
    dm = dev(torch, m)
    o, lse = ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], mask=dm,
                               want_lse=True)
    want, wlse = oracle_out(wl, mask=m)
    assert_close(host(o), want, "dense mask")
    assert_lse_close(host(lse), wlse, "dense mask lse")
    # with status bytes: skipped blocks and unread open blocks change nothing
    for qt in (1, 8):
        st = ds4a.block_mask(L, qt, mask=dm)
        o2 = ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], mask=dm, status=st,
                               q_tile=qt)
        assert np.array_equal(host(o2).view(np.uint16), host(o).view(np.uint16)), qt
    ones = torch.ones_like(ds4a.block_mask(L, 8, mask=dm))
    o3 = ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], mask=dm, status=ones,
                           q_tile=8)
    assert np.array_equal(host(o3).view(np.uint16), host(o).view(np.uint16))


def test_dense_mask_of_the_window_equals_structural(torch, ds4a):
    wl = W.tiny()
    L = wl.layout
    vis, _ = oracle.pair_visibility(L)
    m = np.where(vis, 0.0, -np.inf).astype(np.float16)
    d = upload(torch, wl)
    a = host(ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"]))
    b = host(ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"], mask=dev(torch, m)))
    assert_close(b.astype(np.float64), a.astype(np.float64), "mask == window")


def _random_layout(rng):
    ratio = int(rng.choice([4, 128]))
    T = int(rng.integers(1, 25))
    q_pos0 = int(rng.integers(0, 3000))
    n_raw = int(rng.integers(0, 400))
    # raw rows mostly end around the tokens (the window), sometimes before or after them
    raw_pos0 = max(0, q_pos0 + T - n_raw + int(rng.integers(-160, 161)))
    n_comp = int(rng.integers(0, min(600, (q_pos0 + T) // ratio + 3) + 1))
    return make_layout(T=T, q_pos0=q_pos0, n_raw=n_raw, raw_pos0=raw_pos0, n_comp=n_comp, ratio=ratio)


def test_random_layouts_against_oracle(torch, ds4a):
    """Seeded random geometries (token counts, row counts, offsets, both ratios;
    rows past a token's position, empty segments, tokens that see nothing):
    prefill, and decode with a random split count for the short ones."""
    rng = np.random.default_rng(2024)
    for case in range(32):
        L = _random_layout(rng)
        wl = W.draw(f"rand{case}", 300 + case, L)
        d = upload(torch, wl)
        want, wlse = oracle_out(wl)
        o, lse = ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], want_lse=True)
        assert_close(host(o), want, f"random prefill {case} {L}")
        assert_lse_close(host(lse), wlse, f"random prefill lse {case} {L}")
        if L["T"] <= 4:
            splits = int(rng.integers(1, 9))
            o, lse = ds4a.attn_decode(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], n_splits=splits,
                                      want_lse=True)
            assert_close(host(o), want, f"random decode {case} splits={splits} {L}")
            assert_lse_close(host(lse), wlse, f"random decode lse {case} {L}")


# ------------------------------------------------------------------ decode

def test_decode_r128_32k(torch, ds4a):
    wl = W.decode_r128_32k()
    d = upload(torch, wl)
    want, wlse = oracle_out(wl)
    for splits in (0, 1, 2, 3, 5):
        o, lse = ds4a.attn_decode(wl.layout, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"],
                                  n_splits=splits, want_lse=True)
        assert_close(host(o), want, f"decode splits={splits}")
        assert_lse_close(host(lse), wlse, f"decode lse splits={splits}")


@pytest.mark.parametrize("n_comp", W.LONG_DECODE_SIZES)
def test_decode_long(torch, ds4a, n_comp):
    wl = W.decode_long(n_comp)
    d = upload(torch, wl)
    o, lse = ds4a.attn_decode(wl.layout, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], want_lse=True)
    want, wlse = oracle_out(wl)
    assert_close(host(o), want, f"decode N={n_comp}")
    assert_lse_close(host(lse), wlse, f"decode N={n_comp} lse")


def test_decode_equals_last_prefill_row(torch, ds4a):
    L = make_layout(T=4, q_pos0=2000, n_raw=260, raw_pos0=1744, n_comp=15, ratio=128)
    wl = W.draw("dec_vs_pre", 66, L)
    d = upload(torch, wl)
    full = host(ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"]))
    L1 = dict(L, T=1, q_pos0=2003)
    one = host(ds4a.attn_decode(L1, d["q"][3:4], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], n_splits=2))
    err = np.abs(one[0].astype(np.float64) - full[3].astype(np.float64))
    assert err.max() <= 2 * MAX_ABS


def test_calls_on_the_same_buffers_with_other_shapes(torch, ds4a):
    """Calls on the same device buffers with fewer compressed or raw rows,
    then the first shape again: each matches the oracle on exactly the rows it
    names (state carried from one call to the next, such as a tensor map of an
    earlier shape, would read the wrong rows or none)."""
    L0 = make_layout(T=3, q_pos0=9000, n_raw=200, raw_pos0=8850, n_comp=70, ratio=128)
    wl = W.draw("same_bufs", 81, L0)
    d = upload(torch, wl)
    for n_comp, n_raw in ((70, 200), (40, 200), (70, 140), (33, 151), (70, 200)):
        L = dict(L0, n_comp=n_comp, n_raw=n_raw)
        want, _ = oracle.attention(L, wl.q, wl.k_raw[:n_raw], wl.v_raw[:n_raw], wl.k_comp[:n_comp],
                                   wl.v_comp[:n_comp])
        o = ds4a.attn_decode(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], n_splits=3)
        assert_close(host(o), want, f"decode n_comp={n_comp} n_raw={n_raw}")
        o = ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"])
        assert_close(host(o), want, f"prefill n_comp={n_comp} n_raw={n_raw}")


def test_decode_several_tokens(torch, ds4a):
    L = make_layout(T=3, q_pos0=5000, n_raw=200, raw_pos0=4850, n_comp=39, ratio=128)
    wl = W.draw("dec3", 67, L)
    d = upload(torch, wl)
    want, _ = oracle_out(wl)
    for s in (1, 2, 7):
        o = ds4a.attn_decode(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], n_splits=s)
        assert_close(host(o), want, f"decode T=3 splits={s}")


@pytest.mark.parametrize("splits", [5, 17, 40])
def test_decode_empty_splits_ignore_workspace_contents(torch, ds4a, splits):
    """More splits than tiles (two per token here): the extra splits see no
    row and never write their partials, and the merge (the one-dim-per-thread
    form below 17 splits, the warp-split form from 17) must ignore whatever the
    workspace holds there, NaN in this test."""
    L = make_layout(T=3, q_pos0=5000, n_raw=200, raw_pos0=4850, n_comp=39, ratio=128)
    wl = W.draw("dec_empty", 68, L)
    d = upload(torch, wl)
    want, wlse = oracle_out(wl)
    ws = torch.full((ds4a.decode_workspace_bytes(L, splits) // 4,), float("nan"), dtype=torch.float32,
                    device="cuda")
    o, lse = ds4a.attn_decode(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], n_splits=splits,
                              workspace=ws, want_lse=True)
    assert_close(host(o), want, f"decode T=3 splits={splits}")
    assert_lse_close(host(lse), wlse, f"decode T=3 splits={splits} lse")


def test_decode_batch_matches_oracle(torch, ds4a):
    """Seven sequences, each with its own position, row counts and K/V rows, in
    one batched launch; each equals the oracle on its own layout."""
    from mqa_flash_attention_gb300 import synth
    R, C, ratio = 200, 300, 128
    geo = [  # q_pos, n_raw, raw_pos0, n_comp
        (32767, 128, 32640, 256), (5000, 200, 4801, 39), (130, 131, 0, 1), (70, 71, 0, 0),
        (38399, 150, 38250, 299), (38400, 128, 38273, 300), (1000, 60, 941, 7)]
    B = len(geo)
    q = synth.normal_f16(40, synth.STREAM_Q, (B, 64, 512))
    kr = synth.normal_f16(40, synth.STREAM_K_RAW, (B, R, 512))
    vr = synth.normal_f16(40, synth.STREAM_V_RAW, (B, R, 512))
    kc = synth.normal_f16(40, synth.STREAM_K_COMP, (B, C, 512))
    vc = synth.normal_f16(40, synth.STREAM_V_COMP, (B, C, 512))
    g = dev(torch, np.array(geo, dtype=np.int32))
    shape = make_layout(T=1, q_pos0=0, n_raw=0, raw_pos0=0, n_comp=0, ratio=ratio)
    for splits in (0, 1, 3):
        o, lse = ds4a.attn_decode_batch(shape, g, dev(torch, q), dev(torch, kr), dev(torch, vr), dev(torch, kc),
                                        dev(torch, vc), n_splits=splits, want_lse=True)
        o, lse = host(o), host(lse)
        for b, (qp, nr, rp, nc) in enumerate(geo):
            L = make_layout(T=1, q_pos0=qp, n_raw=nr, raw_pos0=rp, n_comp=nc, ratio=ratio)
            want, wlse = oracle.attention(L, q[b:b + 1], kr[b, :nr], vr[b, :nr], kc[b, :nc], vc[b, :nc])
            assert_close(o[b:b + 1], want, f"batch seq {b} splits={splits}")
            assert_lse_close(lse[b:b + 1], wlse, f"batch seq {b} lse")


# ------------------------------------------------------------------ indexed

def test_indexed_ratio4_all_tokens(torch, ds4a):
    """Full-size indexed ratio-4 chunk (2048 tokens, top-512 of 8192 rows),
    every token against the oracle (output pre-filled with NaN)."""
    wl = W.indexed_r4_2048()
    d = upload(torch, wl)
    idx = dev(torch, wl.idx)
    out = torch.full_like(d["q"], float("nan"))
    o, lse = ds4a.attn_indexed(wl.layout, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], idx, out=out,
                               want_lse=True)
    want, wlse = oracle_out(wl, idx=wl.idx)
    assert_close(host(o), want, "indexed")
    assert_lse_close(host(lse), wlse, "indexed lse")


def test_indexed_edge_cases(torch, ds4a):
    L = make_layout(T=7, q_pos0=700, n_raw=140, raw_pos0=600, n_comp=175, ratio=4)
    wl = W.draw("idx_edge", 68, L)
    idx = np.full((7, 200), -1, np.int32)
    idx[0, :3] = [4, 4, 9]                         # duplicates
    idx[1, 50:60] = np.arange(10)                  # -1 around the entries
    idx[2, :] = np.arange(200) % 175               # every row, some twice
    idx[3, 0] = 174
    idx[4, 199] = 0                                # last slot only
    idx[5, :6] = [175, 3, 176, 2 ** 31 - 1, 8, 100000]   # entries past the last row are empty slots
    idx[6, 10:140] = np.arange(175, 305)           # only entries past the last row: raw window alone
    d = upload(torch, wl)
    o, lse = ds4a.attn_indexed(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], dev(torch, idx),
                               want_lse=True)
    want, wlse = oracle_out(wl, idx=idx)
    assert_close(host(o), want, "indexed edges")
    assert_lse_close(host(lse), wlse, "indexed edges lse")
    # entries past the last row behave exactly like -1 (bit-identical output)
    idx_m1 = np.where(idx >= 175, -1, idx).astype(np.int32)
    o2 = ds4a.attn_indexed(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], dev(torch, idx_m1))
    assert np.array_equal(host(o2).view(np.uint16), host(o).view(np.uint16))


def test_indexed_all_available_equals_dense(torch, ds4a):
    """Index lists naming every pooled row once give the dense (ratio rule) result."""
    L = make_layout(T=6, q_pos0=1000, n_raw=200, raw_pos0=850, n_comp=300, ratio=4)
    wl = W.draw("idx_all", 69, L)
    idx = np.full((6, 256), -1, np.int32)
    for t in range(6):
        n = min(300, (1000 + t + 1) // 4)
        assert n <= 256
        idx[t, :n] = np.arange(n)
    d = upload(torch, wl)
    o = host(ds4a.attn_indexed(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], dev(torch, idx)))
    want, _ = oracle_out(wl, idx=idx)
    assert_close(o, want, "indexed all")
    dense = host(ds4a.attn_prefill(L, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"]))
    assert_close(o.astype(np.float64), dense.astype(np.float64), "indexed all vs dense kernel")


# ------------------------------------------------------------------ bounded waits

def test_stuck_wait_ends_as_a_status(torch, ds4a):
    assert ds4a.device_status(clear=True) == ds4a.OK
    ds4a.selftest_wait_timeout(2_000_000)          # 2 ms bound
    assert ds4a.device_error_word(clear=False) == 0x01000000 | 12   # the self test's wait site
    assert ds4a.device_status(clear=True) == ds4a.ERR_TIMEOUT
    assert ds4a.device_status(clear=True) == ds4a.OK
    # the context is still usable
    wl = W.tiny()
    d = upload(torch, wl)
    o = ds4a.attn_prefill(wl.layout, d["q"], d["k_raw"], d["v_raw"])
    assert_close(host(o), oracle_out(wl)[0], "after timeout")
    assert ds4a.device_status() == ds4a.OK


def test_decode_partials_then_merge(torch, ds4a):
    wl = W.decode_long(1024)
    d = upload(torch, wl)
    ws = ds4a.attn_decode_partials(wl.layout, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], n_splits=4)
    out = torch.empty_like(d["q"])
    lse = torch.empty((1, 64), dtype=torch.float32, device="cuda")
    ds4a.attn_decode_merge(wl.layout, ws, n_splits=4, out=out, lse=lse)
    want, wlse = oracle_out(wl)
    assert_close(host(out), want, "partials + merge")
    assert_lse_close(host(lse), wlse, "partials + merge lse")


def test_prepared_decode_equals_call(torch, ds4a):
    """The prepared call (arguments built once, the C entry point called each
    time) gives the same bits as the regular binding, call after call."""
    wl = W.decode_r128_32k()
    d = {k: dev(torch, getattr(wl, k)) for k in ("q", "k_raw", "v_raw", "k_comp", "v_comp")}
    ref = ds4a.attn_decode(wl.layout, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"])
    ws = torch.empty(ds4a.decode_workspace_bytes(wl.layout), dtype=torch.uint8, device="cuda")
    out = torch.full_like(ref, 7.0)
    call = ds4a.prepare_decode(wl.layout, d["q"], d["k_raw"], d["v_raw"], d["k_comp"], d["v_comp"], workspace=ws,
                               out=out)
    for _ in range(3):
        out.fill_(7.0)
        call()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
