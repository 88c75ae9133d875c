"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments before touching CUDA."""

import ctypes
import os
import re

import pytest

from mqa_flash_attention_gb300 import build as ds4a_build
from mqa_flash_attention_gb300 import ds4a

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ds4a.h")


@pytest.fixture(scope="module")
def lib():
    ds4a_build.build()
    return ds4a.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ds4a_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("ds4a_pad_kv", "ds4a_block_mask", "ds4a_attn_prefill", "ds4a_attn_decode", "ds4a_attn_indexed"):
        assert n in names


def test_header_is_plain_c(tmp_path):
    """The boundary header compiles as ISO C99 (no C++ or CUDA types), and a C
    program that takes the address of every declared function links against
    the library."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = tmp_path / "uses_header.c"
    src.write_text('#include "ds4a.h"\n#include <stddef.h>\ntypedef void (*fn)(void);\n'
                   "fn table[] = {\n" + ",\n".join(f"  (fn)&{n}" for n in names) + "\n};\n"
                   "int main(void) { return table[0] == NULL; }\n")
    ds4a_build.build()
    libdir = os.path.dirname(ds4a._LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), "-c", str(src), "-o", str(tmp_path / "u.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([cc, str(tmp_path / "u.o"), "-o", str(tmp_path / "u"), "-L", libdir, "-lds4a",
                        "-Wl,--allow-shlib-undefined"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    for s in range(6):
        assert ds4a.status_string(s)
    assert ds4a.status_string(99) == "unknown status"
    # 0.2: the decode workspace holds fp16 normalised partials (0.1 held fp32 sums)
    assert ds4a.version() == "ds4a 0.2 sm_103a"
    assert ds4a.last_cuda_error() == ""  # no CUDA call has failed on this thread


def _layout(**kw):
    base = dict(T=4, q_pos0=100, n_raw=50, raw_pos0=60, n_comp=0, ratio=128, window=128, scale=0.0441941738)
    base.update(kw)
    return ds4a.make_layout(base)


def test_block_count(lib):
    assert ds4a.block_count(_layout(n_raw=0, n_comp=0)) == 0
    assert ds4a.block_count(_layout(n_raw=1, n_comp=0)) == 1
    assert ds4a.block_count(_layout(n_raw=32, n_comp=33)) == 1 + 2
    assert ds4a.block_count(_layout(n_raw=2175, n_comp=8192)) == 68 + 256
    assert lib.ds4a_block_count(None) == -1


def test_decode_workspace_size(lib):
    L = _layout(T=3, n_comp=1000, ratio=128)
    per_split = 64 * (512 * 2 + 8)
    assert lib.ds4a_attn_decode_workspace_size(ctypes.byref(L), 5) == 3 * 5 * per_split
    assert lib.ds4a_attn_decode_workspace_size(None, 5) == 0


def test_default_split_count_is_the_fewest_with_the_shortest_chain(lib):
    """Without a GPU the library assumes 148 SMs.  For T tokens of n tiles
    each, s0 = min(ceil(148 / T), n) splits give a longest range of
    ceil(n / s0) tiles; the default is the fewest splits with no longer a
    range (one fewer split would lengthen it).  Tiles are 64 rows when every
    (token, split) item of 64-row tiles fits on its own SM and a token has at
    most 32 of them, else 128 rows."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("the SM count of a present GPU replaces the 148 assumed here")
    import numpy as np
    rng = np.random.default_rng(7)
    cdiv = lambda a, b: -(-a // b)  # noqa: E731
    for _ in range(400):
        T = int(rng.choice([1, 1, 1, 2, 3, 5, 8, 17, 64, 200]))
        n_raw = int(rng.integers(0, 400))
        n_comp = int(rng.integers(0, 70000)) if rng.random() < 0.7 else int(rng.integers(0, 600))
        window = int(rng.integers(1, 300))
        if n_raw + n_comp == 0:
            n_comp = 1
        L = _layout(T=T, q_pos0=10 ** 7, n_raw=n_raw, raw_pos0=10 ** 7 - n_raw + 1, n_comp=n_comp, ratio=128,
                    window=window)
        raw = min(window, n_raw)
        tiles = lambda rows: cdiv(raw, rows) + cdiv(n_comp, rows)  # noqa: E731
        half = 2 * tiles(128)
        n = tiles(64) if (half <= 32 and half * T <= 148) else tiles(128)
        got = lib.ds4a_attn_decode_default_splits(ctypes.byref(L))
        s0 = min(cdiv(148, T), n)
        assert 1 <= got <= s0, (T, n, got)
        assert cdiv(n, got) == cdiv(n, s0), (T, n, got)
        if got > 1:
            assert cdiv(n, got - 1) > cdiv(n, s0), (T, n, got)


FAKE = ctypes.c_void_p(1 << 20)       # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p((1 << 20) + 8)


def _tensors(**kw):
    base = dict(q=FAKE, q_tok_stride=65536, k_raw=FAKE, v_raw=FAKE, raw_row_stride=1024, k_comp=None, v_comp=None,
                comp_row_stride=1024, o=FAKE, o_tok_stride=65536, lse=None)
    base.update(kw)
    return ds4a.Tensors(**base)


def _prefill(lib, L, X):
    return lib.ds4a_attn_prefill(ctypes.byref(L), ctypes.byref(X), None, 0, None, 1, None)


@pytest.mark.parametrize("bad", [
    dict(T=-1), dict(q_pos0=-3), dict(n_raw=-1), dict(window=0), dict(n_comp=5, ratio=0),
    dict(scale=float("inf")), dict(scale=float("nan")), dict(q_pos0=2**31 - 2),
])
def test_bad_layout_is_rejected(lib, bad):
    assert _prefill(lib, _layout(**bad), _tensors()) == ds4a.ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [
    dict(q=None), dict(q=MISALIGNED), dict(q_tok_stride=65535), dict(q_tok_stride=4096),
    dict(o=None), dict(o_tok_stride=65536 + 8), dict(k_raw=None), dict(v_raw=MISALIGNED),
    dict(raw_row_stride=1000), dict(raw_row_stride=1032), dict(lse=ctypes.c_void_p((1 << 20) + 2)),
])
def test_bad_tensors_are_rejected(lib, bad):
    assert _prefill(lib, _layout(), _tensors(**bad)) == ds4a.ERR_INVALID_ARG


def test_compressed_rows_need_pointers(lib):
    L = _layout(n_comp=10, ratio=4)
    assert _prefill(lib, L, _tensors()) == ds4a.ERR_INVALID_ARG
    assert _prefill(lib, L, _tensors(k_comp=FAKE, v_comp=FAKE, comp_row_stride=16)) == ds4a.ERR_INVALID_ARG


def test_empty_call_is_a_no_op(lib):
    assert _prefill(lib, _layout(T=0), _tensors(q=None, o=None)) == ds4a.OK
    assert lib.ds4a_pad_kv(None, 0, 0, None, 0, None) == ds4a.OK
    L = _layout(T=0)
    assert lib.ds4a_attn_indexed(ctypes.byref(L), ctypes.byref(_tensors()), None, 0, 512, None) == ds4a.OK


def test_dense_mask_stride_is_checked(lib):
    L = _layout()
    X = _tensors()
    # 2 blocks of 32 rows need 128 bytes per mask row
    assert lib.ds4a_attn_prefill(ctypes.byref(L), ctypes.byref(X), FAKE, 64, None, 1, None) == ds4a.ERR_INVALID_ARG
    assert lib.ds4a_block_mask(ctypes.byref(L), FAKE, 112, 1, FAKE, None) == ds4a.ERR_INVALID_ARG
    assert lib.ds4a_block_mask(ctypes.byref(L), None, 0, 0, FAKE, None) == ds4a.ERR_INVALID_ARG


def test_decode_workspace_is_checked(lib):
    L = _layout(T=1, n_comp=300, ratio=128)
    X = _tensors(k_comp=FAKE, v_comp=FAKE)
    assert lib.ds4a_attn_decode(ctypes.byref(L), ctypes.byref(X), 2, None, 0, None) == ds4a.ERR_WORKSPACE
    small = lib.ds4a_attn_decode_workspace_size(ctypes.byref(L), 2) - 1
    assert lib.ds4a_attn_decode(ctypes.byref(L), ctypes.byref(X), 2, FAKE, small, None) == ds4a.ERR_WORKSPACE
    assert lib.ds4a_attn_decode(ctypes.byref(L), ctypes.byref(X), 2, ctypes.c_void_p((1 << 20) + 128), 1 << 30,
                                None) == ds4a.ERR_WORKSPACE


def test_prefill_fp8kv_workspace_size(lib):
    """Two fp16 rows (K and V) per raw row that some query sees, when the call
    takes the pair kernel (no compressed rows, window <= 128, T >= 2); else 0."""
    f = lib.ds4a_attn_prefill_fp8kv_workspace_size
    # Queries at 1000..1063 with a 128-row window see positions 873..1063.
    L = _layout(T=64, q_pos0=1000, n_raw=2000, raw_pos0=0, n_comp=0, window=128)
    assert f(ctypes.byref(L)) == (1063 - 873 + 1) * 2 * 1024
    # Rows clipped at both ends: positions 950..989 exist, all of them seen.
    L = _layout(T=6, q_pos0=1000, n_raw=40, raw_pos0=950, n_comp=0, window=128)
    assert f(ctypes.byref(L)) == 40 * 2 * 1024
    # Rows that no query sees (all after the last query).
    L = _layout(T=4, q_pos0=100, n_raw=50, raw_pos0=500, n_comp=0, window=128)
    assert f(ctypes.byref(L)) == 0
    for kw in (dict(T=1), dict(window=129), dict(n_comp=8, ratio=4), dict(n_raw=0), dict(window=0)):
        base = dict(T=64, q_pos0=1000, n_raw=2000, raw_pos0=0, n_comp=0, window=128)
        base.update(kw)
        assert f(ctypes.byref(_layout(**base))) == 0, kw
    assert f(None) == 0


def test_prefill_fp8kv_workspace_covers_exactly_the_visible_rows(lib):
    """On random raw-only layouts the workspace holds two fp16 rows for each
    raw row the oracle's window rule makes visible to at least one query (the
    union over the queries is one run of rows), and nothing more."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(20261203)
    f = lib.ds4a_attn_prefill_fp8kv_workspace_size
    for _ in range(300):
        T = int(rng.integers(2, 200))
        window = int(rng.integers(1, 129))
        n_raw = int(rng.integers(1, 700))
        raw_pos0 = int(rng.integers(0, 2000))
        q_pos0 = int(rng.integers(max(0, raw_pos0 - 300), raw_pos0 + n_raw + 300))
        L = dict(T=T, q_pos0=q_pos0, n_raw=n_raw, raw_pos0=raw_pos0, n_comp=0, ratio=128, window=window)
        seen = np.zeros(n_raw, dtype=bool)
        for t in range(T):
            seen |= oracle.raw_visible(L, q_pos0 + t)
        idx = np.flatnonzero(seen)
        if idx.size:
            assert idx[-1] - idx[0] + 1 == idx.size, L  # one run of rows
        got = f(ctypes.byref(_layout(**L)))
        assert got == idx.size * 2 * 1024, (L, got, idx.size)


def test_prefill_fp8kv_workspace_is_checked(lib):
    """The pair path rejects a missing, short or misaligned workspace and bad
    code rows or scales before any device access."""
    L = _layout(T=6, q_pos0=1000, n_raw=40, raw_pos0=950, n_comp=0, window=128)
    X = _tensors()
    S = ds4a.Fp8Scales(FAKE, FAKE, None, None)
    f = lib.ds4a_attn_prefill_fp8kv_ws
    need = lib.ds4a_attn_prefill_fp8kv_workspace_size(ctypes.byref(L))
    assert f(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S), None, 0, None) == ds4a.ERR_WORKSPACE
    assert f(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S), FAKE, need - 1, None) == ds4a.ERR_WORKSPACE
    assert f(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S), ctypes.c_void_p((1 << 20) + 128), need,
             None) == ds4a.ERR_WORKSPACE
    S1 = ds4a.Fp8Scales(FAKE, None, None, None)
    assert f(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S1), FAKE, need, None) == ds4a.ERR_INVALID_ARG
    X1 = _tensors(raw_row_stride=520)
    assert f(ctypes.byref(L), ctypes.byref(X1), ctypes.byref(S), FAKE, need, None) == ds4a.ERR_INVALID_ARG
    X2 = _tensors(o=MISALIGNED)
    assert f(ctypes.byref(L), ctypes.byref(X2), ctypes.byref(S), FAKE, need, None) == ds4a.ERR_INVALID_ARG


def test_graph_arguments_are_checked(lib):
    """Recording needs a created stream and a handle slot; launching needs a
    graph; destroying NULL is a no-op.  All refused before any CUDA call."""
    assert lib.ds4a_graph_begin(None) == ds4a.ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert lib.ds4a_graph_end(None, ctypes.byref(h)) == ds4a.ERR_INVALID_ARG
    assert not h
    assert lib.ds4a_graph_launch(None, FAKE) == ds4a.ERR_INVALID_ARG
    lib.ds4a_graph_destroy(None)


def test_indexed_fp8kv_arguments_are_checked(lib):
    """Rejected before any device access: no scales, a missing compressed-row
    scale, top_k out of 1..4096, no lists, a list stride below 4 * top_k."""
    L = _layout(n_comp=64, ratio=4)
    X = _tensors(k_comp=FAKE, v_comp=FAKE)
    S = ds4a.Fp8Scales(None, None, FAKE, FAKE)
    f = lib.ds4a_attn_indexed_fp8kv
    assert f(ctypes.byref(L), ctypes.byref(X), None, FAKE, 2048, 512, None) == ds4a.ERR_INVALID_ARG
    S1 = ds4a.Fp8Scales(None, None, None, FAKE)
    assert f(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S1), FAKE, 2048, 512, None) == ds4a.ERR_INVALID_ARG
    assert f(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S), FAKE, 2048, 0, None) == ds4a.ERR_INVALID_ARG
    assert f(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S), FAKE, 2048, 4097, None) == ds4a.ERR_INVALID_ARG
    assert f(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S), None, 2048, 512, None) == ds4a.ERR_INVALID_ARG
    assert f(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S), FAKE, 2040, 512, None) == ds4a.ERR_INVALID_ARG


def test_indexed_arguments_are_checked(lib):
    L = _layout(n_comp=64, ratio=4)
    X = _tensors(k_comp=FAKE, v_comp=FAKE)
    assert lib.ds4a_attn_indexed(ctypes.byref(L), ctypes.byref(X), FAKE, 2048, 0, None) == ds4a.ERR_INVALID_ARG
    assert lib.ds4a_attn_indexed(ctypes.byref(L), ctypes.byref(X), FAKE, 2048, 4097, None) == ds4a.ERR_INVALID_ARG
    assert lib.ds4a_attn_indexed(ctypes.byref(L), ctypes.byref(X), None, 2048, 512, None) == ds4a.ERR_INVALID_ARG
    assert lib.ds4a_attn_indexed(ctypes.byref(L), ctypes.byref(X), FAKE, 2040, 512, None) == ds4a.ERR_INVALID_ARG
    assert lib.ds4a_attn_indexed(ctypes.byref(L), ctypes.byref(X), FAKE, 2056, 512, None) == ds4a.ERR_INVALID_ARG


def test_pad_arguments_are_checked(lib):
    assert lib.ds4a_pad_kv(FAKE, 1024, -1, FAKE, 1024, None) == ds4a.ERR_INVALID_ARG
    assert lib.ds4a_pad_kv(FAKE, 1024, 10, None, 1024, None) == ds4a.ERR_INVALID_ARG
    assert lib.ds4a_pad_kv(FAKE, 1000, 10, ctypes.c_void_p(1 << 30), 1024, None) == ds4a.ERR_INVALID_ARG
    # in place needs equal strides; overlapping distinct ranges are refused
    assert lib.ds4a_pad_kv(FAKE, 1024, 10, FAKE, 2048, None) == ds4a.ERR_INVALID_ARG
    assert lib.ds4a_pad_kv(FAKE, 1024, 10, ctypes.c_void_p((1 << 20) + 4096), 1024, None) == ds4a.ERR_INVALID_ARG


def test_selftest_bound_is_checked(lib):
    assert lib.ds4a_selftest_wait_timeout(10, None) == ds4a.ERR_INVALID_ARG
    assert lib.ds4a_selftest_wait_timeout(10**11, None) == ds4a.ERR_INVALID_ARG


def test_compress_arguments_are_checked(lib):
    A = lambda x: ctypes.c_void_p(x)  # noqa: E731
    assert lib.ds4a_compress_rows(3, 6, 4) == 2
    assert lib.ds4a_compress_rows(0, 2048, 128) == 16
    for bad in [(4, 1, 4), (-1, 1, 4), (0, -1, 4), (0, 1, 0), (0, 1, 65537)]:
        assert lib.ds4a_compress_rows(*bad) == -1
    kv, sc, skv, ssc, out = A(1 << 30), A(2 << 30), A(3 << 30), A(4 << 30), A(5 << 30)

    def call(width=512, ratio=4, n_state=0, kv=kv, sc=sc, ns=2048, n_new=8, skv=skv, ssc=ssc, ss=2048, out=out,
             os_=1024):
        return lib.ds4a_compress_append(width, ratio, n_state, kv, sc, ns, n_new, skv, ssc, ss, out, os_, None)

    assert call(n_new=0) == ds4a.OK
    assert call(width=510) == ds4a.ERR_INVALID_ARG           # width % 4
    assert call(n_state=4) == ds4a.ERR_INVALID_ARG           # n_state >= ratio
    assert call(ns=2040) == ds4a.ERR_INVALID_ARG             # row shorter than width
    assert call(ns=2056) == ds4a.ERR_INVALID_ARG             # not a multiple of 16
    assert call(kv=None) == ds4a.ERR_INVALID_ARG
    assert call(kv=A((1 << 30) + 8)) == ds4a.ERR_INVALID_ARG  # 16-byte alignment
    assert call(skv=None) == ds4a.ERR_INVALID_ARG             # ratio > 1 needs a state
    assert call(out=None) == ds4a.ERR_INVALID_ARG             # two rows are pooled
    assert call(os_=1000) == ds4a.ERR_INVALID_ARG            # shorter than a row
    assert call(os_=1028) == ds4a.ERR_INVALID_ARG            # not a multiple of 8
    assert call(width=132, ns=528, ss=528, os_=264, out=None) == ds4a.ERR_INVALID_ARG   # only the output missing
    assert call(out=A((1 << 30) + 4096)) == ds4a.ERR_INVALID_ARG   # output inside the new rows
    assert call(ssc=A((3 << 30) + 2048)) == ds4a.ERR_INVALID_ARG   # the two states overlap
