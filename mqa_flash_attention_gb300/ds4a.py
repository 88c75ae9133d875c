"""Python binding of ``libds4a.so`` (the C ABI in ``include/ds4a.h``).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current
stream.  There is no fallback: if the library is missing, importing the
functions raises.
"""

from __future__ import annotations

import ctypes
import math
import os

from .workloads import H, D

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libds4a.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(6)
BLOCK_ROWS = 32
ROW_BYTES = 1024


class Ds4aError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class Layout(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("q_pos0", ctypes.c_int32),
                ("n_raw", ctypes.c_int32), ("raw_pos0", ctypes.c_int32),
                ("n_comp", ctypes.c_int32), ("ratio", ctypes.c_int32),
                ("window", ctypes.c_int32), ("scale", ctypes.c_float)]


class Tensors(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("q_tok_stride", ctypes.c_int64),
                ("k_raw", ctypes.c_void_p), ("v_raw", ctypes.c_void_p), ("raw_row_stride", ctypes.c_int64),
                ("k_comp", ctypes.c_void_p), ("v_comp", ctypes.c_void_p), ("comp_row_stride", ctypes.c_int64),
                ("o", ctypes.c_void_p), ("o_tok_stride", ctypes.c_int64),
                ("lse", ctypes.c_void_p)]


class Fp8Scales(ctypes.Structure):
    _fields_ = [("k_raw", ctypes.c_void_p), ("v_raw", ctypes.c_void_p),
                ("k_comp", ctypes.c_void_p), ("v_comp", ctypes.c_void_p)]


class BatchTensors(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("q_seq_stride", ctypes.c_int64),
                ("k_raw", ctypes.c_void_p), ("v_raw", ctypes.c_void_p), ("raw_row_stride", ctypes.c_int64),
                ("raw_seq_stride", ctypes.c_int64), ("raw_rows", ctypes.c_int32),
                ("k_comp", ctypes.c_void_p), ("v_comp", ctypes.c_void_p), ("comp_row_stride", ctypes.c_int64),
                ("comp_seq_stride", ctypes.c_int64), ("comp_rows", ctypes.c_int32),
                ("o", ctypes.c_void_p), ("o_seq_stride", ctypes.c_int64), ("lse", ctypes.c_void_p)]


_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Loads the library once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"{_LIB_PATH} is missing: build it with `python -m mqa_flash_attention_gb300.build`")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i32, i64, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
        PL, PT = ctypes.POINTER(Layout), ctypes.POINTER(Tensors)
        L.ds4a_status_string.restype = ctypes.c_char_p
        L.ds4a_status_string.argtypes = [ctypes.c_int]
        L.ds4a_version.restype = ctypes.c_char_p
        L.ds4a_version.argtypes = []
        L.ds4a_last_cuda_error.restype = ctypes.c_char_p
        L.ds4a_last_cuda_error.argtypes = []
        L.ds4a_pad_kv.restype = st
        L.ds4a_pad_kv.argtypes = [vp, i64, i32, vp, i64, vp]
        L.ds4a_block_count.restype = i32
        L.ds4a_block_count.argtypes = [PL]
        L.ds4a_block_mask.restype = st
        L.ds4a_block_mask.argtypes = [PL, vp, i64, i32, vp, vp]
        L.ds4a_attn_prefill.restype = st
        L.ds4a_attn_prefill.argtypes = [PL, PT, vp, i64, vp, i32, vp]
        L.ds4a_attn_decode_default_splits.restype = i32
        L.ds4a_attn_decode_default_splits.argtypes = [PL]
        L.ds4a_attn_decode_workspace_size.restype = ctypes.c_size_t
        L.ds4a_attn_decode_workspace_size.argtypes = [PL, i32]
        L.ds4a_attn_decode.restype = st
        L.ds4a_attn_decode.argtypes = [PL, PT, i32, vp, ctypes.c_size_t, vp]
        L.ds4a_attn_decode_partials.restype = st
        L.ds4a_attn_decode_partials.argtypes = [PL, PT, i32, vp, ctypes.c_size_t, vp]
        L.ds4a_attn_decode_merge.restype = st
        L.ds4a_attn_decode_merge.argtypes = [PL, PT, i32, vp, ctypes.c_size_t, vp]
        L.ds4a_attn_decode_noalloc.restype = st
        L.ds4a_attn_decode_noalloc.argtypes = [PL, PT, i32, vp]
        L.ds4a_attn_indexed.restype = st
        L.ds4a_attn_indexed.argtypes = [PL, PT, vp, i64, i32, vp]
        L.ds4a_indexer_scores.restype = st
        L.ds4a_indexer_scores.argtypes = [PL, vp, i64, i32, i32, vp, i64, vp, ctypes.c_float, i32, vp, i64, vp]
        L.ds4a_attn_decode_batch.restype = st
        L.ds4a_attn_decode_batch.argtypes = [i32, PL, vp, ctypes.POINTER(BatchTensors), i32, vp, ctypes.c_size_t, vp]
        L.ds4a_attn_decode_batch_workspace_size.restype = ctypes.c_size_t
        L.ds4a_attn_decode_batch_workspace_size.argtypes = [i32, i32]
        L.ds4a_attn_decode_batch_default_splits.restype = i32
        L.ds4a_attn_decode_batch_default_splits.argtypes = [i32, PL, i32, i32]
        L.ds4a_attn_decode_fp8.restype = st
        L.ds4a_attn_decode_fp8.argtypes = [PL, PT, vp, vp, i32, vp, ctypes.c_size_t, vp]
        L.ds4a_attn_decode_fp8kv.restype = st
        L.ds4a_attn_decode_fp8kv.argtypes = [PL, PT, ctypes.POINTER(Fp8Scales), i32, vp, ctypes.c_size_t, vp]
        L.ds4a_attn_prefill_fp8kv.restype = st
        L.ds4a_attn_prefill_fp8kv.argtypes = [PL, PT, ctypes.POINTER(Fp8Scales), vp]
        L.ds4a_attn_prefill_fp8kv_workspace_size.restype = ctypes.c_size_t
        L.ds4a_attn_prefill_fp8kv_workspace_size.argtypes = [PL]
        L.ds4a_attn_prefill_fp8kv_ws.restype = st
        L.ds4a_attn_prefill_fp8kv_ws.argtypes = [PL, PT, ctypes.POINTER(Fp8Scales), vp, ctypes.c_size_t, vp]
        L.ds4a_attn_indexed_fp8kv.restype = st
        L.ds4a_attn_indexed_fp8kv.argtypes = [PL, PT, ctypes.POINTER(Fp8Scales), vp, i64, i32, vp]
        L.ds4a_quantize_kv_fp8.restype = st
        L.ds4a_quantize_kv_fp8.argtypes = [vp, i64, i32, vp, i64, vp, vp]
        L.ds4a_compress_rows.restype = i32
        L.ds4a_compress_rows.argtypes = [i32, i32, i32]
        L.ds4a_compress_append.restype = st
        L.ds4a_compress_append.argtypes = [i32, i32, i32, vp, vp, i64, i32, vp, vp, i64, vp, i64, vp]
        L.ds4a_indexer_topk.restype = st
        L.ds4a_indexer_topk.argtypes = [PL, vp, i64, i32, vp, i64, vp]
        L.ds4a_device_status.restype = st
        L.ds4a_device_status.argtypes = [vp, ctypes.c_int]
        L.ds4a_device_error_word.restype = st
        L.ds4a_device_error_word.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
        L.ds4a_selftest_wait_timeout.restype = st
        L.ds4a_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        L.ds4a_graph_begin.restype = st
        L.ds4a_graph_begin.argtypes = [vp]
        L.ds4a_graph_end.restype = st
        L.ds4a_graph_end.argtypes = [vp, ctypes.POINTER(vp)]
        L.ds4a_graph_launch.restype = st
        L.ds4a_graph_launch.argtypes = [vp, vp]
        L.ds4a_graph_destroy.restype = None
        L.ds4a_graph_destroy.argtypes = [vp]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().ds4a_status_string(int(status)).decode()


def version() -> str:
    return lib().ds4a_version().decode()


def last_cuda_error() -> str:
    """The CUDA call and code behind the latest ERR_CUDA on this thread ("" if none)."""
    return lib().ds4a_last_cuda_error().decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise Ds4aError(status, what + (" [" + last_cuda_error() + "]" if status == ERR_CUDA else ""))


def make_layout(layout) -> Layout:
    """A ``Layout`` from a dict with the ``ds4a_layout`` fields (or a ``Layout``)."""
    if isinstance(layout, Layout):
        return layout
    return Layout(int(layout["T"]), int(layout["q_pos0"]), int(layout["n_raw"]), int(layout["raw_pos0"]),
                  int(layout["n_comp"]), int(layout.get("ratio", 1) or 1), int(layout["window"]),
                  float(layout.get("scale", 1.0 / math.sqrt(D))))


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _on_device(**named):
    """Every given tensor must live on the current CUDA device: the kernels
    dereference the pointers there, so a host tensor or one on another device
    would be read out of bounds on the GPU rather than rejected."""
    import torch
    for name, t in named.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
        if t.device.index != torch.cuda.current_device():
            raise ValueError(f"{name} is on {t.device}, not on the current device cuda:{torch.cuda.current_device()}")


def _n_blocks(L) -> int:
    return -(-L.n_raw // BLOCK_ROWS) + -(-L.n_comp // BLOCK_ROWS)


def _rows(t, name, need=0):
    """A [rows, 512] fp16 tensor with contiguous rows -> (pointer, byte stride).
    It must hold at least ``need`` rows (the rows the layout says it has)."""
    import torch
    if t is None:
        if need > 0:
            raise ValueError(f"{name} is missing but the layout has {need} rows")
        return None, ROW_BYTES
    if t.dtype != torch.float16 or t.dim() != 2 or t.shape[1] != D or t.stride(1) != 1:
        raise ValueError(f"{name} must be fp16 [rows, 512] with contiguous rows")
    if t.shape[0] < need:
        raise ValueError(f"{name} holds {t.shape[0]} rows, the layout needs {need}")
    return _ptr(t), t.stride(0) * 2


def _tokens(t, name, T=None):
    """A [T, 64, 512] fp16 tensor with contiguous heads -> (pointer, byte stride)."""
    import torch
    if t.dtype != torch.float16 or t.dim() != 3 or t.shape[1:] != (H, D) or t.stride(2) != 1 or t.stride(1) != D:
        raise ValueError(f"{name} must be fp16 [T, 64, 512] with contiguous heads")
    if T is not None and t.shape[0] != T:
        raise ValueError(f"{name} has {t.shape[0]} tokens, the layout has T = {T}")
    return _ptr(t), t.stride(0) * 2


def _lse_ok(lse, T):
    import torch
    if lse is None:
        return
    if lse.dtype != torch.float32 or tuple(lse.shape) != (T, H) or not lse.is_contiguous():
        raise ValueError(f"lse must be contiguous fp32 [{T}, 64]")


def _tensors(L, q, k_raw, v_raw, k_comp, v_comp, out, lse, check_device=True) -> Tensors:
    """Operands of one attention call, checked against the layout ``L``: token
    counts, row counts, dtypes, strides and (unless the caller checks them
    after its own size checks) devices."""
    qp, qs = _tokens(q, "q", L.T)
    op, os_ = _tokens(out, "out", L.T) if out is not None else (None, 0)
    krp, rs = _rows(k_raw, "k_raw", L.n_raw)
    vrp, rs2 = _rows(v_raw, "v_raw", L.n_raw)
    kcp, cs = _rows(k_comp, "k_comp", L.n_comp)
    vcp, cs2 = _rows(v_comp, "v_comp", L.n_comp)
    if rs != rs2 or cs != cs2:
        raise ValueError("K and V of a segment must share the row stride")
    _lse_ok(lse, L.T)
    if check_device:
        _on_device(q=q, out=out, k_raw=k_raw, v_raw=v_raw, k_comp=k_comp, v_comp=v_comp, lse=lse)
    return Tensors(qp, qs, krp, vrp, rs, kcp, vcp, cs, op, os_, _ptr(lse))


def _mask_ok(L, mask):
    """A dense mask is fp16 [>= T, >= block_count * 32] with contiguous rows."""
    import torch
    if mask is None:
        return
    cols = _n_blocks(L) * BLOCK_ROWS
    if mask.dtype != torch.float16 or mask.dim() != 2 or mask.stride(1) != 1:
        raise ValueError("mask must be fp16 [T, block_count * 32] with contiguous rows")
    if mask.shape[0] < L.T or mask.shape[1] < cols:
        raise ValueError(f"mask is {tuple(mask.shape)}, the layout needs at least ({L.T}, {cols})")


def _status_ok(L, status, q_tile, name):
    """Status bytes are contiguous uint8 [ceil(T / q_tile), block_count]."""
    import torch
    want = (-(-L.T // int(q_tile)), _n_blocks(L))
    if status.dtype != torch.uint8 or tuple(status.shape) != want or not status.is_contiguous():
        raise ValueError(f"{name} must be contiguous uint8 {want}")


def _outputs(q, out, lse, want_lse):
    import torch
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((q.shape[0], H), dtype=torch.float32, device=q.device)
    return out, lse


# ------------------------------------------------------------------ calls

def pad_kv(src, n_rows: int | None = None, dst=None, stream=None):
    """Rows ``0 .. n_rows-1`` of ``src`` followed by zero rows up to a multiple
    of 32.  ``dst`` defaults to a new tensor; ``dst is src`` pads in place."""
    import torch
    n = src.shape[0] if n_rows is None else int(n_rows)
    n_pad = -(-n // BLOCK_ROWS) * BLOCK_ROWS
    if dst is None:
        dst = torch.empty((n_pad, D), dtype=torch.float16, device=src.device)
    sp, ss = _rows(src, "src", n)
    dp, ds = _rows(dst, "dst", n_pad)
    _on_device(src=src, dst=dst)
    _check(lib().ds4a_pad_kv(sp, ss, n, dp, ds, _stream(stream)), "ds4a_pad_kv")
    return dst


def block_count(layout) -> int:
    return lib().ds4a_block_count(ctypes.byref(make_layout(layout)))


def block_mask(layout, q_tile: int, mask=None, out=None, stream=None):
    """Status bytes ``uint8 [ceil(T/q_tile), block_count]``."""
    import torch
    L = make_layout(layout)
    if int(q_tile) < 1:
        raise ValueError("q_tile must be >= 1")
    nb = _n_blocks(L)
    _mask_ok(L, mask)
    if out is None:
        out = torch.empty((-(-L.T // q_tile), nb), dtype=torch.uint8, device="cuda")
    _status_ok(L, out, q_tile, "out")
    _on_device(mask=mask, out=out)
    ms = 0 if mask is None else mask.stride(0) * 2
    _check(lib().ds4a_block_mask(ctypes.byref(L), _ptr(mask), ms, int(q_tile), _ptr(out), _stream(stream)),
           "ds4a_block_mask")
    return out


def attn_prefill(layout, q, k_raw, v_raw, k_comp=None, v_comp=None, *, mask=None, status=None, q_tile=1,
                 out=None, lse=None, want_lse=False, stream=None):
    L = make_layout(layout)
    _mask_ok(L, mask)
    if status is not None:
        if mask is None:
            raise ValueError("status bytes are read only with a dense mask")
        _status_ok(L, status, q_tile, "status")
    out, lse = _outputs(q, out, lse, want_lse)
    X = _tensors(L, q, k_raw, v_raw, k_comp, v_comp, out, lse)
    _on_device(mask=mask, status=status)
    ms = 0 if mask is None else mask.stride(0) * 2
    _check(lib().ds4a_attn_prefill(ctypes.byref(L), ctypes.byref(X), _ptr(mask), ms, _ptr(status), int(q_tile),
                                   _stream(stream)), "ds4a_attn_prefill")
    return (out, lse) if (want_lse or lse is not None) else out


def decode_workspace_bytes(layout, n_splits: int = 0) -> int:
    return lib().ds4a_attn_decode_workspace_size(ctypes.byref(make_layout(layout)), int(n_splits))


def decode_default_splits(layout) -> int:
    return lib().ds4a_attn_decode_default_splits(ctypes.byref(make_layout(layout)))


def attn_decode(layout, q, k_raw, v_raw, k_comp=None, v_comp=None, *, n_splits=0, workspace=None, out=None,
                lse=None, want_lse=False, stream=None):
    import torch
    L = make_layout(layout)
    out, lse = _outputs(q, out, lse, want_lse)
    X = _tensors(L, q, k_raw, v_raw, k_comp, v_comp, out, lse)
    need = decode_workspace_bytes(L, n_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _on_device(workspace=workspace)
    _check(lib().ds4a_attn_decode(ctypes.byref(L), ctypes.byref(X), int(n_splits), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)),
           "ds4a_attn_decode")
    return (out, lse) if (want_lse or lse is not None) else out


class PreparedCall:
    """A library call whose ctypes arguments were built once.  Each ``call()``
    goes through the C ABI with the same tensors, layout and stream; the
    tensors are kept alive by the object.  For loops that call the library
    every step on fixed buffers, where building the arguments again would cost
    more host time than the call itself."""

    def __init__(self, fn, name, args, keep):
        self._fn, self._name, self._args, self._keep = fn, name, args, keep

    def __call__(self) -> None:
        st = self._fn(*self._args)
        if st != OK:
            raise Ds4aError(st, self._name)


class Graph:
    """The library calls made on ``stream`` inside ``with graph:``, recorded
    once and replayed by ``graph()`` as one CUDA graph launch
    (``ds4a_graph_begin`` / ``_end`` / ``_launch``).  Each replay runs the
    recorded kernels on the same buffers, sizes and layouts with whatever the
    buffers hold then.  Give every recorded call its outputs and workspace
    explicitly (an allocation inside the recording would be freed while the
    graph still uses it), keep the tensors alive while the graph is used, and
    do not overlap replays that share a workspace."""

    def __init__(self, stream):
        if stream is None:
            raise ValueError("a graph records a created stream, not the default stream")
        self._stream = stream
        self._h = ctypes.c_void_p()
        self._args = None

    def __enter__(self):
        if self._h:
            raise RuntimeError("this graph was already recorded")
        _check(lib().ds4a_graph_begin(_stream(self._stream)), "ds4a_graph_begin")
        return self

    def __exit__(self, exc_type, exc, tb):
        st = lib().ds4a_graph_end(_stream(self._stream), ctypes.byref(self._h))
        if exc_type is None:
            _check(st, "ds4a_graph_end")
        self._args = (self._h, _stream(self._stream))
        self._fn = lib().ds4a_graph_launch
        return False

    def __call__(self, stream=None) -> None:
        """One replay on the recording stream (or on ``stream``)."""
        args = self._args if stream is None else (self._h, _stream(stream))
        if args is None or not self._h:
            raise RuntimeError("the graph holds no recording")
        st = self._fn(*args)
        if st != OK:
            raise Ds4aError(st, "ds4a_graph_launch")

    def close(self) -> None:
        if self._h:
            lib().ds4a_graph_destroy(self._h)
            self._h = ctypes.c_void_p()
            self._args = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def prepare_decode(layout, q, k_raw, v_raw, k_comp=None, v_comp=None, *, n_splits=0, workspace, out, lse=None,
                   stream=None) -> PreparedCall:
    """:func:`attn_decode` on fixed buffers, as a :class:`PreparedCall`."""
    L = make_layout(layout)
    X = _tensors(L, q, k_raw, v_raw, k_comp, v_comp, out, lse)
    need = decode_workspace_bytes(L, n_splits)
    nbytes = workspace.numel() * workspace.element_size()
    if nbytes < need:
        raise ValueError(f"workspace of {nbytes} bytes, {need} needed")
    _on_device(workspace=workspace)
    args = (ctypes.byref(L), ctypes.byref(X), int(n_splits), _ptr(workspace), nbytes, _stream(stream))
    return PreparedCall(lib().ds4a_attn_decode, "ds4a_attn_decode", args,
                        (L, X, q, k_raw, v_raw, k_comp, v_comp, workspace, out, lse, stream))


def attn_decode_fp8(layout, q, k_raw, v_raw, k_codes, k_scale, v_codes, v_scale, *, n_splits=0, workspace=None,
                    out=None, lse=None, want_lse=False, stream=None):
    """:func:`attn_decode` with E4M3 compressed rows (codes uint8 [n, 512] and
    fp32 row scales [n], as made by :func:`quantize_kv_fp8`)."""
    import torch
    L = make_layout(layout)
    out, lse = _outputs(q, out, lse, want_lse)
    L0 = make_layout(layout)
    L0.n_comp = 0
    X = _tensors(L0, q, k_raw, v_raw, None, None, out, lse, check_device=False)
    for c, nm in ((k_codes, "k_codes"), (v_codes, "v_codes")):
        if c.dtype != torch.uint8 or c.dim() != 2 or c.shape[1] != D or c.stride(1) != 1:
            raise ValueError(f"{nm} must be uint8 [n, 512] with contiguous rows")
        if c.shape[0] < L.n_comp:
            raise ValueError(f"{nm} holds {c.shape[0]} rows, the layout needs {L.n_comp}")
    for sc, nm in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if sc.dtype != torch.float32 or sc.dim() != 1 or sc.stride(0) != 1 or sc.shape[0] < L.n_comp:
            raise ValueError(f"{nm} must be contiguous fp32 [>= {L.n_comp}]")
    if k_codes.stride(0) != v_codes.stride(0):
        raise ValueError("k_codes and v_codes must share the row stride")
    _on_device(q=q, out=out, lse=lse, k_raw=k_raw, v_raw=v_raw, k_codes=k_codes, v_codes=v_codes, k_scale=k_scale,
               v_scale=v_scale)
    X.k_comp, X.v_comp, X.comp_row_stride = k_codes.data_ptr(), v_codes.data_ptr(), k_codes.stride(0)
    need = decode_workspace_bytes(L, n_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _on_device(workspace=workspace)
    _check(lib().ds4a_attn_decode_fp8(ctypes.byref(L), ctypes.byref(X), _ptr(k_scale), _ptr(v_scale), int(n_splits),
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream(stream)), "ds4a_attn_decode_fp8")
    return (out, lse) if (want_lse or lse is not None) else out


def _codes(t, name, need):
    """E4M3 rows: uint8 [>= need, 512] with contiguous rows -> (pointer, byte stride)."""
    import torch
    if t.dtype != torch.uint8 or t.dim() != 2 or t.shape[1] != D or t.stride(1) != 1:
        raise ValueError(f"{name} must be uint8 [rows, 512] with contiguous rows")
    if t.shape[0] < need:
        raise ValueError(f"{name} holds {t.shape[0]} rows, the layout needs {need}")
    return t.data_ptr(), t.stride(0)


def _scales(t, name, need):
    import torch
    if t.dtype != torch.float32 or t.dim() != 1 or t.stride(0) != 1 or t.shape[0] < need:
        raise ValueError(f"{name} must be contiguous fp32 [>= {need}]")
    return t.data_ptr()


def _fp8kv(L, q, k_raw, v_raw, k_comp, v_comp, out, lse, k_raw_scale, v_raw_scale, k_comp_scale, v_comp_scale):
    """Operands of an E4M3 call: compressed rows (and raw rows when their scales
    are given) as codes with per-row scales."""
    raw_fp8 = k_raw_scale is not None or v_raw_scale is not None
    L0 = Layout(L.T, L.q_pos0, 0 if raw_fp8 else L.n_raw, L.raw_pos0, 0, L.ratio, L.window, L.scale)
    X = _tensors(L0, q, None if raw_fp8 else k_raw, None if raw_fp8 else v_raw, None, None, out, lse,
                 check_device=False)
    S = Fp8Scales(None, None, None, None)
    if raw_fp8 and L.n_raw > 0:
        kp, ks = _codes(k_raw, "k_raw", L.n_raw)
        vp, vs = _codes(v_raw, "v_raw", L.n_raw)
        if ks != vs:
            raise ValueError("k_raw and v_raw codes must share the row stride")
        X.k_raw, X.v_raw, X.raw_row_stride = kp, vp, ks
        S.k_raw, S.v_raw = _scales(k_raw_scale, "k_raw_scale", L.n_raw), _scales(v_raw_scale, "v_raw_scale", L.n_raw)
    if L.n_comp > 0:
        kp, ks = _codes(k_comp, "k_comp", L.n_comp)
        vp, vs = _codes(v_comp, "v_comp", L.n_comp)
        if ks != vs:
            raise ValueError("k_comp and v_comp codes must share the row stride")
        X.k_comp, X.v_comp, X.comp_row_stride = kp, vp, ks
        S.k_comp = _scales(k_comp_scale, "k_comp_scale", L.n_comp)
        S.v_comp = _scales(v_comp_scale, "v_comp_scale", L.n_comp)
    _on_device(q=q, out=out, lse=lse, k_raw=k_raw, v_raw=v_raw, k_comp=k_comp, v_comp=v_comp,
               k_raw_scale=k_raw_scale, v_raw_scale=v_raw_scale, k_comp_scale=k_comp_scale,
               v_comp_scale=v_comp_scale)
    return X, S


def attn_decode_fp8kv(layout, q, k_raw, v_raw, k_comp, v_comp, *, k_comp_scale, v_comp_scale, k_raw_scale=None,
                      v_raw_scale=None, n_splits=0, workspace=None, out=None, lse=None, want_lse=False, stream=None):
    """Split-KV decode over E4M3 rows: compressed rows k/v_comp as uint8 codes
    [n_comp, 512] with fp32 row scales; raw rows as codes too when their
    scales are given, else fp16 [n_raw, 512]."""
    import torch
    L = make_layout(layout)
    out, lse = _outputs(q, out, lse, want_lse)
    X, S = _fp8kv(L, q, k_raw, v_raw, k_comp, v_comp, out, lse, k_raw_scale, v_raw_scale, k_comp_scale,
                  v_comp_scale)
    need = decode_workspace_bytes(L, n_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _on_device(workspace=workspace)
    _check(lib().ds4a_attn_decode_fp8kv(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S), int(n_splits),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)), "ds4a_attn_decode_fp8kv")
    return (out, lse) if (want_lse or lse is not None) else out


def prefill_fp8kv_workspace_size(layout) -> int:
    """Workspace bytes of :func:`attn_prefill_fp8kv` with E4M3 raw rows (0: none needed)."""
    return int(lib().ds4a_attn_prefill_fp8kv_workspace_size(ctypes.byref(make_layout(layout))))


def attn_prefill_fp8kv(layout, q, k_raw, v_raw, k_comp=None, v_comp=None, *, k_comp_scale=None, v_comp_scale=None,
                       k_raw_scale=None, v_raw_scale=None, workspace=None, out=None, lse=None, want_lse=False,
                       stream=None):
    """Structural prefill over E4M3 rows (operands as in :func:`attn_decode_fp8kv`).

    With E4M3 raw rows and no compressed rows (window <= 128, T >= 2) the rows
    are decoded once into ``workspace`` (allocated here when None) and the
    prefill runs on the pair kernel; ``workspace=False`` keeps the call on the
    one-token kernel without a workspace."""
    import torch
    L = make_layout(layout)
    out, lse = _outputs(q, out, lse, want_lse)
    X, S = _fp8kv(L, q, k_raw, v_raw, k_comp, v_comp, out, lse, k_raw_scale, v_raw_scale, k_comp_scale,
                  v_comp_scale)
    if workspace is False:
        _check(lib().ds4a_attn_prefill_fp8kv(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S), _stream(stream)),
               "ds4a_attn_prefill_fp8kv")
    else:
        need = lib().ds4a_attn_prefill_fp8kv_workspace_size(ctypes.byref(L)) if k_raw_scale is not None else 0
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        wp, wb = None, 0
        if workspace is not None:
            _on_device(workspace=workspace)
            wp, wb = _ptr(workspace), workspace.numel() * workspace.element_size()
        _check(lib().ds4a_attn_prefill_fp8kv_ws(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S), wp, wb,
                                                _stream(stream)), "ds4a_attn_prefill_fp8kv_ws")
    return (out, lse) if (want_lse or lse is not None) else out


def attn_decode_batch(shape, seq_geom, q, k_raw, v_raw, k_comp=None, v_comp=None, *, n_splits=0, workspace=None,
                      out=None, lse=None, want_lse=False, stream=None):
    """One decode step for B sequences: q fp16 [B, 64, 512]; k/v_raw fp16
    [B, raw_rows, 512]; k/v_comp fp16 [B, comp_rows, 512] (rows contiguous);
    seq_geom int32 [B, 4] on the device: (q_pos, n_raw, raw_pos0, n_comp)."""
    import torch
    S = make_layout(shape)
    B = q.shape[0]
    if seq_geom.dtype != torch.int32 or tuple(seq_geom.shape) != (B, 4) or not seq_geom.is_contiguous():
        raise ValueError("seq_geom must be contiguous int32 [B, 4]")
    out, lse = _outputs(q, out, lse, want_lse)
    qp, qs = _tokens(q, "q")
    op, os_ = _tokens(out, "out", B)
    _lse_ok(lse, B)
    _on_device(seq_geom=seq_geom, q=q, out=out, lse=lse, k_raw=k_raw, v_raw=v_raw, k_comp=k_comp, v_comp=v_comp)

    def seg(k, v):
        if k is None:
            return None, None, ROW_BYTES, ROW_BYTES, 0
        for t, nm in ((k, "k"), (v, "v")):
            if t.dtype != torch.float16 or t.dim() != 3 or t.shape[0] != B or t.shape[2] != D or t.stride(2) != 1:
                raise ValueError(f"{nm} must be fp16 [B, rows, 512] with contiguous rows")
        if k.stride() != v.stride() or k.shape != v.shape:
            raise ValueError("K and V of a segment must share shape and strides")
        return k.data_ptr(), v.data_ptr(), k.stride(1) * 2, k.stride(0) * 2, k.shape[1]

    kr, vr, rrs, rss, rr = seg(k_raw, v_raw)
    kc, vc, crs, css, cr = seg(k_comp, v_comp)
    X = BatchTensors(qp, qs, kr, vr, rrs, rss, rr, kc, vc, crs, css, cr, op, os_, _ptr(lse))
    if n_splits <= 0:
        n_splits = lib().ds4a_attn_decode_batch_default_splits(B, ctypes.byref(S), rr, cr)
    need = lib().ds4a_attn_decode_batch_workspace_size(B, int(n_splits))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _on_device(workspace=workspace)
    _check(lib().ds4a_attn_decode_batch(B, ctypes.byref(S), _ptr(seq_geom), ctypes.byref(X), int(n_splits),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream)), "ds4a_attn_decode_batch")
    return (out, lse) if (want_lse or lse is not None) else out


def attn_decode_partials(layout, q, k_raw, v_raw, k_comp=None, v_comp=None, *, n_splits=0, workspace=None,
                         stream=None):
    """First half of :func:`attn_decode`: per-split partials into ``workspace``."""
    import torch
    L = make_layout(layout)
    X = _tensors(L, q, k_raw, v_raw, k_comp, v_comp, None, None)
    if workspace is None:
        workspace = torch.empty(max(decode_workspace_bytes(L, n_splits), 256), dtype=torch.uint8, device=q.device)
    _on_device(workspace=workspace)
    _check(lib().ds4a_attn_decode_partials(ctypes.byref(L), ctypes.byref(X), int(n_splits), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream(stream)),
           "ds4a_attn_decode_partials")
    return workspace


def attn_decode_merge(layout, workspace, *, n_splits=0, out, lse=None, stream=None):
    """Second half of :func:`attn_decode`: merges the partials into ``out``."""
    L = make_layout(layout)
    op, os_ = _tokens(out, "out", L.T)
    _lse_ok(lse, L.T)
    _on_device(workspace=workspace, out=out, lse=lse)
    X = Tensors(None, 0, None, None, ROW_BYTES, None, None, ROW_BYTES, op, os_, _ptr(lse))
    _check(lib().ds4a_attn_decode_merge(ctypes.byref(L), ctypes.byref(X), int(n_splits), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream)),
           "ds4a_attn_decode_merge")
    return out


def attn_decode_noalloc(layout, q, k_raw, v_raw, k_comp=None, v_comp=None, *, n_splits=0, out=None, lse=None,
                        want_lse=False, stream=None):
    """:func:`attn_decode` without a workspace: the library's own 8 MiB scratch
    array holds the split partials (for callers that cannot allocate)."""
    L = make_layout(layout)
    out, lse = _outputs(q, out, lse, want_lse)
    X = _tensors(L, q, k_raw, v_raw, k_comp, v_comp, out, lse)
    _check(lib().ds4a_attn_decode_noalloc(ctypes.byref(L), ctypes.byref(X), int(n_splits), _stream(stream)),
           "ds4a_attn_decode_noalloc")
    return (out, lse) if (want_lse or lse is not None) else out


def attn_indexed(layout, q, k_raw, v_raw, k_comp, v_comp, idx, *, out=None, lse=None, want_lse=False, stream=None):
    import torch
    L = make_layout(layout)
    if idx.dtype != torch.int32 or idx.dim() != 2 or idx.stride(1) != 1:
        raise ValueError("idx must be int32 [T, top_k] with contiguous rows")
    if idx.shape[0] < L.T:
        raise ValueError(f"idx has {idx.shape[0]} lists, the layout has T = {L.T}")
    out, lse = _outputs(q, out, lse, want_lse)
    X = _tensors(L, q, k_raw, v_raw, k_comp, v_comp, out, lse)
    _on_device(idx=idx)
    _check(lib().ds4a_attn_indexed(ctypes.byref(L), ctypes.byref(X), _ptr(idx), idx.stride(0) * 4, idx.shape[1],
                                   _stream(stream)), "ds4a_attn_indexed")
    return (out, lse) if (want_lse or lse is not None) else out


def attn_indexed_fp8kv(layout, q, k_raw, v_raw, k_comp, v_comp, idx, *, k_comp_scale, v_comp_scale,
                       k_raw_scale=None, v_raw_scale=None, out=None, lse=None, want_lse=False, stream=None):
    """:func:`attn_indexed` over E4M3 rows: the listed compressed rows as uint8
    codes [n_comp, 512] with fp32 row scales; raw rows as codes too when their
    scales are given, else fp16 [n_raw, 512]."""
    import torch
    L = make_layout(layout)
    if idx.dtype != torch.int32 or idx.dim() != 2 or idx.stride(1) != 1:
        raise ValueError("idx must be int32 [T, top_k] with contiguous rows")
    if idx.shape[0] < L.T:
        raise ValueError(f"idx has {idx.shape[0]} lists, the layout has T = {L.T}")
    out, lse = _outputs(q, out, lse, want_lse)
    X, S = _fp8kv(L, q, k_raw, v_raw, k_comp, v_comp, out, lse, k_raw_scale, v_raw_scale, k_comp_scale,
                  v_comp_scale)
    _on_device(idx=idx)
    _check(lib().ds4a_attn_indexed_fp8kv(ctypes.byref(L), ctypes.byref(X), ctypes.byref(S), _ptr(idx),
                                         idx.stride(0) * 4, idx.shape[1], _stream(stream)), "ds4a_attn_indexed_fp8kv")
    return (out, lse) if (want_lse or lse is not None) else out


def indexer_scores(layout, q_idx, k_idx, head_weights, *, scale, relu=True, out=None, stream=None):
    """Indexer scores: fp32 [T, n_comp] (non-candidate rows -inf).

    q_idx: fp16 [T, n_heads, head_dim] with contiguous heads; k_idx: fp16
    [n_comp, head_dim] with contiguous rows; head_weights: fp32 [T, n_heads].
    """
    import torch
    L = make_layout(layout)
    T, n_heads, head_dim = q_idx.shape
    if q_idx.dtype != torch.float16 or q_idx.stride(2) != 1 or q_idx.stride(1) != head_dim:
        raise ValueError("q_idx must be fp16 [T, n_heads, head_dim] with contiguous heads")
    if k_idx.dtype != torch.float16 or k_idx.dim() != 2 or k_idx.stride(1) != 1 or k_idx.shape[1] != head_dim:
        raise ValueError("k_idx must be fp16 [n_comp, head_dim] with contiguous rows")
    w = head_weights
    if w.dtype != torch.float32 or not w.is_contiguous() or tuple(w.shape) != (T, n_heads):
        raise ValueError("head_weights must be contiguous fp32 [T, n_heads]")
    n_comp = L.n_comp
    if T != L.T:
        raise ValueError(f"q_idx has {T} tokens, the layout has T = {L.T}")
    if k_idx.shape[0] < n_comp:
        raise ValueError(f"k_idx holds {k_idx.shape[0]} rows, the layout needs {n_comp}")
    if out is None:
        stride = (n_comp + 3) // 4 * 4
        out = torch.empty((T, stride), dtype=torch.float32, device=q_idx.device)[:, :n_comp]
    if out.dtype != torch.float32 or out.dim() != 2 or out.stride(1) != 1 or out.shape[0] < T or \
            out.shape[1] < n_comp:
        raise ValueError(f"out must be fp32 [>= {T}, >= {n_comp}] with contiguous rows")
    _on_device(q_idx=q_idx, k_idx=k_idx, head_weights=w, out=out)
    _check(lib().ds4a_indexer_scores(ctypes.byref(L), _ptr(q_idx), q_idx.stride(0) * 2, n_heads, head_dim,
                                     _ptr(k_idx), k_idx.stride(0) * 2, _ptr(w), float(scale), 1 if relu else 0,
                                     _ptr(out), out.stride(0) * 4, _stream(stream)), "ds4a_indexer_scores")
    return out


def indexer_topk(layout, scores, top_k, *, out=None, stream=None):
    """Index lists: int32 [T, top_k], ascending rows, -1 padded."""
    import torch
    L = make_layout(layout)
    if scores.dtype != torch.float32 or scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be fp32 [T, >= n_comp] with contiguous rows")
    T = scores.shape[0]
    if T < L.T or scores.shape[1] < L.n_comp:
        raise ValueError(f"scores is {tuple(scores.shape)}, the layout needs at least ({L.T}, {L.n_comp})")
    if out is None:
        stride = (top_k + 3) // 4 * 4
        out = torch.empty((T, stride), dtype=torch.int32, device=scores.device)[:, :top_k]
    if out.dtype != torch.int32 or out.dim() != 2 or out.stride(1) != 1 or out.shape[0] < L.T or \
            out.shape[1] < top_k:
        raise ValueError(f"out must be int32 [>= {L.T}, >= {top_k}] with contiguous rows")
    _on_device(scores=scores, out=out)
    _check(lib().ds4a_indexer_topk(ctypes.byref(L), _ptr(scores), scores.stride(0) * 4, int(top_k), _ptr(out),
                                   out.stride(0) * 4, _stream(stream)), "ds4a_indexer_topk")
    return out


def quantize_kv_fp8(rows, *, codes=None, scales=None, stream=None):
    """E4M3 codes (uint8 [n, 512]) and per-row fp32 scales of fp16 rows [n, 512]."""
    import torch
    ptr, stride = _rows(rows, "rows")
    n = rows.shape[0]
    if codes is None:
        codes = torch.empty((n, 512), dtype=torch.uint8, device=rows.device)
    if scales is None:
        scales = torch.empty((n,), dtype=torch.float32, device=rows.device)
    if codes.dtype != torch.uint8 or codes.dim() != 2 or codes.stride(1) != 1 or codes.shape[1] != 512 or \
            codes.shape[0] < n:
        raise ValueError(f"codes must be uint8 [>= {n}, 512] with contiguous rows")
    if scales.dtype != torch.float32 or scales.dim() != 1 or scales.stride(0) != 1 or scales.shape[0] < n:
        raise ValueError(f"scales must be contiguous fp32 [>= {n}]")
    _on_device(rows=rows, codes=codes, scales=scales)
    _check(lib().ds4a_quantize_kv_fp8(ptr, stride, n, _ptr(codes), codes.stride(0), _ptr(scales), _stream(stream)),
           "ds4a_quantize_kv_fp8")
    return codes, scales


def _f32_rows(t, name, width):
    import torch
    if t.dtype != torch.float32 or t.dim() != 2 or t.shape[1] != width or t.stride(1) != 1:
        raise ValueError(f"{name} must be fp32 [rows, {width}] with contiguous rows")
    return _ptr(t), t.stride(0) * 4


def compress_rows(n_state: int, n_new: int, ratio: int) -> int:
    """Pooled rows one compressor append writes (-1 for invalid arguments)."""
    return lib().ds4a_compress_rows(n_state, n_new, ratio)


def compress_append(kv, score, state_kv, state_score, n_state, ratio, *, out=None, stream=None):
    """Appends fp32 rows kv / score [n_new, width] to a compressor state
    (fp32 [>= ratio - 1, width] each, updated in place, holding n_state rows).
    Returns (pooled fp16 rows [n_out, width], rows left in the state)."""
    import torch
    n_new, width = kv.shape
    kp, ks = _f32_rows(kv, "kv", width)
    sp, ss = _f32_rows(score, "score", width)
    if ks != ss or score.shape[0] != n_new:
        raise ValueError("kv and score must have the same shape and row stride")
    n_out = compress_rows(n_state, n_new, ratio)
    if n_out < 0:
        raise ValueError("invalid n_state / ratio")
    stp, sts = _f32_rows(state_kv, "state_kv", width)
    scp, scs = _f32_rows(state_score, "state_score", width)
    if sts != scs or state_kv.shape[0] < ratio - 1 or state_score.shape[0] < ratio - 1:
        raise ValueError("the state tensors must hold ratio - 1 rows at one row stride")
    if out is None:
        out = torch.empty((n_out, width), dtype=torch.float16, device=kv.device)
    if out.dtype != torch.float16 or out.dim() != 2 or out.shape[0] < n_out or out.shape[1] != width or \
            out.stride(1) != 1:
        raise ValueError("out must be fp16 [>= n_out, width] with contiguous rows")
    _on_device(kv=kv, score=score, state_kv=state_kv, state_score=state_score, out=out)
    _check(lib().ds4a_compress_append(width, ratio, n_state, kp, sp, ks, n_new, stp, scp, sts, _ptr(out),
                                      out.stride(0) * 2, _stream(stream)), "ds4a_compress_append")
    return out[:n_out], (n_state + n_new) % ratio


def device_status(clear: bool = True, stream=None) -> int:
    """Synchronises the stream and returns the device error status code."""
    return lib().ds4a_device_status(_stream(stream), 1 if clear else 0)


def device_error_word(clear: bool = True, stream=None) -> int:
    """Synchronises the stream and returns the raw device error word (0 = none)."""
    w = ctypes.c_uint32(0)
    _check(lib().ds4a_device_error_word(_stream(stream), ctypes.byref(w), 1 if clear else 0),
           "ds4a_device_error_word")
    return w.value


def selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(lib().ds4a_selftest_wait_timeout(int(timeout_ns), _stream(stream)), "ds4a_selftest_wait_timeout")
