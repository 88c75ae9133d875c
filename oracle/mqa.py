"""Plain fp64 CPU oracle of the fused multi-query attention forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module; the product path never does.  It
shares no code with the CUDA library: the two meet only through the seeded
inputs of ``mqa_flash_attention_gb300.synth``.

What it computes, and from which passage:

* Fused attention ("How DeepSeek V4 Flash Model Inference Works on Apple Silicon
  with Metal Backend", sections "FlashAttention Kernel Architecture" and the
  FAQ "What Metal kernels are used for FlashAttention in ds4?"): the kernels
  fuse the Q-K product, the softmax normalisation and the value weighting.  A
  fused FlashAttention reaches exactly (up to rounding order) plain softmax
  attention, so this oracle is that plain definition, one query token at a
  time: ``o = sum_j softmax_j(scale * q.k_j + bias_j) v_j`` over the rows
  ``j`` the token may see.
* Shape ("DwarfStar 4 (DS4) - DeepSeek V4 Flash Inference Engine", section
  "Fixed Model Shape"): 64 query heads, one K/V head (multi-query), head dim
  512, a 128-token sliding window.
* Which rows a token sees (same page, sections "Layer Compression" and "KV Cache
  Design"): the raw sliding-window rows, plus compressed rows pooled at ratio
  boundaries - all of them on ratio-128 layers, an indexer's top-512 list on
  ratio-4 layers.
* Block status (first page, section "Mask Handling and Block Skipping"): one
  byte per block of the padded K/V sequence that says whether the block can be
  skipped.
* Padding (first page, section "KV-Cache Management on Metal Device Buffers"):
  the K/V rows are padded to a multiple of 32.

Readings taken where the pages are silent (each one is pinned by a test):

* scale = 1/sqrt(512) unless the layout says otherwise;
* the window holds 128 positions including the token's own: ``p-127 .. p``;
* compressed row ``c`` pools positions ``[c*ratio, (c+1)*ratio-1]`` and is
  visible to position ``p`` once that span has ended: ``(c+1)*ratio <= p+1``;
* the logical sequence used for block numbering is
  ``[raw rows padded to 32 | compressed rows padded to 32]``; pad rows are never
  visible;
* block status 0 = no visible (token, row) pair in the block, 2 = every pair
  visible with zero bias, 1 = anything else;
* with a dense mask, the mask replaces the structural rule: a real row is
  visible iff its mask entry is not -inf, and the entry is added to the scaled
  score (natural-log units);
* an index list entry < 0 is an empty slot, and so is an entry >= n_comp (a
  list slot that names no stored row: the library's interface declares such
  entries empty); every other entry counts once per occurrence (plain gather);
* a token with no visible row gets o = 0 and lse = -inf.

Numbers: every fp16 input is widened exactly to float64 and all arithmetic is
float64.  Matrix products use numpy's ``@`` (a library primitive).
"""

from __future__ import annotations

import numpy as np

H = 64
D = 512
BLOCK = 32


def ceil_to(n: int, m: int) -> int:
    return -(-n // m) * m


# ------------------------------------------------------------------ visibility

def raw_visible(layout: dict, p: int) -> np.ndarray:
    """Raw row ``i`` sits at position ``raw_pos0 + i`` and is visible to
    position ``p`` inside the causal sliding window ``p-window+1 .. p``."""
    pos = layout["raw_pos0"] + np.arange(layout["n_raw"], dtype=np.int64)
    return (pos >= p - layout["window"] + 1) & (pos <= p)


def comp_visible(layout: dict, p: int) -> np.ndarray:
    """Compressed row ``c`` pools positions ``[c*ratio, (c+1)*ratio-1]`` and is
    visible to position ``p`` once its span has ended."""
    c = np.arange(layout["n_comp"], dtype=np.int64)
    return (c + 1) * layout["ratio"] <= p + 1


def padded_lengths(layout: dict) -> tuple[int, int]:
    """Lengths of the two padded segments of the logical K/V sequence."""
    return ceil_to(layout["n_raw"], BLOCK), ceil_to(layout["n_comp"], BLOCK)


def pair_visibility(layout: dict, mask: np.ndarray | None = None):
    """``vis[t, j]`` and ``bias[t, j]`` over the padded logical sequence
    ``[raw | comp]`` (each part padded to 32), for every query token ``t``.

    Without a mask the structural rule applies; with a dense mask (fp16
    ``[T, n_pad_total]``) a real row is visible iff its entry is not -inf and
    the entry is the bias.  Pad rows are never visible."""
    T = layout["T"]
    npr, npc = padded_lengths(layout)
    vis = np.zeros((T, npr + npc), dtype=bool)
    bias = np.zeros((T, npr + npc), dtype=np.float64)
    real = np.zeros(npr + npc, dtype=bool)
    real[: layout["n_raw"]] = True
    real[npr: npr + layout["n_comp"]] = True
    for t in range(T):
        p = layout["q_pos0"] + t
        if mask is None:
            vis[t, : layout["n_raw"]] = raw_visible(layout, p)
            vis[t, npr: npr + layout["n_comp"]] = comp_visible(layout, p)
        else:
            m = mask[t, : npr + npc].astype(np.float64)
            vis[t] = real & (m != -np.inf)
            bias[t] = np.where(vis[t], m, 0.0)
    return vis, bias


def listed_rows(lst, n_comp: int) -> np.ndarray:
    """Compressed rows named by one token's index list: every entry ``c`` with
    ``0 <= c < n_comp``, once per occurrence, in list order.  Entries < 0 and
    entries >= n_comp name no stored row and are empty slots (the top-512
    lists of "DwarfStar 4 (DS4) - DeepSeek V4 Flash Inference Engine",
    section "Layer Compression", pick among the stored compressed rows)."""
    lst = np.asarray(lst, dtype=np.int64)
    return lst[(lst >= 0) & (lst < n_comp)]


# ------------------------------------------------------------------ attention

def _softmax_weighted(q_t, keys, vals, bias, scale):
    """Plain softmax attention of the heads of one token over given rows.

    ``q_t`` [heads, 512], ``keys``/``vals`` [n, 512], ``bias`` [n]; float64."""
    if keys.shape[0] == 0:
        return np.zeros(q_t.shape), np.full(q_t.shape[0], -np.inf)
    s = scale * (q_t @ keys.T) + bias[None, :]          # [64, n]
    m = s.max(axis=1, keepdims=True)
    w = np.exp(s - m)
    den = w.sum(axis=1, keepdims=True)
    o = (w @ vals) / den
    lse = m[:, 0] + np.log(den[:, 0])
    return o, lse


def attention(layout: dict, q, k_raw, v_raw, k_comp=None, v_comp=None, *,
              idx=None, mask=None, tokens=None):
    """Attention output of the listed query tokens (all by default).

    Modes: structural (no ``idx``, no ``mask``), indexed (``idx`` int [T, top_k]:
    raw window rows plus the listed compressed rows) and dense-mask (``mask``
    fp16 [T, n_pad_total]).  Returns ``(o, lse)``: float64 ``[n_tok, 64, 512]``
    and ``[n_tok, 64]`` (natural log)."""
    if idx is not None and mask is not None:
        raise ValueError("indexed mode takes no dense mask")
    T = layout["T"]
    toks = range(T) if tokens is None else [int(t) for t in tokens]
    f = np.float64
    kr = np.asarray(k_raw, dtype=f)
    vr = np.asarray(v_raw, dtype=f)
    kc = np.zeros((0, D)) if k_comp is None else np.asarray(k_comp, dtype=f)
    vc = np.zeros((0, D)) if v_comp is None else np.asarray(v_comp, dtype=f)
    npr, npc = padded_lengths(layout)
    n_raw, n_comp = layout["n_raw"], layout["n_comp"]
    n_heads = np.shape(q)[1]            # 64 for the model; a smaller sample of heads is allowed
    out_o = np.zeros((len(toks), n_heads, D))
    out_l = np.zeros((len(toks), n_heads))
    for n, t in enumerate(toks):
        p = layout["q_pos0"] + t
        qt = np.asarray(q[t], dtype=f)
        if mask is not None:
            m = np.asarray(mask[t], dtype=f)
            rsel = np.nonzero(m[:n_raw] != -np.inf)[0]
            csel = np.nonzero(m[npr: npr + n_comp] != -np.inf)[0]
            keys = np.concatenate([kr[rsel], kc[csel]])
            vals = np.concatenate([vr[rsel], vc[csel]])
            bias = np.concatenate([m[rsel], m[npr + csel]])
        else:
            rsel = np.nonzero(raw_visible(layout, p))[0]
            if idx is None:
                csel = np.nonzero(comp_visible(layout, p))[0]
            else:
                csel = listed_rows(idx[t], n_comp)
            keys = np.concatenate([kr[rsel], kc[csel]])
            vals = np.concatenate([vr[rsel], vc[csel]])
            bias = np.zeros(keys.shape[0])
        out_o[n], out_l[n] = _softmax_weighted(qt, keys, vals, bias, layout["scale"])
    return out_o, out_l


# ------------------------------------------------------------------ block status

def block_status(layout: dict, q_tile: int, mask=None) -> np.ndarray:
    """One byte per (q-tile of ``q_tile`` tokens, 32-row block of the padded
    logical sequence), by brute force over every (token, row) pair:
    0 = no visible pair, 2 = every pair visible with zero bias, 1 = otherwise."""
    vis, bias = pair_visibility(layout, mask)
    T = layout["T"]
    n_blk = vis.shape[1] // BLOCK
    n_qt = -(-T // q_tile)
    out = np.zeros((n_qt, n_blk), dtype=np.uint8)
    for b in range(n_qt):
        rows = slice(b * q_tile, min(T, (b + 1) * q_tile))
        v = vis[rows].reshape(-1, n_blk, BLOCK)
        full = (vis[rows] & (bias[rows] == 0.0)).reshape(-1, n_blk, BLOCK)
        any_ = v.any(axis=(0, 2))
        all_ = full.all(axis=(0, 2))
        out[b] = np.where(all_, 2, np.where(any_, 1, 0))
    return out


# ------------------------------------------------------------------ padding

def pad_rows(src: np.ndarray, n_rows: int) -> np.ndarray:
    """The first ``n_rows`` rows of ``src`` followed by +0.0 rows up to the next
    multiple of 32."""
    out = np.zeros((ceil_to(n_rows, BLOCK), src.shape[1]), dtype=src.dtype)
    out[:n_rows] = src[:n_rows]
    return out
