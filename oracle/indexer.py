"""Plain CPU oracle of the indexer: scoring of compressed rows and top-k selection.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module; the product path never does.  It
shares no code with the CUDA library.

What it computes, and from which passage ("DwarfStar 4 (DS4) - DeepSeek V4
Flash Inference Engine", section "Architecture Deep Dive"):

* "Layer Compression": even layers from 2 upward use ratio-4 compression with a
  learned indexer that selects the top-512 compressed rows for each query; the
  attention then reads only those rows.
* "GPU Backend Architecture": the GPU op list includes indexer scoring and
  top-k.
* "KV Cache Design": the indexer keeps its own compressed rows
  (``index_comp_kv``), pooled at the same ratio boundaries as the attention's.

The pages give no formula for the score.  Readings taken (each pinned by a
test):

* candidates: compressed row ``c`` is a candidate for the token at position
  ``p`` iff its pooled span has ended, ``(c+1)*ratio <= p+1`` (the attention's
  visibility rule for compressed rows);
* score: ``s[t,c] = sum_h w[t,h] * f(scale * q[t,h,:] . k[c,:])`` over the
  indexer's heads ``h``, with ``f`` the identity or ``max(0, x)``.  One head,
  ``w = 1`` and the identity is the plain dot product; several weighted heads
  with ``max(0, x)`` is the multi-head form.  Non-candidates score ``-inf``;
* selection: the ``top_k`` candidates with the largest scores; equal scores go
  to the lower row index; a NaN score counts as ``-inf``;
* output: the selected rows in ascending order, then ``-1`` up to ``top_k``
  (the index-list convention of the indexed attention).

Numbers: fp16 inputs are widened exactly to float64; all score arithmetic is
float64 (numpy ``@`` is the only library primitive).  The selection compares
the scores it is given as they are (for GPU parity it is run on the kernel's
own fp32 scores, so both sides take the decision in the same precision).
"""

from __future__ import annotations

import numpy as np


def candidates(layout: dict, p: int, n_rows: int) -> np.ndarray:
    """Rows c < n_rows whose pooled span [c*ratio, (c+1)*ratio - 1] ended at or before p."""
    c = np.arange(n_rows, dtype=np.int64)
    return (c + 1) * int(layout["ratio"]) <= p + 1


def scores(layout: dict, q_idx, k_idx, w, scale: float, relu: bool, tokens=None) -> np.ndarray:
    """s[t, c] for the tokens listed (all by default): float64 [len(tokens), n_rows].

    q_idx: [T, heads, dim] (fp16); k_idx: [n_rows, dim] (fp16); w: [T, heads].
    """
    q = np.asarray(q_idx)
    k = np.asarray(k_idx).astype(np.float64)
    w = np.asarray(w, dtype=np.float64)
    n_rows = k.shape[0]
    toks = range(q.shape[0]) if tokens is None else tokens
    out = np.full((len(toks), n_rows), -np.inf)
    for i, t in enumerate(toks):
        p = int(layout["q_pos0"]) + int(t)
        cand = candidates(layout, p, n_rows)
        if not cand.any():
            continue
        dots = scale * (q[t].astype(np.float64) @ k[cand].T)  # [heads, n_cand]
        if relu:
            dots = np.maximum(dots, 0.0)
        out[i, cand] = w[t] @ dots
    return out


def topk(layout: dict, s, top_k: int, tokens=None) -> np.ndarray:
    """Selected rows per token: int32 [len(tokens), top_k], ascending, -1 padded.

    s: [T, n_rows] scores (any float type; compared as given, NaN as -inf).
    """
    s = np.asarray(s)
    n_rows = s.shape[1]
    toks = range(s.shape[0]) if tokens is None else tokens
    out = np.full((len(toks), top_k), -1, dtype=np.int32)
    for i, t in enumerate(toks):
        p = int(layout["q_pos0"]) + int(t)
        cand = np.nonzero(candidates(layout, p, n_rows))[0]
        if cand.size == 0:
            continue
        v = s[t, cand].astype(np.float64)
        v = np.where(np.isnan(v), -np.inf, v)
        # Order: score descending, then row index ascending.
        order = np.lexsort((cand, -v))
        chosen = np.sort(cand[order[:top_k]])
        out[i, :chosen.size] = chosen
    return out
