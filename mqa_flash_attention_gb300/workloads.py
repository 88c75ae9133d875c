"""The five synthetic workloads the attention calls are checked and timed on.

Shapes follow the DeepSeek V4 Flash attention layer described on the ds4 pages
("DwarfStar 4 (DS4) - DeepSeek V4 Flash Inference Engine", sections "Fixed Model
Shape", "Layer Compression", "KV Cache Design" and "Whole-Model Graph Execution"):
64 query heads over one shared K/V head, head dim 512, a 128-token sliding
window over raw rows, compressed rows pooled every 4 or 128 tokens, 2048-token
prefill chunks, single-token decode.  Values are N(0, 1) rounded to fp16 from
the seeded generator in :mod:`synth`; no dataset is involved.

A layout is a plain dict with the fields of ``ds4a_layout``:
``T, q_pos0, n_raw, raw_pos0, n_comp, ratio, window, scale``.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import synth

H = 64
D = 512
WINDOW = 128
SCALE = 1.0 / math.sqrt(D)


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    layout: dict
    q: np.ndarray                 # fp16 [T, 64, 512]
    k_raw: np.ndarray             # fp16 [n_raw, 512]
    v_raw: np.ndarray
    k_comp: np.ndarray            # fp16 [n_comp, 512]
    v_comp: np.ndarray
    idx: np.ndarray | None = None  # int32 [T, top_k], sorted, -1 = empty slot
    top_k: int = 0


def make_layout(T, q_pos0, n_raw, raw_pos0, n_comp=0, ratio=128, window=WINDOW, scale=SCALE) -> dict:
    return dict(T=int(T), q_pos0=int(q_pos0), n_raw=int(n_raw), raw_pos0=int(raw_pos0),
                n_comp=int(n_comp), ratio=int(ratio), window=int(window), scale=float(scale))


def draw(name: str, seed: int, layout: dict, top_k: int = 0) -> Workload:
    """Draws Q, K, V (and the index lists when ``top_k`` > 0) for ``layout``."""
    T, n_raw, n_comp = layout["T"], layout["n_raw"], layout["n_comp"]
    wl = Workload(
        name=name, seed=seed, layout=layout,
        q=synth.normal_f16(seed, synth.STREAM_Q, (T, H, D)),
        k_raw=synth.normal_f16(seed, synth.STREAM_K_RAW, (n_raw, D)),
        v_raw=synth.normal_f16(seed, synth.STREAM_V_RAW, (n_raw, D)),
        k_comp=synth.normal_f16(seed, synth.STREAM_K_COMP, (n_comp, D)),
        v_comp=synth.normal_f16(seed, synth.STREAM_V_COMP, (n_comp, D)),
        top_k=top_k,
    )
    if top_k:
        wl.idx = draw_index_lists(seed, layout, top_k)
    return wl


def draw_index_lists(seed: int, layout: dict, top_k: int) -> np.ndarray:
    """Per query token, ``top_k`` compressed rows drawn uniformly without
    replacement among the rows whose pooled span has ended by the token's
    position, sorted ascending; ``-1`` fills the slots a short list leaves.

    Row ``c`` pools positions ``[c*ratio, (c+1)*ratio - 1]`` (the compressor
    "appends pooled rows at ratio boundaries", ds4 page, "Layer Compression"),
    so the rows available to position ``p`` are ``c < (p + 1) // ratio``.  This
    is how the workload's index lists are shaped; the attention calls do not
    re-check it.
    """
    T, q_pos0, n_comp, ratio = layout["T"], layout["q_pos0"], layout["n_comp"], layout["ratio"]
    out = np.full((T, top_k), -1, dtype=np.int32)
    for t in range(T):
        avail = min(n_comp, (q_pos0 + t + 1) // ratio)
        k = min(top_k, avail)
        if k:
            out[t, :k] = synth.sample_without_replacement(seed, synth.STREAM_IDX, t, avail, k)
    return out


# ---------------------------------------------------------------- the five configs

def tiny() -> Workload:
    """T=16 query tokens at positions 144..159 over 160 raw rows (positions 0..159)."""
    return draw("tiny_T16_raw160", 1, make_layout(T=16, q_pos0=144, n_raw=160, raw_pos0=0))


def decode_r128_32k() -> Workload:
    """Decode at 32768 context on a ratio-128 layer: 128 raw rows + 256 compressed rows."""
    return draw("decode_ratio128_ctx32768", 2,
                make_layout(T=1, q_pos0=32767, n_raw=128, raw_pos0=32640, n_comp=256, ratio=128))


def prefill_raw_2048() -> Workload:
    """2048-token prefill chunk after 2048 prior tokens on a raw-only layer (2175 raw rows)."""
    return draw("prefill_raw_T2048", 3, make_layout(T=2048, q_pos0=2048, n_raw=2175, raw_pos0=1921))


def indexed_r4_2048() -> Workload:
    """Indexed ratio-4 layer: 2048-token prefill at context 32768, 8192 compressed rows,
    top-512 index list per token, plus the 128-row raw window."""
    return draw("indexed_ratio4_T2048_ctx32768", 4,
                make_layout(T=2048, q_pos0=30720, n_raw=2175, raw_pos0=30593, n_comp=8192, ratio=4),
                top_k=512)


def decode_long(n_comp: int) -> Workload:
    """Decode over ``n_comp`` compressed rows (ratio 128, all pooled) + 128 raw rows."""
    seed = 5 + int(round(math.log2(n_comp)))
    return draw(f"decode_long_N{n_comp}", seed,
                make_layout(T=1, q_pos0=128 * n_comp - 1, n_raw=128, raw_pos0=128 * n_comp - 128,
                            n_comp=n_comp, ratio=128))


LONG_DECODE_SIZES = (1024, 8192, 65536, 262144)


@dataclasses.dataclass
class IndexerWorkload:
    """Inputs of the indexer (scoring + top-k) of one ratio-4 layer."""
    name: str
    seed: int
    layout: dict
    q_idx: np.ndarray   # fp16 [T, n_heads, head_dim]
    k_idx: np.ndarray   # fp16 [n_comp, head_dim]: the indexer's own compressed rows
    w: np.ndarray       # fp32 [T, n_heads]
    scale: float
    relu: bool
    top_k: int


def draw_indexer(name: str, seed: int, layout: dict, n_heads: int, head_dim: int, top_k: int,
                 relu: bool = True) -> IndexerWorkload:
    T, n = layout["T"], layout["n_comp"]
    return IndexerWorkload(name, seed, layout,
                           synth.normal_f16(seed, synth.STREAM_IDX_Q, (T, n_heads, head_dim)),
                           synth.normal_f16(seed, synth.STREAM_IDX_K, (n, head_dim)),
                           synth.normal_f32(seed, synth.STREAM_IDX_W, (T, n_heads)),
                           1.0 / math.sqrt(head_dim), relu, top_k)


def indexer_r4_2048(n_heads: int = 64, head_dim: int = 128) -> IndexerWorkload:
    """Indexer of the indexed ratio-4 layer: 2048 tokens at context 32768 over
    8192 indexer rows, top-512.  The pages give no indexer shape; 64 heads of
    128 dims with max(0, x) is the multi-head reading (one head is the plain
    dot product)."""
    return draw_indexer("indexer_ratio4_T2048_ctx32768", 12,
                        make_layout(T=2048, q_pos0=30720, n_raw=2175, raw_pos0=30593, n_comp=8192, ratio=4),
                        n_heads, head_dim, 512)


@dataclasses.dataclass
class CompressorWorkload:
    name: str
    seed: int
    ratio: int
    kv: np.ndarray      # fp32 [n, width]
    score: np.ndarray   # fp32 [n, width]


def draw_compressor(name: str, seed: int, n: int, width: int, ratio: int, score_std: float = 2.0) -> CompressorWorkload:
    """Rows entering a compressor: kv ~ N(0, 1), scores ~ N(0, score_std^2), fp32."""
    return CompressorWorkload(name, seed, ratio, synth.normal_f32(seed, synth.STREAM_CMP_KV, (n, width)),
                              (synth.normal_f32(seed, synth.STREAM_CMP_S, (n, width)) * np.float32(score_std)))


def compressor_prefill(ratio: int, width: int = D) -> CompressorWorkload:
    """One 2048-token prefill chunk entering a compressor of 512-dim K/V rows
    (a fresh state), on a ratio-4 or a ratio-128 layer."""
    return draw_compressor(f"compressor_ratio{ratio}_T2048_w{width}", 13, 2048, width, ratio)
