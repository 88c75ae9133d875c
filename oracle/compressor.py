"""Plain CPU oracle of the compressor: pooled K/V rows at ratio boundaries.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module; the product path never does.  It
shares no code with the CUDA library.

Passage: "DwarfStar 4 (DS4) - DeepSeek V4 Flash Inference Engine", section
"Layer Compression" (the compressor keeps a rolling K/V and score state and
appends pooled rows at ratio boundaries) and section "KV Cache Design"
(attn_state_kv / attn_state_score hold that rolling state; compressed rows are
pooled every 4 or 128 tokens).  The pages give no pooling formula.  Readings
(each pinned by a test):

* every raw position brings a K/V row kv[i] and a score row s[i] of the same
  width (the "score state" beside the "KV state");
* a completed span of `ratio` consecutive positions becomes one row, pooled
  per dimension by a softmax over the span's scores:
  ``row[d] = sum_i softmax_i(s[i][d]) * kv[i][d]``;
* positions of a span that is not complete yet stay in the state (in order)
  and are pooled with the next call's rows;
* the learned initial states the pages mention for ratio-4 layers are not
  modelled: a state starts empty.

Numbers: float64 throughout (fp16 K/V rows widened exactly).
"""

from __future__ import annotations

import numpy as np


def pool(kv, s, ratio: int) -> np.ndarray:
    """Pooled rows of complete spans: [n // ratio, width] float64."""
    kv = np.asarray(kv, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    n = kv.shape[0] // ratio
    out = np.empty((n, kv.shape[1]))
    for c in range(n):
        sk = s[c * ratio:(c + 1) * ratio]
        vk = kv[c * ratio:(c + 1) * ratio]
        w = np.exp(sk - sk.max(axis=0, keepdims=True))
        out[c] = (w * vk).sum(axis=0) / w.sum(axis=0)
    return out


def append(state_kv, state_s, kv_new, s_new, ratio: int):
    """One call: (pooled rows, new state K/V, new state scores).  The state is
    the rows of the incomplete span, oldest first."""
    kv_all = np.concatenate([np.asarray(state_kv), np.asarray(kv_new)], axis=0)
    s_all = np.concatenate([np.asarray(state_s), np.asarray(s_new)], axis=0)
    n_out = kv_all.shape[0] // ratio
    rows = pool(kv_all[:n_out * ratio], s_all[:n_out * ratio], ratio)
    return rows, kv_all[n_out * ratio:], s_all[n_out * ratio:]
