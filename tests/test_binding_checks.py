"""The Python binding rejects operands that do not match the layout (CPU only).

The C side trusts the layout for sizes: it builds tensor maps from n_raw,
n_comp and T and writes T tokens of o and lse.  A tensor shorter than the
layout says, or one that does not live on the current CUDA device, would be
read or written out of bounds on the GPU.  So the binding checks every size
and device against the layout and raises ValueError before the library is
called.  Host tensors are used here: the size checks run first, and a tensor
with the right sizes is then refused for living on the host.
"""

import math

import pytest
import torch

from mqa_flash_attention_gb300 import ds4a

H, D = 64, 512
F16 = torch.float16


def layout(**kw):
    base = dict(T=4, q_pos0=300, n_raw=200, raw_pos0=120, n_comp=50, ratio=4, window=128,
                scale=1.0 / math.sqrt(D))
    base.update(kw)
    return base


def ops(T=4, n_raw=200, n_comp=50):
    return dict(q=torch.zeros((T, H, D), dtype=F16), k_raw=torch.zeros((n_raw, D), dtype=F16),
                v_raw=torch.zeros((n_raw, D), dtype=F16), k_comp=torch.zeros((n_comp, D), dtype=F16),
                v_comp=torch.zeros((n_comp, D), dtype=F16))


def prefill(L, o, **kw):
    return ds4a.attn_prefill(L, o["q"], o["k_raw"], o["v_raw"], o["k_comp"], o["v_comp"], **kw)


def raises(match, fn, *a, **kw):
    with pytest.raises(ValueError, match=match):
        fn(*a, **kw)


def test_correct_sizes_on_the_host_are_refused_for_the_device():
    raises("must be a CUDA tensor", prefill, layout(), ops())


@pytest.mark.parametrize("field,bad,match", [
    ("q", torch.zeros((3, H, D), dtype=F16), "q has 3 tokens"),
    ("k_raw", torch.zeros((199, D), dtype=F16), "k_raw holds 199 rows"),
    ("v_raw", torch.zeros((10, D), dtype=F16), "v_raw holds 10 rows"),
    ("k_comp", torch.zeros((49, D), dtype=F16), "k_comp holds 49 rows"),
    ("v_comp", None, "v_comp is missing"),
    ("q", torch.zeros((4, H, D), dtype=torch.float32), "fp16"),
    ("k_raw", torch.zeros((200, 256), dtype=F16), "fp16"),
])
def test_short_or_malformed_inputs(field, bad, match):
    o = ops()
    o[field] = bad
    raises(match, prefill, layout(), o)


def test_output_and_lse_sizes():
    o = ops()
    raises("out has 5 tokens", prefill, layout(), o, out=torch.zeros((5, H, D), dtype=F16))
    raises("lse must be", prefill, layout(), o, lse=torch.zeros((4, 63), dtype=torch.float32))
    raises("lse must be", prefill, layout(), o, lse=torch.zeros((4, 64), dtype=F16))


def test_dense_mask_and_status_sizes():
    o = ops()
    L = layout()                                     # 7 raw + 2 compressed blocks = 288 columns
    raises("mask is", prefill, L, o, mask=torch.zeros((4, 287), dtype=F16))
    raises("mask is", prefill, L, o, mask=torch.zeros((3, 288), dtype=F16))
    raises("status must be", prefill, L, o, mask=torch.zeros((4, 288), dtype=F16),
           status=torch.zeros((4, 8), dtype=torch.uint8), q_tile=1)
    raises("status must be", prefill, L, o, mask=torch.zeros((4, 288), dtype=F16),
           status=torch.zeros((2, 9), dtype=torch.uint8), q_tile=1)
    raises("only with a dense mask", prefill, L, o, status=torch.zeros((4, 9), dtype=torch.uint8))
    raises("must be a CUDA tensor", prefill, L, o, mask=torch.zeros((4, 288), dtype=F16),
           status=torch.zeros((1, 9), dtype=torch.uint8), q_tile=4)


def test_block_mask_sizes():
    raises("out must be", ds4a.block_mask, layout(), 2, out=torch.zeros((2, 8), dtype=torch.uint8))
    raises("mask is", ds4a.block_mask, layout(), 2, mask=torch.zeros((4, 100), dtype=F16),
           out=torch.zeros((2, 9), dtype=torch.uint8))
    raises("q_tile", ds4a.block_mask, layout(), 0)


def test_index_list_sizes():
    o = ops()
    idx = torch.zeros((3, 16), dtype=torch.int32)
    raises("idx has 3 lists", ds4a.attn_indexed, layout(), o["q"], o["k_raw"], o["v_raw"], o["k_comp"],
           o["v_comp"], idx)
    raises("int32", ds4a.attn_indexed, layout(), o["q"], o["k_raw"], o["v_raw"], o["k_comp"], o["v_comp"],
           torch.zeros((4, 16), dtype=torch.int64))


def test_decode_calls():
    o = ops(T=1)
    L = layout(T=1)
    raises("k_comp holds", ds4a.attn_decode, L, o["q"], o["k_raw"], o["v_raw"], o["k_comp"][:10], o["v_comp"])
    raises("must be a CUDA tensor", ds4a.attn_decode_noalloc, L, o["q"], o["k_raw"], o["v_raw"], o["k_comp"],
           o["v_comp"])
    raises("out has", ds4a.attn_decode_merge, L, torch.zeros(16, dtype=torch.uint8),
           out=torch.zeros((2, H, D), dtype=F16))
    codes = torch.zeros((50, D), dtype=torch.uint8)
    scales = torch.zeros(50, dtype=torch.float32)
    raises("k_codes holds", ds4a.attn_decode_fp8, L, o["q"], o["k_raw"], o["v_raw"], codes[:20], scales, codes,
           scales)
    raises("v_scale must be", ds4a.attn_decode_fp8, L, o["q"], o["k_raw"], o["v_raw"], codes, scales, codes,
           scales[:49])


def test_pad_and_quantize_sizes():
    src = torch.zeros((40, D), dtype=F16)
    raises("src holds 40 rows", ds4a.pad_kv, src, 41, dst=torch.zeros((64, D), dtype=F16))
    raises("dst holds 32 rows", ds4a.pad_kv, src, 40, dst=torch.zeros((32, D), dtype=F16))
    raises("codes must be", ds4a.quantize_kv_fp8, src, codes=torch.zeros((39, D), dtype=torch.uint8),
           scales=torch.zeros(40, dtype=torch.float32))
    raises("scales must be", ds4a.quantize_kv_fp8, src, codes=torch.zeros((40, D), dtype=torch.uint8),
           scales=torch.zeros(39, dtype=torch.float32))


def test_indexer_sizes():
    L = layout(T=4, n_comp=300)
    q_idx = torch.zeros((4, 64, 128), dtype=F16)
    k_idx = torch.zeros((300, 128), dtype=F16)
    w = torch.zeros((4, 64), dtype=torch.float32)
    raises("k_idx holds 299", ds4a.indexer_scores, L, q_idx, k_idx[:299], w, scale=0.1)
    raises("q_idx has 3 tokens", ds4a.indexer_scores, L, q_idx[:3], k_idx, w[:3], scale=0.1)
    raises("out must be", ds4a.indexer_scores, L, q_idx, k_idx, w, scale=0.1,
           out=torch.zeros((4, 299), dtype=torch.float32))
    raises("must be a CUDA tensor", ds4a.indexer_scores, L, q_idx, k_idx, w, scale=0.1)
    s = torch.zeros((4, 300), dtype=torch.float32)
    raises("scores is", ds4a.indexer_topk, L, s[:, :299], 16)
    raises("out must be", ds4a.indexer_topk, L, s, 16, out=torch.zeros((4, 15), dtype=torch.int32))


def test_fp8_prefill_and_graph_arguments():
    """E4M3 raw rows shorter than the layout, or on the host, are refused
    before any workspace is sized or allocated; a recording needs a created
    stream."""
    o = ops(n_comp=0)
    L = layout(n_comp=0)
    codes = torch.zeros((200, D), dtype=torch.uint8)
    scales = torch.zeros(200, dtype=torch.float32)
    raises("k_raw holds", ds4a.attn_prefill_fp8kv, L, o["q"], codes[:150], codes, k_raw_scale=scales,
           v_raw_scale=scales)
    raises("k_raw_scale must be", ds4a.attn_prefill_fp8kv, L, o["q"], codes, codes, k_raw_scale=scales[:10],
           v_raw_scale=scales)
    raises("must be a CUDA tensor", ds4a.attn_prefill_fp8kv, L, o["q"], codes, codes, k_raw_scale=scales,
           v_raw_scale=scales)
    raises("created stream", ds4a.Graph, None)
