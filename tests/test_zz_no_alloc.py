"""The allocation-free decode entry point (needs a GB300).

Some callers cannot allocate device memory (a host framework whose memory pool
owns the device, a serving loop that forbids allocation once running), so
ds4a_attn_decode_noalloc keeps its split-KV partials in a fixed array inside the
library instead of a caller workspace.  Called here through the C ABI, twice in
a row with different sizes (the array keeps the first call's contents), and
compared with ds4a_attn_decode within the parity tolerance (max abs 5e-3, mean
abs 5e-4).  This file sorts last so a stop-at-first-failure run has already run
every other test.
"""

import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_decode_on_two_calls():
    import torch
    from mqa_flash_attention_gb300 import build, ds4a
    from mqa_flash_attention_gb300 import workloads as W

    build.build()
    lib = ds4a.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.ds4a_device_status(stream, 1) == ds4a.OK

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    for wl in (W.decode_long(8192), W.decode_r128_32k()):
        L = ds4a.make_layout(wl.layout)
        q, kr, vr, kc, vc = (up(a) for a in (wl.q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp))
        out = torch.full_like(q, float("nan"))
        lse = torch.full((1, 64), float("nan"), dtype=torch.float32, device="cuda")
        X = ds4a.Tensors(q.data_ptr(), q.stride(0) * 2, kr.data_ptr(), vr.data_ptr(), kr.stride(0) * 2,
                         kc.data_ptr(), vc.data_ptr(), kc.stride(0) * 2, out.data_ptr(), out.stride(0) * 2,
                         lse.data_ptr())
        st = lib.ds4a_attn_decode_noalloc(ctypes.byref(L), ctypes.byref(X), 0, stream)
        assert st == ds4a.OK, ds4a.status_string(st)
        ref, ref_lse = ds4a.attn_decode(wl.layout, q, kr, vr, kc, vc, want_lse=True)
        torch.cuda.synchronize()
        err = (out.double() - ref.double()).abs()
        assert bool(torch.isfinite(out).all())
        assert err.max().item() <= 5e-3 and err.mean().item() <= 5e-4, (wl.name, err.max().item())
        assert (lse - ref_lse).abs().max().item() <= 1e-3
        assert lib.ds4a_device_status(stream, 1) == ds4a.OK

    # a request that cannot fit in the 8 MiB array (127 items) is refused before any launch
    L = ds4a.make_layout(W.make_layout(T=128, q_pos0=40000, n_raw=128, raw_pos0=39873, n_comp=300, ratio=128))
    assert lib.ds4a_attn_decode_noalloc(ctypes.byref(L), ctypes.byref(X), 0, stream) == ds4a.ERR_WORKSPACE
    L1 = ds4a.make_layout(W.decode_r128_32k().layout)
    assert lib.ds4a_attn_decode_noalloc(ctypes.byref(L1), ctypes.byref(X), 128, stream) == ds4a.ERR_WORKSPACE
