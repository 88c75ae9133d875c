"""The allocation-free decode entry point (needs a GB300).

Some callers cannot allocate device memory: code running inside a host
framework whose memory pool owns the device, or a serving loop that forbids
allocation once it is running.  ds4a_attn_decode_noalloc serves them by keeping
its split-KV partials in a fixed 8 MiB array inside the library instead of a
caller workspace (at most 127 (token, split) items per call).

Each case below is called through the C ABI, one right after the other, so
every call finds the array holding the previous call's partials.  Every output
is pre-filled with NaN and compared with the fp64 oracle within the parity
tolerance (max abs 5e-3, mean abs 5e-4; log-sum-exp within 1e-3), and with
ds4a_attn_decode at the same split count, which runs the same kernels on a
caller workspace and must give the same bits.  The cases cover T = 1 and T > 1,
both ends of the capacity (127 items: one token with 127 splits, 127 tokens with
one split each), and splits with no rows (their stale slots must be ignored).
Requests beyond the capacity are refused before any launch.  This file sorts
last, so a stop-at-first-failure run has already run every other test.
"""

import ctypes

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 5e-3, 5e-4, 1e-3


def test_noalloc_decode_against_the_oracle_call_after_call():
    import torch
    from mqa_flash_attention_gb300 import build, ds4a
    from mqa_flash_attention_gb300 import workloads as W

    build.build()
    lib = ds4a.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.ds4a_device_status(stream, 1) == ds4a.OK

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    mk = W.make_layout
    cases = [  # (workload, n_splits requested (0: the library's choice, capped to 127 items), items required)
        (W.decode_r128_32k(), 0, None),
        # 129 tiles: the default split count is capped to the array's 127 items
        (W.draw("noalloc_cap1", 71, mk(T=1, q_pos0=128 * 16384 - 1, n_raw=128, raw_pos0=128 * 16384 - 128,
                                       n_comp=16384, ratio=128)), 0, 127),
        # T > 1 at the capacity: 127 tokens with one split each
        (W.draw("noalloc_cap127", 72, mk(T=127, q_pos0=40000, n_raw=254, raw_pos0=39873, n_comp=312,
                                         ratio=128)), 1, 127),
        # more splits than tiles: most splits see no row and leave their slots stale
        (W.draw("noalloc_empty", 73, mk(T=4, q_pos0=5000, n_raw=200, raw_pos0=4850, n_comp=39, ratio=128)), 31,
         124),
        (W.draw("noalloc_t3", 74, mk(T=3, q_pos0=9000, n_raw=131, raw_pos0=8873, n_comp=70, ratio=128)), 7, 21),
        (W.decode_r128_32k(), 2, 2),
    ]
    for wl, n_splits, items in cases:
        Lp = ds4a.make_layout(wl.layout)
        T = Lp.T
        splits_used = n_splits if n_splits > 0 else min(ds4a.decode_default_splits(Lp), 127 // T)
        if items is not None:
            assert T * splits_used == items, (wl.name, T * splits_used)
        q, kr, vr, kc, vc = (up(a) for a in (wl.q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp))
        out = torch.full_like(q, float("nan"))
        lse = torch.full((T, 64), float("nan"), dtype=torch.float32, device="cuda")
        X = ds4a.Tensors(q.data_ptr(), q.stride(0) * 2, kr.data_ptr(), vr.data_ptr(), kr.stride(0) * 2,
                         kc.data_ptr(), vc.data_ptr(), kc.stride(0) * 2, out.data_ptr(), out.stride(0) * 2,
                         lse.data_ptr())
        st = lib.ds4a_attn_decode_noalloc(ctypes.byref(Lp), ctypes.byref(X), n_splits, stream)
        assert st == ds4a.OK, (wl.name, ds4a.status_string(st))
        torch.cuda.synchronize()
        assert lib.ds4a_device_status(stream, 1) == ds4a.OK, wl.name

        want, wlse = oracle.attention(wl.layout, wl.q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp)
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), wl.name
        err = np.abs(got - want)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (wl.name, err.max(), err.mean())
        gl = lse.cpu().numpy().astype(np.float64)
        assert np.abs(gl - wlse).max() <= LSE_ABS, wl.name

        # the same kernels on a caller workspace, at the split count the call used
        ref = ds4a.attn_decode(wl.layout, q, kr, vr, kc, vc, n_splits=splits_used)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), wl.name

    # requests beyond the 127 items are refused before any launch
    wl = W.decode_r128_32k()
    q, kr, vr, kc, vc = (up(a) for a in (wl.q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp))
    out = torch.zeros_like(q)
    X = ds4a.Tensors(q.data_ptr(), q.stride(0) * 2, kr.data_ptr(), vr.data_ptr(), kr.stride(0) * 2, kc.data_ptr(),
                     vc.data_ptr(), kc.stride(0) * 2, out.data_ptr(), out.stride(0) * 2, None)
    for layout, n_splits in ((mk(T=128, q_pos0=40000, n_raw=128, raw_pos0=39873, n_comp=300, ratio=128), 0),
                             (wl.layout, 128), (dict(wl.layout, T=2), 64)):
        L = ds4a.make_layout(layout)
        assert lib.ds4a_attn_decode_noalloc(ctypes.byref(L), ctypes.byref(X), n_splits, stream) == \
            ds4a.ERR_WORKSPACE, (layout, n_splits)
    torch.cuda.synchronize()
    assert bool((out == 0).all()), "a refused call wrote its output"
