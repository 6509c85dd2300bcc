"""fa_bwd_noalloc, the backward entry point for callers that cannot allocate
device memory (it draws its scratch from a fixed array inside libfa instead of
a caller workspace). Checked through the C ABI against fa_bwd, the entry point
with a caller workspace, on two calls in a row with different inputs, so that
the second call runs on scratch the first call left behind.

This file is collected last on purpose (test_zz_*): a run that stops at the
first failure has run every other test before it.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import fa_inputs

GRAD_REL, GRAD_FLOOR = 2e-2, 1e-3   # the backward tolerance of the parity tests
FA_ERR_NOALLOC_LIMIT = -9


def _noalloc_fn(fa):
    fn = fa.lib().fa_bwd_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp] * 9 + [i32, i32, i32, i32, i32, i32, ctypes.c_float, i32, vp]
    fn.restype = i32
    return fn


def test_noalloc_rejects_sizes_over_the_limit(fa_lib):
    fn = _noalloc_fn(fa_lib)
    # long_8k needs a 136 MB workspace, beyond the 32 MiB scratch: rejected on
    # the host before anything is enqueued (no GPU needed)
    assert fa_lib.fa_bwd_workspace_bytes(1, 32, 32, 8192, 128) > fa_lib.NOALLOC_SCRATCH_BYTES
    rc = fn(256, 256, 256, 256, 256, 256, 256, 256, 256, 1, 32, 32, 8192, 128, 1, 0.088, 2, None)
    assert rc == FA_ERR_NOALLOC_LIMIT
    assert "scratch" in fa_lib.fa_strerror(rc)


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward_twice(fa_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa = fa_lib
    fn = _noalloc_fn(fa)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    B, Hq, Hkv, S, d = 2, 4, 2, 700, 128
    assert fa.fa_bwd_workspace_bytes(B, Hq, Hkv, S, d) <= fa.NOALLOC_SCRATCH_BYTES
    scale = 1.0 / math.sqrt(d)
    for call, seed in enumerate((41, 42)):
        q, k, v, do = (x.to(dev) for x in fa_inputs.make_custom(B, Hq, Hkv, S, d, "bf16",
                                                                seed=seed))
        out, lse = fa.attention_forward(q, k, v, True, scale)
        ref = fa.attention_backward(q, k, v, out, do, lse, True, scale)
        got = [torch.full_like(x, float("nan")) for x in ref]
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), do.data_ptr(),
                lse.data_ptr(), got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(),
                B, Hq, Hkv, S, d, 1, scale, fa.DTYPE_CODES[q.dtype], stream.cuda_stream)
        assert rc == 0, fa.fa_strerror(rc)
        torch.cuda.synchronize(dev)
        assert fa.fa_last_device_status(stream) == 0
        for name, r, g in zip(("dq", "dk", "dv"), ref, got):
            r64, g64 = r.double().cpu().numpy(), g.double().cpu().numpy()
            assert np.isfinite(g64).all(), (call, name)
            err = np.abs(g64 - r64).max()
            assert err <= GRAD_REL * max(np.abs(r64).max(), GRAD_FLOOR), (call, name, err)
