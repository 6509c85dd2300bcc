"""fa_bwd_noalloc, the backward entry point for callers that cannot allocate
device memory (it draws its scratch from a fixed array inside libfa instead of
a caller workspace). Checked through the C ABI, call after call, against the
fp64 oracle at the parity bars and against fa_bwd, the entry point with a
caller workspace. The calls differ in size, dtype and mask, and the later ones
are smaller than the first, so they run on scratch an earlier call left behind.

This file is collected last on purpose (test_zz_*): a run that stops at the
first failure has run every other test before it.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from parity import GRAD_FLOOR, GRAD_REL

FA_ERR_NULL, FA_ERR_ALIGN, FA_ERR_NOALLOC_LIMIT = -3, -4, -9
# fa_bwd_noalloc runs the same kernels as fa_bwd; only the order of the fp32
# additions into the dQ accumulator may differ between two runs, which can
# move a 16-bit dQ element by one unit in the last place (at most 2^-7 of the
# largest |dQ|). dK and dV have no such additions and must match exactly.
DQ_REL_SAME_KERNELS = 2.0 ** -7


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


def test_noalloc_reports_argument_errors_before_the_limit(fa_lib):
    fn = _noalloc_fn(fa_lib)
    # sizes over the limit, but a null or misaligned pointer: fa_bwd's argument
    # error comes first
    rc = fn(256, 256, None, 256, 256, 256, 256, 256, 256, 1, 32, 32, 8192, 128, 1, 0.088, 2, None)
    assert rc == FA_ERR_NULL
    rc = fn(256, 256, 264, 256, 256, 256, 256, 256, 256, 1, 32, 32, 8192, 128, 1, 0.088, 2, None)
    assert rc == FA_ERR_ALIGN


CALLS = [   # (B, Hq, Hkv, S, d, dtype, causal, seed): largest first
    (2, 4, 2, 700, 128, "bf16", True, 41),
    (1, 2, 2, 300, 64, "fp16", False, 42),
    (1, 2, 1, 130, 64, "fp32", True, 43),
]


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_workspace_backward(fa_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fa = fa_lib
    fn = _noalloc_fn(fa)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    for call, (B, Hq, Hkv, S, d, dtype, causal, seed) in enumerate(CALLS):
        assert fa.fa_bwd_workspace_bytes(B, Hq, Hkv, S, d) <= fa.NOALLOC_SCRATCH_BYTES
        scale = 1.0 / math.sqrt(d)
        q, k, v, do = (x.to(dev) for x in fa_inputs.make_custom(B, Hq, Hkv, S, d, dtype,
                                                                seed=seed))
        out, lse = fa.attention_forward(q, k, v, causal, scale)
        ws_ref = fa.attention_backward(q, k, v, out, do, lse, causal, scale)
        got = [torch.full_like(x, float("nan")) for x in ws_ref]
        rc = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), do.data_ptr(),
                lse.data_ptr(), got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(),
                B, Hq, Hkv, S, d, int(causal), scale, fa.DTYPE_CODES[q.dtype],
                stream.cuda_stream)
        assert rc == 0, fa.fa_strerror(rc)
        torch.cuda.synchronize(dev)
        assert fa.fa_last_device_status(stream) == 0

        f64 = lambda t: t.detach().to("cpu", torch.float64).numpy()
        refs = oracle.backward(*(f64(x) for x in (q, k, v, do)), causal, scale)
        for name, o, w, g in zip(("dq", "dk", "dv"), refs, ws_ref, got):
            g64, w64 = f64(g), f64(w)
            assert np.isfinite(g64).all(), (call, name)
            err = np.abs(g64 - o).max()
            assert err <= GRAD_REL * max(np.abs(o).max(), GRAD_FLOOR), (call, name, err)
            if name == "dq" and dtype != "fp32":
                same = np.abs(g64 - w64).max() <= DQ_REL_SAME_KERNELS * np.abs(w64).max()
            else:
                same = np.array_equal(g64, w64)
            assert same, (call, name, np.abs(g64 - w64).max())
