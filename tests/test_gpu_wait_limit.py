"""Failure handling on the GPU: a bounded wait that runs out.

Every mbarrier wait in the kernels is bounded; when one runs out the kernel
sets an abort flag that stops its other roles, lets the copies and MMAs it has
already issued finish, frees its tensor memory, returns, and ORs bit 1 into
the library's device status word, which fa_last_device_status reads and
clears. libfa_waittest.so is the same library built with the wait limit cut to
about a millisecond and each tensor-core kernel's MMA issuer made to wait
first for a barrier phase that nothing completes (built by
causal_flash_attention_gb300.build.build_all). The forward runs in both its
single-CTA forms (one tile per CTA and two) and its CTA-pair form, and
both head dimensions' kernels run. Nothing faults, traps or
hangs: the wait ends at its limit. The test checks that each call returns,
that the status reports the timeout and is cleared by the read, and that the
product library, called next in the same process and context, still computes
results that match the oracle with a clean status.
"""
import ctypes
import math
import os

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from causal_flash_attention_gb300 import build as fa_build
from parity import check_fwd, check_grad, f64

STATUS_WAIT_TIMEOUT = 1


def _load_waittest():
    L = ctypes.CDLL(fa_build.build(variant="waittest"))
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp]
    L.fa_fwd.restype = i32
    L.fa_bwd_workspace_bytes.argtypes = [i32] * 5
    L.fa_bwd_workspace_bytes.restype = sz
    L.fa_bwd.argtypes = [vp] * 9 + [i32] * 6 + [f32, i32, vp, sz, vp]
    L.fa_bwd.restype = i32
    L.fa_fwd_splitkv.argtypes = [vp] * 5 + [i32] * 7 + [f32, i32, i32, vp, sz, vp]
    L.fa_fwd_splitkv.restype = i32
    L.fa_fwd_splitkv_workspace_bytes.argtypes = [i32] * 7
    L.fa_fwd_splitkv_workspace_bytes.restype = sz
    L.fa_last_device_status.argtypes = [vp, ctypes.POINTER(i32)]
    L.fa_last_device_status.restype = i32
    return L


def _status(L, stream):
    st = ctypes.c_int(-1)
    assert L.fa_last_device_status(stream, ctypes.byref(st)) == 0
    return st.value


@pytest.mark.gpu
def test_wait_that_runs_out_ends_the_kernel_with_an_error_status(fa):
    L = _load_waittest()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev).cuda_stream
    B, Hq, Hkv, S, d = 1, 2, 1, 640, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = fa_inputs.make_custom(B, Hq, Hkv, S, d, "bf16", seed=640)
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    out = torch.zeros_like(qd)
    lse = torch.zeros(qd.shape[:3], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.zeros_like(qd), torch.zeros_like(kd), torch.zeros_like(vd)
    nws = L.fa_bwd_workspace_bytes(B, Hq, Hkv, S, d)
    ws = torch.empty(nws, dtype=torch.uint8, device=dev)
    assert _status(L, stream) == 0

    # forward
    assert L.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), lse.data_ptr(),
                    B, Hq, Hkv, S, d, 1, scale, 2, stream) == 0
    torch.cuda.synchronize(dev)   # the kernel ended
    assert _status(L, stream) & STATUS_WAIT_TIMEOUT
    assert _status(L, stream) == 0   # the read cleared it

    # the CTA-pair forward (d = 128): both CTAs of every pair end
    os.environ["FA_FWD_CTA_PAIR"] = "1"
    try:
        assert L.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(),
                        lse.data_ptr(), B, Hq, Hkv, S, d, 1, scale, 2, stream) == 0
        torch.cuda.synchronize(dev)
    finally:
        del os.environ["FA_FWD_CTA_PAIR"]
    assert _status(L, stream) & STATUS_WAIT_TIMEOUT
    assert _status(L, stream) == 0

    # backward (on the product forward's out and lse)
    ref_out, ref_lse = fa.attention_forward(qd, kd, vd, True, scale)
    assert L.fa_bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), ref_out.data_ptr(),
                    dod.data_ptr(), ref_lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                    dv.data_ptr(), B, Hq, Hkv, S, d, 1, scale, 2, ws.data_ptr(), nws,
                    stream) == 0
    torch.cuda.synchronize(dev)
    assert _status(L, stream) & STATUS_WAIT_TIMEOUT
    assert _status(L, stream) == 0

    # the one-tile forward (d = 128, forced) and the d = 64 kernels (the
    # one-tile forward with its separate P buffer, the backward with its own
    # P^T and dQ columns): each ends with the timeout reported
    os.environ["FA_FWD_TILES"] = "1"
    try:
        assert L.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(),
                        lse.data_ptr(), B, Hq, Hkv, S, d, 1, scale, 2, stream) == 0
        torch.cuda.synchronize(dev)
    finally:
        del os.environ["FA_FWD_TILES"]
    assert _status(L, stream) & STATUS_WAIT_TIMEOUT
    assert _status(L, stream) == 0
    d64 = 64
    q6, k6, v6, do6 = (x.to(dev) for x in fa_inputs.make_custom(B, Hq, Hkv, S, d64, "bf16", seed=641))
    out6 = torch.zeros_like(q6)
    lse6 = torch.zeros(q6.shape[:3], dtype=torch.float32, device=dev)
    assert L.fa_fwd(q6.data_ptr(), k6.data_ptr(), v6.data_ptr(), out6.data_ptr(), lse6.data_ptr(),
                    B, Hq, Hkv, S, d64, 1, 1.0 / math.sqrt(d64), 2, stream) == 0
    torch.cuda.synchronize(dev)
    assert _status(L, stream) & STATUS_WAIT_TIMEOUT
    assert _status(L, stream) == 0
    ref6_out, ref6_lse = fa.attention_forward(q6, k6, v6, True, 1.0 / math.sqrt(d64))
    dq6, dk6, dv6 = torch.zeros_like(q6), torch.zeros_like(k6), torch.zeros_like(v6)
    nws6 = L.fa_bwd_workspace_bytes(B, Hq, Hkv, S, d64)
    ws6 = torch.empty(nws6, dtype=torch.uint8, device=dev)
    assert L.fa_bwd(q6.data_ptr(), k6.data_ptr(), v6.data_ptr(), ref6_out.data_ptr(),
                    do6.data_ptr(), ref6_lse.data_ptr(), dq6.data_ptr(), dk6.data_ptr(),
                    dv6.data_ptr(), B, Hq, Hkv, S, d64, 1, 1.0 / math.sqrt(d64), 2,
                    ws6.data_ptr(), nws6, stream) == 0
    torch.cuda.synchronize(dev)
    assert _status(L, stream) & STATUS_WAIT_TIMEOUT
    assert _status(L, stream) == 0

    # split-KV decode: one query row per head over the 640 keys, 3 ranges
    q1 = qd[:, :, -1:].contiguous()
    out1 = torch.zeros_like(q1)
    lse1 = torch.zeros(q1.shape[:3], dtype=torch.float32, device=dev)
    nsp = L.fa_fwd_splitkv_workspace_bytes(B, Hq, Hkv, 1, S, d, 3)
    wsp = torch.empty(max(nsp, 256), dtype=torch.uint8, device=dev)
    assert L.fa_fwd_splitkv(q1.data_ptr(), kd.data_ptr(), vd.data_ptr(), out1.data_ptr(),
                            lse1.data_ptr(), B, Hq, Hkv, 1, S, d, 1, scale, 2, 3,
                            wsp.data_ptr(), nsp, stream) == 0
    torch.cuda.synchronize(dev)
    assert _status(L, stream) & STATUS_WAIT_TIMEOUT
    assert _status(L, stream) == 0

    # the context is intact: the product library computes correct results
    Q, K, V, DO = map(f64, (q, k, v, do))
    out_ref, lse_ref = oracle.forward(Q, K, V, True, scale)
    got_out, got_lse = fa.attention_forward(qd, kd, vd, True, scale)
    gq, gk, gv = fa.attention_backward(qd, kd, vd, got_out, dod, got_lse, True, scale)
    torch.cuda.synchronize(dev)
    assert fa.fa_last_device_status() == 0
    check_fwd({"out": f64(got_out), "lse": f64(got_lse)}, out_ref, lse_ref)
    for name, g, r in zip(("dq", "dk", "dv"), (gq, gk, gv), oracle.backward(Q, K, V, DO, True, scale)):
        check_grad(name, f64(g), r)
