"""GPU parity: libfa's CUDA kernels (through the C ABI) against the fp64 oracle
on the same seeded inputs.

Bars: forward max|out - out_oracle| <= 1e-2
and max|lse - lse_oracle| <= 2e-3; backward max|dX - dX_oracle| <=
2e-2 * max(max|dX_oracle|, 1e-3) for X in {Q, K, V}, per tensor (the 1e-3
floor only matters where the oracle's gradient is exactly zero, e.g. dQ and dK
at S = 1, where the bar becomes 2e-5 absolute). The oracle runs on the
bf16 / fp16 / fp32 values the GPU sees, widened to float64.

Workloads at full size: tiny_fp32, gpt2_small and gqa_qwen3 are compared
element by element; long_8k (256 sampled query rows and 256 sampled key rows
per head) and fp16_32k (128 sampled query rows per head, forward only) are
compared on sampled rows the oracle evaluates one by one. Edge shapes span
several tiles and ragged tails.
"""
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle

pytestmark = pytest.mark.gpu

from parity import (GRAD_FLOOR, GRAD_REL, LSE_TOL, OUT_TOL, check_fwd, check_grad, f64,
                    run_gpu)


# ------------------------------------------------------------ full size --
@pytest.mark.parametrize("name", ["tiny_fp32", "gpt2_small", "gqa_qwen3"])
def test_workload_dense(fa, name):
    w = fa_inputs.WORKLOADS[name]
    q, k, v, do = fa_inputs.make_inputs(w)
    got = run_gpu(fa, q, k, v, do, w.causal, w.scale)
    Q, K, V, DO = map(f64, (q, k, v, do))
    out_ref, lse_ref = oracle.forward(Q, K, V, w.causal, w.scale)
    check_fwd(got, out_ref, lse_ref)
    dq, dk, dv = oracle.backward(Q, K, V, DO, w.causal, w.scale)
    check_grad("dq", got["dq"], dq)
    check_grad("dk", got["dk"], dk)
    check_grad("dv", got["dv"], dv)


def test_long_8k_sampled(fa):
    w = fa_inputs.WORKLOADS["long_8k"]
    q, k, v, do = fa_inputs.make_inputs(w)
    got = run_gpu(fa, q, k, v, do, w.causal, w.scale)
    Q, K, V, DO = map(f64, (q, k, v, do))
    rows = fa_inputs.sample_rows(w.S, 256, seed=11)
    ref_dq_max = 0.0
    errs = {"out": 0.0, "lse": 0.0, "dq": 0.0, "dk": 0.0, "dv": 0.0}
    refmax = {"dq": 0.0, "dk": 0.0, "dv": 0.0}
    for h in range(w.Hq):
        o_r, l_r, dq_r = oracle.rows(Q, K, V, DO, 0, h, rows, w.causal, w.scale)
        errs["out"] = max(errs["out"], np.abs(got["out"][0, h, rows] - o_r).max())
        errs["lse"] = max(errs["lse"], np.abs(got["lse"][0, h, rows] - l_r).max())
        errs["dq"] = max(errs["dq"], np.abs(got["dq"][0, h, rows] - dq_r).max())
        refmax["dq"] = max(refmax["dq"], np.abs(dq_r).max())
    keys = fa_inputs.sample_rows(w.S, 256, seed=12)
    for g in range(w.Hkv):
        dk_c, dv_c = oracle.key_columns(Q, K, V, DO, 0, g, keys, w.causal, w.scale,
                                        row_block=1024)
        errs["dk"] = max(errs["dk"], np.abs(got["dk"][0, g, keys] - dk_c).max())
        errs["dv"] = max(errs["dv"], np.abs(got["dv"][0, g, keys] - dv_c).max())
        refmax["dk"] = max(refmax["dk"], np.abs(dk_c).max())
        refmax["dv"] = max(refmax["dv"], np.abs(dv_c).max())
    assert errs["out"] <= OUT_TOL, errs
    assert errs["lse"] <= LSE_TOL, errs
    for n in ("dq", "dk", "dv"):
        assert errs[n] <= GRAD_REL * max(refmax[n], GRAD_FLOOR), (n, errs, refmax)
    del ref_dq_max


def test_fp16_32k_sampled_forward(fa):
    w = fa_inputs.WORKLOADS["fp16_32k"]
    q, k, v = fa_inputs.make_inputs(w, with_dout=False)
    got = run_gpu(fa, q, k, v, None, w.causal, w.scale, backward=False)
    Q, K, V = map(f64, (q, k, v))
    rows = fa_inputs.sample_rows(w.S, 128, seed=13)
    zeros = np.zeros_like(Q[:, :, :1])
    for h in range(w.Hq):
        o_r, l_r, _ = oracle.rows(Q, K, V, np.broadcast_to(zeros, Q.shape), 0, h, rows,
                                  w.causal, w.scale)
        assert np.abs(got["out"][0, h, rows] - o_r).max() <= OUT_TOL
        assert np.abs(got["lse"][0, h, rows] - l_r).max() <= LSE_TOL


# ----------------------------------------------------------- edge shapes --
EDGE = [
    # B, Hq, Hkv, S, d, dtype
    (1, 1, 1, 1, 64, "bf16"), (1, 1, 1, 2, 128, "bf16"), (1, 2, 1, 63, 64, "bf16"),
    (1, 1, 1, 64, 128, "fp16"), (2, 2, 2, 65, 64, "bf16"), (1, 4, 2, 127, 128, "bf16"),
    (1, 2, 2, 128, 64, "fp16"), (1, 8, 1, 129, 128, "bf16"), (2, 4, 4, 200, 64, "bf16"),
    (1, 2, 1, 255, 128, "fp16"), (1, 1, 1, 256, 64, "bf16"), (1, 2, 2, 257, 128, "bf16"),
    (1, 4, 1, 383, 64, "bf16"), (1, 2, 2, 640, 128, "bf16"),
    # 16 query heads per key/value head: a backward CTA walks 16 heads' query
    # tiles (and their dQ boxes) in one loop; ragged last tile
    (1, 16, 1, 300, 128, "bf16"), (2, 16, 1, 200, 64, "fp16"),
    (1, 2, 1, 65, 64, "fp32"), (1, 2, 2, 130, 128, "fp32"), (1, 1, 1, 1, 64, "fp32"),
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", EDGE, ids=lambda s: "B{}H{}-{}S{}d{}{}".format(*s))
def test_edge_shapes(fa, shape, causal):
    B, Hq, Hkv, S, d, dtype = shape
    q, k, v, do = fa_inputs.make_custom(B, Hq, Hkv, S, d, dtype, seed=S * 7 + d + Hq)
    scale = 1.0 / math.sqrt(d)
    got = run_gpu(fa, q, k, v, do, causal, scale)
    Q, K, V, DO = map(f64, (q, k, v, do))
    out_ref, lse_ref = oracle.forward(Q, K, V, causal, scale)
    check_fwd(got, out_ref, lse_ref)
    dq, dk, dv = oracle.backward(Q, K, V, DO, causal, scale)
    check_grad("dq", got["dq"], dq)
    check_grad("dk", got["dk"], dk)
    check_grad("dv", got["dv"], dv)


def test_non_default_scale_and_large_values(fa):
    """Inputs 3 x N(0,1) and scale 0.3: outputs reach ~12, where one bf16 ulp is
    0.06, so the forward bars are taken relative to the output magnitude
    (1e-2 * max|out| for out, 1e-4 * max|lse| for lse); gradient bars as usual."""
    q, k, v, do = fa_inputs.make_custom(1, 2, 2, 300, 128, "bf16", seed=99, value_scale=3.0)
    got = run_gpu(fa, q, k, v, do, True, 0.3)
    Q, K, V, DO = map(f64, (q, k, v, do))
    out_ref, lse_ref = oracle.forward(Q, K, V, True, 0.3)
    e_out = np.abs(got["out"] - out_ref).max()
    e_lse = np.abs(got["lse"] - lse_ref).max()
    assert e_out <= 1e-2 * np.abs(out_ref).max(), e_out
    assert e_lse <= 1e-4 * np.abs(lse_ref).max(), e_lse
    dq, dk, dv = oracle.backward(Q, K, V, DO, True, 0.3)
    check_grad("dq", got["dq"], dq)
    check_grad("dk", got["dk"], dk)
    check_grad("dv", got["dv"], dv)


def test_row_zero_and_outputs_untouched_outside(fa):
    """Causal row 0 equals V[0] (up to output rounding); buffers around the
    outputs are not written."""
    q, k, v, do = fa_inputs.make_custom(1, 2, 2, 300, 64, "bf16", seed=5)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    n = q.numel()
    big = torch.full((n + 64,), 7.0, dtype=q.dtype, device=dev)
    out = big[32:32 + n].view_as(q)
    lse_big = torch.full((q.shape[0] * q.shape[1] * q.shape[2] + 8,), 5.0, device=dev)
    lse = lse_big[4:4 + q.shape[0] * q.shape[1] * q.shape[2]].view(q.shape[:3])
    fa.fa_fwd(qd, kd, vd, out, lse, True, None)
    torch.cuda.synchronize()
    assert torch.all(big[:32] == 7.0) and torch.all(big[32 + n:] == 7.0)
    assert torch.all(lse_big[:4] == 5.0) and torch.all(lse_big[-4:] == 5.0)
    assert torch.equal(out[:, :, 0].cpu(), v[:, :, 0])


def test_repeat_calls_same_result(fa):
    q, k, v, do = fa_inputs.make_custom(2, 4, 2, 333, 128, "bf16", seed=3)
    a = run_gpu(fa, q, k, v, do, True, 1 / math.sqrt(128))
    b = run_gpu(fa, q, k, v, do, True, 1 / math.sqrt(128))
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])
    assert np.array_equal(a["dk"], b["dk"]) and np.array_equal(a["dv"], b["dv"])
    # dQ is summed with atomics across key tiles: equal up to fp32 summation order
    assert np.abs(a["dq"] - b["dq"]).max() <= 1e-2 * np.abs(a["dq"]).max()


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp16", 64)])
def test_backward_workspace_garbage_and_reuse(fa, dtype, d):
    """The workspace's contents on entry do not matter: filled with 0xFF bytes
    (the dQ accumulator, the row vectors and the counter from which the
    persistent backward's CTAs claim key-tile items), then reused by a second
    call, every result matches the oracle, and the two calls agree (dK, dV
    bit for bit). 4 x 8 heads x 10 key tiles = 320 items, more than one per
    SM."""
    B, H, S = 4, 8, 1280
    q, k, v, do = fa_inputs.make_custom(B, H, H, S, d, dtype, seed=320 + d)
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    out, lse = fa.attention_forward(qd, kd, vd, True, scale)
    ws = fa.workspace_for(qd, kd)
    ws.fill_(0xFF)
    first = [f64(t) for t in fa.attention_backward(qd, kd, vd, out, dod, lse, True, scale, ws)]
    second = [f64(t) for t in fa.attention_backward(qd, kd, vd, out, dod, lse, True, scale, ws)]
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    Q, K, V, DO = map(f64, (q, k, v, do))
    refs = oracle.backward(Q, K, V, DO, True, scale)
    for got in (first, second):
        for name, g, r in zip(("dq", "dk", "dv"), got, refs):
            check_grad(name, g, r)
    assert np.array_equal(first[1], second[1]) and np.array_equal(first[2], second[2])
    assert np.abs(first[0] - second[0]).max() <= 1e-2 * np.abs(first[0]).max()


def test_backward_repeatable_over_random_shapes(fa):
    """Races in the backward's cross-step and cross-item barrier phases would
    show as results that change between calls: over 60 seeded random shapes
    (d, GQA ratio, heads, batch, ragged lengths, causal or not, bf16 or fp16),
    three calls each give bit-identical dK and dV (no atomics touch them), dQ
    equal up to the fp32 summation order of its reduce-adds, and a clean
    device status."""
    import random
    rng = random.Random(60)
    dev = torch.device("cuda", 0)
    for n in range(60):
        d = rng.choice([64, 128]); G = rng.choice([1, 2, 4]); Hkv = rng.choice([1, 2, 3, 8])
        B = rng.choice([1, 2, 3]); S = rng.choice([1, 17, 128, 129, 300, 640, 1024, 2049])
        causal = rng.random() < 0.8; dt = rng.choice(["bf16", "fp16"])
        q, k, v, do = fa_inputs.make_custom(B, Hkv * G, Hkv, S, d, dt, seed=1000 + n)
        scale = 1 / math.sqrt(d)
        qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
        out, lse = fa.attention_forward(qd, kd, vd, causal, scale)
        ws = fa.workspace_for(qd, kd)
        r = [fa.attention_backward(qd, kd, vd, out, dod, lse, causal, scale, ws) for _ in range(3)]
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == 0
        shape = (B, Hkv * G, Hkv, S, d, causal, dt)
        for i in (1, 2):
            assert torch.equal(r[0][1], r[i][1]) and torch.equal(r[0][2], r[i][2]), shape
            e = float((r[0][0].float() - r[i][0].float()).abs().max())
            assert e <= 1e-2 * float(r[0][0].float().abs().max()) + 1e-6, shape


@pytest.mark.parametrize("d", [64, 128])
def test_cuda_graph_capture_and_replay(fa, d):
    """fa_fwd + fa_bwd captured in a CUDA graph (the backward's three kernels
    chained by programmatic dependent launch, its work-item counter reset by
    the pre-pass on every replay) and replayed twice give the eager results:
    out, LSE, dK, dV bit for bit, dQ up to the summation order of its fp32
    reduce-adds."""
    B, Hq, Hkv, S = 2, 8, 4, 1100
    q, k, v, do = fa_inputs.make_custom(B, Hq, Hkv, S, d, "bf16", seed=77 + d)
    scale = 1 / math.sqrt(d)
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    out, lse = torch.empty_like(qd), torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = fa.workspace_for(qd, kd)

    def step():
        fa.fa_fwd(qd, kd, vd, out, lse, True, scale)
        fa.fa_bwd(qd, kd, vd, out, dod, lse, dq, dk, dv, ws, True, scale)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                      # eager, on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (out, lse, dq, dk, dv)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        step()
    for _ in range(2):
        for t in (out, lse, dq, dk, dv):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == 0
        for name, a, b in zip(("out", "lse", "dk", "dv"), eager[:2] + eager[3:],
                              (out, lse, dk, dv)):
            assert torch.equal(a, b), name
        e = float((eager[2].float() - dq.float()).abs().max())
        assert e <= 1e-2 * float(eager[2].float().abs().max())


# ------------------------------------------------------------ large sizes --
def test_longest_sequence_sampled(fa):
    """S = 65536 (twice the longest workload), one head, d = 64: forward and dQ
    on sampled query rows, dK and dV on sampled key rows (the oracle evaluates
    every query row for those, streaming 512 rows at a time)."""
    B, H, S, d = 1, 1, 65536, 64
    q, k, v, do = fa_inputs.make_custom(B, H, H, S, d, "bf16", seed=65)
    scale = 1.0 / math.sqrt(d)
    got = run_gpu(fa, q, k, v, do, True, scale)
    Q, K, V, DO = map(f64, (q, k, v, do))
    rows = fa_inputs.sample_rows(S, 48, seed=66)
    o_r, l_r, dq_r = oracle.rows(Q, K, V, DO, 0, 0, rows, True, scale)
    assert np.abs(got["out"][0, 0, rows] - o_r).max() <= OUT_TOL
    assert np.abs(got["lse"][0, 0, rows] - l_r).max() <= LSE_TOL
    check_grad("dq", got["dq"][0, 0, rows], dq_r)
    assert np.isfinite(got["dk"]).all() and np.isfinite(got["dv"]).all()
    keys = fa_inputs.sample_rows(S, 32, seed=67)
    dk_c, dv_c = oracle.key_columns(Q, K, V, DO, 0, 0, keys, True, scale)
    check_grad("dk", got["dk"][0, 0, keys], dk_c)
    check_grad("dv", got["dv"][0, 0, keys], dv_c)


def test_many_heads_gqa(fa):
    """1024 query heads in groups of 8 over 128 key/value heads."""
    B, Hq, Hkv, S, d = 16, 64, 8, 256, 128
    q, k, v, do = fa_inputs.make_custom(B, Hq, Hkv, S, d, "bf16", seed=1024)
    scale = 1.0 / math.sqrt(d)
    got = run_gpu(fa, q, k, v, do, True, scale)
    Q, K, V, DO = map(f64, (q, k, v, do))
    out_ref, lse_ref = oracle.forward(Q, K, V, True, scale)
    check_fwd(got, out_ref, lse_ref)
    dq, dk, dv = oracle.backward(Q, K, V, DO, True, scale)
    check_grad("dq", got["dq"], dq)
    check_grad("dk", got["dk"], dk)
    check_grad("dv", got["dv"], dv)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("fp16", 64)])
def test_non_causal_multi_tile(fa, dtype, d):
    B, Hq, Hkv, S = 1, 4, 2, 1024
    q, k, v, do = fa_inputs.make_custom(B, Hq, Hkv, S, d, dtype, seed=77 + d)
    scale = 1.0 / math.sqrt(d)
    got = run_gpu(fa, q, k, v, do, False, scale)
    Q, K, V, DO = map(f64, (q, k, v, do))
    out_ref, lse_ref = oracle.forward(Q, K, V, False, scale)
    check_fwd(got, out_ref, lse_ref)
    dq, dk, dv = oracle.backward(Q, K, V, DO, False, scale)
    check_grad("dq", got["dq"], dq)
    check_grad("dk", got["dk"], dk)
    check_grad("dv", got["dv"], dv)
