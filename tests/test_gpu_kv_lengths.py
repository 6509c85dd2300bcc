"""GPU parity for separate query and key/value lengths (fa_fwd_kv / fa_bwd_kv)
against the fp64 oracle, with the causal mask aligned to the last key: query
row i stands at position i + (Skv - Sq) ("Phase 14: Flash Attention 2 for
SM120", section Causal Mask, kv_offset = kv_len - q_len).

Same bars as the self-attention parity tests (tests/parity.py). Edge shapes
put the diagonal at offsets that are and are not multiples of the 128-key tile
(so the masked band spans one or two key tiles), single-query rows, and
unmasked calls with fewer keys than queries. Full size: prefill_8k (a 2048-query chunk over 8192 keys, GQA 32/8)
and the unmasked long_8k_nc / gqa_qwen3_nc, in the launch configuration the
benchmark times.
"""
import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from parity import (GRAD_FLOOR, GRAD_REL, LSE_TOL, OUT_TOL, check_fwd, check_grad, f64,
                    run_gpu)

pytestmark = pytest.mark.gpu

KV_EDGE = [
    # B, Hq, Hkv, Sq, Skv, d, dtype, causal
    (1, 1, 1, 1, 1, 64, "bf16", True),
    (1, 2, 1, 1, 300, 128, "bf16", True),        # one new token over a longer cache
    (1, 2, 2, 5, 129, 64, "fp16", True),
    (1, 4, 2, 64, 200, 128, "bf16", True),
    (2, 2, 1, 127, 128, 64, "bf16", True),
    (1, 2, 2, 128, 384, 128, "bf16", True),      # offset 256: tile-aligned diagonal
    (1, 2, 1, 130, 1000, 128, "bf16", True),     # offset 870: band over two key tiles
    (1, 8, 2, 200, 457, 64, "bf16", True),
    (1, 2, 2, 333, 640, 128, "fp16", True),
    (1, 2, 1, 300, 129, 128, "bf16", False),     # unmasked, fewer keys than queries
    (1, 2, 2, 77, 1000, 64, "bf16", False),
    (1, 1, 1, 129, 3, 128, "fp16", False),
    (1, 2, 1, 65, 200, 64, "fp32", True),
    (1, 2, 2, 130, 70, 128, "fp32", False),
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,d,dtype,causal", KV_EDGE)
def test_kv_lengths_edge(fa, B, Hq, Hkv, Sq, Skv, d, dtype, causal):
    q, k, v, do = fa_inputs.make_custom(B, Hq, Hkv, Sq, d, dtype, seed=Sq * 7 + Skv, Skv=Skv)
    assert k.shape[2] == Skv
    scale = 1.0 / np.sqrt(d)
    got = run_gpu(fa, q, k, v, do, causal, scale)
    Q, K, V, DO = map(f64, (q, k, v, do))
    out_ref, lse_ref = oracle.forward(Q, K, V, causal, scale)
    check_fwd(got, out_ref, lse_ref)
    dq, dk, dv = oracle.backward(Q, K, V, DO, causal, scale)
    check_grad("dq", got["dq"], dq)
    check_grad("dk", got["dk"], dk)
    check_grad("dv", got["dv"], dv)


def test_kv_entry_with_equal_lengths_is_the_self_attention_call(fa):
    """fa_fwd_kv / fa_bwd_kv with Sq = Skv run the same kernels as fa_fwd /
    fa_bwd: identical out, lse, dk and dv bits (dQ sums with atomics, so
    only within the bar)."""
    dev = torch.device("cuda", 0)
    q, k, v, do = (x.to(dev) for x in fa_inputs.make_custom(1, 4, 2, 300, 128, "bf16", seed=3))
    outs = []
    for kv in (False, True):
        out, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = fa.workspace_for(q, k)
        if kv:
            fa.fa_fwd_kv(q, k, v, out, lse, True)
            fa.fa_bwd_kv(q, k, v, out, do, lse, dq, dk, dv, ws, True)
        else:
            fa.fa_fwd(q, k, v, out, lse, True)
            fa.fa_bwd(q, k, v, out, do, lse, dq, dk, dv, ws, True)
        outs.append((out, lse, dq, dk, dv))
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    for a, b in zip(outs[0][:2] + outs[0][3:], outs[1][:2] + outs[1][3:]):
        assert torch.equal(a, b)
    check_grad("dq", f64(outs[1][2]), f64(outs[0][2]))


def test_causal_with_fewer_keys_is_rejected(fa):
    dev = torch.device("cuda", 0)
    q, k, v, _ = (x.to(dev) for x in fa_inputs.make_custom(1, 1, 1, 200, 64, "bf16", seed=1,
                                                           Skv=100))
    out, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    with pytest.raises(fa.FAError, match="invalid shape"):
        fa.fa_fwd_kv(q, k, v, out, lse, True)


def test_workload_gqa_qwen3_nc_dense(fa):
    w = fa_inputs.WORKLOADS["gqa_qwen3_nc"]
    q, k, v, do = fa_inputs.make_inputs(w)
    got = run_gpu(fa, q, k, v, do, w.causal, w.scale)
    Q, K, V, DO = map(f64, (q, k, v, do))
    out_ref, lse_ref = oracle.forward(Q, K, V, w.causal, w.scale)
    check_fwd(got, out_ref, lse_ref)
    dq, dk, dv = oracle.backward(Q, K, V, DO, w.causal, w.scale)
    check_grad("dq", got["dq"], dq)
    check_grad("dk", got["dk"], dk)
    check_grad("dv", got["dv"], dv)


@pytest.mark.parametrize("name,n_rows,n_keys", [("prefill_8k", 256, 256),
                                                ("long_8k_nc", 128, 128)])
def test_workload_sampled(fa, name, n_rows, n_keys):
    """Sampled query rows (out, lse, dQ) of every query head and sampled key
    rows (dK, dV) of every key/value head, evaluated one by one by the oracle."""
    w = fa_inputs.WORKLOADS[name]
    q, k, v, do = fa_inputs.make_inputs(w)
    got = run_gpu(fa, q, k, v, do, w.causal, w.scale)
    Q, K, V, DO = map(f64, (q, k, v, do))
    rows = fa_inputs.sample_rows(w.S, n_rows, seed=21)
    keys = fa_inputs.sample_rows(w.kv_len, n_keys, seed=22)
    errs = dict.fromkeys(("out", "lse", "dq", "dk", "dv"), 0.0)
    refmax = dict.fromkeys(("dq", "dk", "dv"), 0.0)
    for h in range(w.Hq):
        o_r, l_r, dq_r = oracle.rows(Q, K, V, DO, 0, h, rows, w.causal, w.scale)
        errs["out"] = max(errs["out"], np.abs(got["out"][0, h, rows] - o_r).max())
        errs["lse"] = max(errs["lse"], np.abs(got["lse"][0, h, rows] - l_r).max())
        errs["dq"] = max(errs["dq"], np.abs(got["dq"][0, h, rows] - dq_r).max())
        refmax["dq"] = max(refmax["dq"], np.abs(dq_r).max())
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
