"""GPU parity of the CTA-pair forward (fa_fwd_pair.cu: two CTAs on two SMs run
M = 256 tcgen05 products with cta_group::2, each loading half of every key and
value tile), selected with FA_FWD_CTA_PAIR=1, at d = 128.

Checked against the fp64 oracle at the forward bars (tests/parity.py), and
against the single-CTA forward, which runs the same per-row arithmetic in the
same order: out and LSE must match it bit for bit. Shapes cover a 512-row
block with 1, 2, 3 and 4 live query tiles, ragged tails, grouped-query heads,
the unmasked case, Sq != Skv with the causal mask aligned to the last key, and
full-size workloads in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from parity import LSE_TOL, OUT_TOL, check_fwd, f64

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, Hq, Hkv, Sq, Skv, dtype, causal
    (1, 1, 1, 1, 1, "bf16", True),
    (1, 2, 2, 128, 128, "bf16", True),      # one live tile of the block (peer's slot-0 tile empty)
    (1, 2, 1, 200, 200, "fp16", True),      # two tiles, ragged
    (1, 2, 2, 300, 300, "bf16", True),      # three tiles: slot 1's peer tile past the end
    (2, 4, 2, 512, 512, "bf16", True),      # one full block
    (1, 2, 2, 640, 640, "bf16", False),     # unmasked, a second block with one tile
    (1, 4, 1, 1000, 1000, "bf16", True),    # GQA 4:1, ragged
    (1, 2, 2, 130, 1000, "bf16", True),     # kv_offset 870: masked band over two key tiles
    (1, 2, 1, 1, 300, "bf16", True),        # one query over a longer cache
    (1, 2, 1, 300, 129, "fp16", False),     # unmasked, fewer keys than queries
]


def _fwd(fa, q, k, v, causal, scale, pair, monkeypatch):
    monkeypatch.setenv("FA_FWD_CTA_PAIR", "1" if pair else "0")
    out, lse = fa.attention_forward(q, k, v, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    return out, lse


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,dtype,causal", SHAPES)
def test_pair_forward_shapes(fa, monkeypatch, B, Hq, Hkv, Sq, Skv, dtype, causal):
    d = 128
    q, k, v = fa_inputs.make_custom(B, Hq, Hkv, Sq, d, dtype, seed=Sq * 3 + Skv + Hq,
                                    with_dout=False, Skv=Skv)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    scale = 1.0 / np.sqrt(d)
    out_p, lse_p = _fwd(fa, qd, kd, vd, causal, scale, True, monkeypatch)
    out_s, lse_s = _fwd(fa, qd, kd, vd, causal, scale, False, monkeypatch)
    out_ref, lse_ref = oracle.forward(*map(f64, (q, k, v)), causal, scale)
    check_fwd({"out": f64(out_p), "lse": f64(lse_p)}, out_ref, lse_ref)
    assert torch.equal(out_p, out_s) and torch.equal(lse_p, lse_s)


def test_pair_forward_gqa_qwen3_dense(fa, monkeypatch):
    w = fa_inputs.WORKLOADS["gqa_qwen3"]
    q, k, v = fa_inputs.make_inputs(w, with_dout=False)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    out_p, lse_p = _fwd(fa, qd, kd, vd, w.causal, w.scale, True, monkeypatch)
    out_s, lse_s = _fwd(fa, qd, kd, vd, w.causal, w.scale, False, monkeypatch)
    assert torch.equal(out_p, out_s) and torch.equal(lse_p, lse_s)
    out_ref, lse_ref = oracle.forward(*map(f64, (q, k, v)), w.causal, w.scale)
    check_fwd({"out": f64(out_p), "lse": f64(lse_p)}, out_ref, lse_ref)


def test_pair_forward_long_8k_sampled(fa, monkeypatch):
    w = fa_inputs.WORKLOADS["long_8k"]
    q, k, v = fa_inputs.make_inputs(w, with_dout=False)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    out_p, lse_p = _fwd(fa, qd, kd, vd, w.causal, w.scale, True, monkeypatch)
    out_s, lse_s = _fwd(fa, qd, kd, vd, w.causal, w.scale, False, monkeypatch)
    assert torch.equal(out_p, out_s) and torch.equal(lse_p, lse_s)
    Q, K, V = map(f64, (q, k, v))
    rows = fa_inputs.sample_rows(w.S, 64, seed=81)
    for h in (0, 31):
        o_r, l_r, _ = oracle.rows(Q, K, V, np.zeros_like(Q), 0, h, rows, True, w.scale)
        assert np.abs(f64(out_p)[0, h, rows] - o_r).max() <= OUT_TOL
        assert np.abs(f64(lse_p)[0, h, rows] - l_r).max() <= LSE_TOL
