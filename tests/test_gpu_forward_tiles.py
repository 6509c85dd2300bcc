"""GPU parity of the forward's two CTA forms: one 128-row query tile per CTA
(two CTAs share an SM) and two tiles per CTA (ping-pong inside the CTA). The
launcher picks by grid size; FA_FWD_TILES=1 or 2 forces one form.

Both run the same per-row arithmetic in the same order, so out and LSE must
match bit for bit, and each is checked against the fp64 oracle at the forward
bars (tests/parity.py). Shapes cover d = 64 and 128, one to several query
tiles with ragged tails, grouped-query heads, the unmasked case, Sq != Skv
with the causal mask aligned to the last key, and a full-size workload.
"""
import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from parity import check_fwd, f64

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, Hq, Hkv, Sq, Skv, d, dtype, causal
    (1, 1, 1, 1, 1, 64, "bf16", True),
    (1, 2, 2, 128, 128, 128, "bf16", True),
    (1, 2, 1, 200, 200, 64, "fp16", True),
    (2, 4, 2, 384, 384, 128, "bf16", True),     # odd tile count: a two-tile CTA with one live tile
    (1, 2, 2, 640, 640, 64, "bf16", False),     # unmasked
    (1, 4, 1, 1000, 1000, 128, "bf16", True),   # GQA 4:1, ragged
    (1, 2, 2, 130, 1000, 128, "bf16", True),    # kv_offset 870
    (1, 2, 1, 300, 129, 64, "fp16", False),     # unmasked, fewer keys than queries
]


def _fwd(fa, q, k, v, causal, scale, tiles, monkeypatch):
    monkeypatch.setenv("FA_FWD_TILES", str(tiles))
    monkeypatch.setenv("FA_FWD_CTA_PAIR", "0")
    out, lse = fa.attention_forward(q, k, v, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    return out, lse


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,d,dtype,causal", SHAPES)
def test_forward_tile_forms_agree(fa, monkeypatch, B, Hq, Hkv, Sq, Skv, d, dtype, causal):
    q, k, v = fa_inputs.make_custom(B, Hq, Hkv, Sq, d, dtype, seed=Sq * 5 + Skv + d,
                                    with_dout=False, Skv=Skv)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    scale = 1.0 / np.sqrt(d)
    out1, lse1 = _fwd(fa, qd, kd, vd, causal, scale, 1, monkeypatch)
    out2, lse2 = _fwd(fa, qd, kd, vd, causal, scale, 2, monkeypatch)
    out_ref, lse_ref = oracle.forward(*map(f64, (q, k, v)), causal, scale)
    check_fwd({"out": f64(out1), "lse": f64(lse1)}, out_ref, lse_ref)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_forward_tile_forms_gpt2_small(fa, monkeypatch):
    """The full gpt2_small workload (d = 64, 768 one-tile CTAs, the launcher's
    default form there is one tile per CTA) in both forms."""
    w = fa_inputs.WORKLOADS["gpt2_small"]
    q, k, v = fa_inputs.make_inputs(w, with_dout=False)
    dev = torch.device("cuda", 0)
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    out1, lse1 = _fwd(fa, qd, kd, vd, w.causal, w.scale, 1, monkeypatch)
    out2, lse2 = _fwd(fa, qd, kd, vd, w.causal, w.scale, 2, monkeypatch)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    out_ref, lse_ref = oracle.forward(*map(f64, (q, k, v)), w.causal, w.scale)
    check_fwd({"out": f64(out1), "lse": f64(lse1)}, out_ref, lse_ref)
