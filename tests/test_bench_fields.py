"""bench.py's reported quantities, checked on the CPU against closed forms: the
FLOP convention of the metric (causal forward 2*B*Hq*S^2*d, backward
5*B*Hq*S^2*d; unmasked and query-chunk counts by visible query-key pairs),
the algorithmic HBM bytes per call, and the HBM side of the roofline."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import fa_inputs  # noqa: E402


def test_visible_pairs():
    assert bench.visible_pairs(8192, 8192, True) == pytest.approx(8192 * 8192 / 2)
    assert bench.visible_pairs(8192, 8192, False) == 8192 * 8192
    # a causal query chunk at the end of a longer context: each of the Sq rows
    # sees Skv - Sq keys plus its own prefix of the chunk
    assert bench.visible_pairs(2048, 8192, True) == pytest.approx(2048 * 8192 - 2048 ** 2 / 2)


def test_flop_convention_long_8k():
    w = fa_inputs.WORKLOADS["long_8k"]
    B, H, S, d = 1, 32, 8192, 128
    assert bench.flops(w, True, False) == pytest.approx(2 * B * H * S * S * d)
    assert bench.flops(w, False, True) == pytest.approx(5 * B * H * S * S * d)
    assert bench.flops(w, True, True) == pytest.approx(7 * B * H * S * S * d)


def test_algorithmic_bytes_long_8k():
    w = fa_inputs.WORKLOADS["long_8k"]
    t = 1 * 32 * 8192 * 128 * 2                     # one [B, H, S, d] bf16 tensor
    lse = 1 * 32 * 8192 * 4
    # forward: read Q, K, V; write O, LSE
    assert bench.fwd_algorithmic_bytes(w) == 4 * t + lse
    # backward: read Q, K, V, O, dO, LSE; write dQ, dK, dV
    assert bench.bwd_algorithmic_bytes(w) == 8 * t + lse


def test_hbm_side_closed_form():
    got = bench.hbm_side(1e9, 3e11, 1.0, 1915.5, 6794.1)   # 1 GB in 1 ms
    assert got["achieved_gbs"] == pytest.approx(1000.0)
    assert got["frac"] == pytest.approx(1000.0 / 6794.1)
    assert got["intensity_flop_per_byte"] == pytest.approx(300.0)
    assert got["ridge_flop_per_byte"] == pytest.approx(1915.5e12 / 6794.1e9)
    assert bench.hbm_side(1e9, 3e11, 0.0, 1915.5, 6794.1) is None
    assert bench.hbm_side(0, 3e11, 1.0, 1915.5, 6794.1) is None


def test_cpu_model_is_text_or_none():
    m = bench.cpu_model()
    assert m is None or (isinstance(m, str) and m)
