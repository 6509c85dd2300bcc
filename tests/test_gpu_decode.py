"""GPU parity for the split-KV forward (fa_fwd_splitkv: few query rows against
a long key/value sequence) against the fp64 oracle, same bars as the other
forward tests (tests/parity.py). The causal mask is aligned to the last key
(query row s at position s + Skv - Sq, "Phase 14: Flash Attention 2 for
SM120", section Causal Mask).

Edge cases: one key; ragged last tiles; G * Sq = 128 (a full query tile);
ranges in which some rows see no key (Sq = 16 over 130 keys in two ranges);
one range (direct write, no merge); as many ranges as key tiles; a requested
range count above the tile count (reduced); unmasked; fp16; fp32 (plain
path). Full size: decode_8k (every row) and spec_32k, in the launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from parity import check_fwd, f64

pytestmark = pytest.mark.gpu

DECODE_EDGE = [
    # B, Hq, Hkv, Sq, Skv, d, dtype, causal, n_splits
    (1, 1, 1, 1, 1, 64, "bf16", True, 0),
    (1, 4, 1, 1, 129, 128, "bf16", True, 0),
    (2, 8, 2, 1, 1000, 128, "bf16", True, 0),
    (1, 8, 2, 3, 777, 64, "fp16", True, 0),
    (1, 8, 1, 16, 4096, 128, "bf16", True, 0),     # R = G * Sq = 128
    (1, 4, 4, 16, 130, 128, "bf16", True, 2),      # rows 0-13 see no key of range 2
    (1, 2, 1, 2, 5000, 128, "bf16", False, 5),
    (3, 6, 3, 1, 2048, 64, "bf16", True, 1),       # one range: no merge
    (1, 4, 2, 8, 8192, 128, "fp16", True, 64),     # one range per key tile
    (1, 4, 2, 1, 640, 128, "bf16", True, 100),     # more ranges requested than tiles
    (1, 2, 2, 1, 300, 128, "fp32", True, 0),
]


def run_decode(fa, q, k, v, causal, scale, n_splits):
    dev = torch.device("cuda", 0)
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    out, lse = fa.decode_forward(qd, kd, vd, causal, scale, n_splits)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    return {"out": f64(out), "lse": f64(lse)}


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,d,dtype,causal,n_splits", DECODE_EDGE)
def test_decode_edge(fa, B, Hq, Hkv, Sq, Skv, d, dtype, causal, n_splits):
    q, k, v, _ = fa_inputs.make_custom(B, Hq, Hkv, Sq, d, dtype, seed=Skv + 31 * Sq, Skv=Skv)
    scale = 1.0 / np.sqrt(d)
    got = run_decode(fa, q, k, v, causal, scale, n_splits)
    out_ref, lse_ref = oracle.forward(*map(f64, (q, k, v)), causal, scale)
    check_fwd(got, out_ref, lse_ref)


def test_decode_range_count_does_not_change_the_result(fa):
    """Different numbers of key ranges give the same result within rounding
    of the fp32 partials (and both pass the oracle bars)."""
    q, k, v, _ = fa_inputs.make_custom(2, 8, 2, 2, 128, "bf16", seed=9, Skv=3000)
    scale = 1.0 / np.sqrt(128)
    ref = oracle.forward(*map(f64, (q, k, v)), True, scale)
    outs = []
    for n in (1, 3, 24):
        got = run_decode(fa, q, k, v, True, scale, n)
        check_fwd(got, *ref)
        outs.append(got)
    for o in outs[1:]:
        assert np.abs(o["out"] - outs[0]["out"]).max() <= 1e-2
        assert np.abs(o["lse"] - outs[0]["lse"]).max() <= 1e-4


@pytest.mark.parametrize("name", ["decode_8k", "spec_32k"])
def test_decode_workload(fa, name):
    w = fa_inputs.WORKLOADS[name]
    q, k, v = fa_inputs.make_inputs(w, with_dout=False)
    got = run_decode(fa, q, k, v, w.causal, w.scale, 0)
    out_ref, lse_ref = oracle.forward(*map(f64, (q, k, v)), w.causal, w.scale)
    check_fwd(got, out_ref, lse_ref)


# ------------------------------------------------------- paged key/value --
PAGED = [
    # B, Hq, Hkv, Sq, Skv, d, dtype, causal, block_size, n_splits
    (2, 8, 2, 1, 1000, 128, "bf16", True, 16, 0),
    (3, 4, 4, 2, 777, 64, "fp16", True, 32, 3),
    (1, 8, 1, 16, 4096, 128, "bf16", True, 64, 0),
    (2, 4, 2, 1, 300, 128, "bf16", False, 128, 0),
    (2, 8, 2, 4, 2500, 128, "bf16", True, 256, 2),
    (1, 2, 1, 1, 5000, 128, "bf16", True, 1024, 0),
]


def run_paged(fa, q, k, v, causal, scale, block_size, n_splits, seed):
    dev = torch.device("cuda", 0)
    kc, vc, table, _ = fa_inputs.make_paged(k, v, block_size, seed)
    qd, kcd, vcd, td = (x.to(dev) for x in (q, kc, vc, table))
    out, lse = fa.decode_forward_paged(qd, kcd, vcd, td, k.shape[2], causal, scale, n_splits)
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    return {"out": f64(out), "lse": f64(lse)}


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,d,dtype,causal,block_size,n_splits", PAGED)
def test_decode_paged(fa, B, Hq, Hkv, Sq, Skv, d, dtype, causal, block_size, n_splits):
    """The paged cache holds the same keys and values at scattered blocks
    (unused rows and blocks hold 1000.0, which must never be read)."""
    q, k, v, _ = fa_inputs.make_custom(B, Hq, Hkv, Sq, d, dtype, seed=Skv + block_size, Skv=Skv)
    scale = 1.0 / np.sqrt(d)
    got = run_paged(fa, q, k, v, causal, scale, block_size, n_splits, seed=block_size)
    out_ref, lse_ref = oracle.forward(*map(f64, (q, k, v)), causal, scale)
    check_fwd(got, out_ref, lse_ref)


def test_decode_paged_out_of_range_entries_read_zeros(fa):
    """A block-table entry outside [0, num_blocks) reads as a zero block: the
    result equals the oracle on K and V with those positions zeroed."""
    dev = torch.device("cuda", 0)
    q, k, v, _ = fa_inputs.make_custom(1, 4, 2, 1, 128, "bf16", seed=3, Skv=512)
    kc, vc, table, nb = fa_inputs.make_paged(k, v, 64, seed=4)
    table[0, 2] = nb + 5          # keys 128..191 read as zeros
    k0, v0 = k.clone(), v.clone()
    k0[:, :, 128:192] = 0
    v0[:, :, 128:192] = 0
    qd, kcd, vcd, td = (x.to(dev) for x in (q, kc, vc, table))
    out, lse = fa.decode_forward_paged(qd, kcd, vcd, td, 512, True, 1 / np.sqrt(128))
    torch.cuda.synchronize()
    assert fa.fa_last_device_status() == 0
    ref = oracle.forward(*map(f64, (q, k0, v0)), True, 1 / np.sqrt(128))
    check_fwd({"out": f64(out), "lse": f64(lse)}, *ref)


def test_decode_paged_workload(fa):
    w = fa_inputs.WORKLOADS["decode_8k_paged"]
    q, k, v = fa_inputs.make_inputs(w, with_dout=False)
    got = run_paged(fa, q, k, v, w.causal, w.scale, w.page_size, 0, seed=w.page_size)
    out_ref, lse_ref = oracle.forward(*map(f64, (q, k, v)), w.causal, w.scale)
    check_fwd(got, out_ref, lse_ref)
