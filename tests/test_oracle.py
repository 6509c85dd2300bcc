"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test fixes the oracle to something the pages or the mathematics determine:
an independently written algorithm (the online-softmax recurrence), closed
forms, invariants, special cases that reduce to a library routine (PyTorch's
own CPU attention in float64), central finite differences, and brute force on
tiny inputs. `test_planted_mistakes_are_caught` plants plausible mistakes in
the oracle and checks that these pins catch them.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from oracle import attention as oa

RNG = np.random.default_rng(1234)


def rand(*shape, rng=None):
    return (rng or RNG).standard_normal(shape)


def rand_qkv(B, Hq, Hkv, S, d, rng=None):
    rng = rng or np.random.default_rng(B * 1000 + Hq * 100 + S * 10 + d)
    return (rand(B, Hq, S, d, rng=rng), rand(B, Hkv, S, d, rng=rng),
            rand(B, Hkv, S, d, rng=rng), rand(B, Hq, S, d, rng=rng))


SHAPES = [(1, 1, 1, 1, 4), (1, 2, 2, 5, 8), (1, 2, 1, 7, 4), (2, 4, 2, 40, 8),
          (1, 2, 2, 128, 16)]


# 1. tiled online softmax (the pages' recurrence) == plain definition
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("block_n", [1, 3, 64, 128])
def test_tiled_matches_dense(shape, causal, block_n):
    q, k, v, _ = rand_qkv(*shape)
    out, lse = oracle.forward(q, k, v, causal)
    out_t, lse_t, m, l = oracle.forward_tiled(q, k, v, causal, block_n=block_n)
    assert np.abs(out - out_t).max() <= 1e-12
    assert np.abs(lse - lse_t).max() <= 1e-12
    assert np.allclose(lse_t, m + np.log(l), atol=1e-13, rtol=0)


# 2. every probability row sums to one and masked entries are zero
@pytest.mark.parametrize("causal", [True, False])
def test_row_sums_and_mask(causal):
    q, k, _, _ = rand_qkv(1, 1, 1, 33, 8)
    p, _ = oracle.head_probs(q[0, 0], k[0, 0], causal, 0.3)
    assert np.abs(p.sum(axis=1) - 1).max() <= 1e-14
    if causal:
        assert np.all(p[np.triu_indices(33, 1)] == 0)
        assert np.all(p[np.tril_indices(33)] > 0)


# 3. causal row 0 sees only key 0: out_0 = V_0 exactly and LSE_0 = s_00
def test_causal_row_zero():
    q, k, v, _ = rand_qkv(2, 4, 2, 19, 8)
    out, lse = oracle.forward(q, k, v, True, scale=0.7)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(out[b, h, 0], v[b, h // 2, 0])
            assert lse[b, h, 0] == pytest.approx(0.7 * q[b, h, 0] @ k[b, h // 2, 0],
                                                 abs=1e-14)


# 4. D_i = <dO_i, O_i> equals sum_j P_ij dP_ij ("Phase T14", Key Design Decisions, item 3)
@pytest.mark.parametrize("causal", [True, False])
def test_d_identity(causal):
    q, k, v, do = rand_qkv(1, 2, 1, 50, 8)
    out, _ = oracle.forward(q, k, v, causal)
    for h in range(2):
        p, _ = oracle.head_probs(q[0, h], k[0, 0], causal, 1 / math.sqrt(8))
        dp = do[0, h] @ v[0, 0].T
        lhs = (do[0, h] * out[0, h]).sum(axis=1)
        rhs = (p * dp).sum(axis=1)
        assert np.abs(lhs - rhs).max() <= 1e-12


# 5. central finite differences of F = sum(W * O) ("Phase T14", section 验证方法)
@pytest.mark.parametrize("B,Hq,Hkv,S,d", [(1, 1, 1, 1, 4), (1, 1, 1, 3, 4),
                                          (1, 2, 2, 5, 8), (1, 2, 1, 5, 4),
                                          (1, 1, 1, 17, 4)])
@pytest.mark.parametrize("causal", [True, False])
def test_finite_differences(B, Hq, Hkv, S, d, causal):
    q, k, v, w = rand_qkv(B, Hq, Hkv, S, d)
    scale = 0.9

    def F(q_, k_, v_):
        return float((w * oracle.forward(q_, k_, v_, causal, scale)[0]).sum())

    dq, dk, dv = oracle.backward(q, k, v, w, causal, scale)
    eps = 1e-6
    for x, g, pos in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args = [q, k, v]
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args[pos] = xp
            fp = F(*args)
            args[pos] = xm
            fm = F(*args)
            num[idx] = (fp - fm) / (2 * eps)
        assert np.abs(num - g).max() <= 1e-7 * max(1.0, np.abs(g).max())


# 6a. PyTorch's CPU attention in float64 is an independent implementation of the
#     same definition (forward, logsumexp and autograd backward)
@pytest.mark.parametrize("shape", [(1, 2, 2, 40, 8), (2, 4, 2, 65, 16), (1, 8, 1, 31, 8)])
@pytest.mark.parametrize("causal", [True, False])
def test_matches_torch_sdpa_float64(shape, causal):
    B, Hq, Hkv, S, d = shape
    q, k, v, do = rand_qkv(*shape)
    scale = 1 / math.sqrt(d)
    out, lse = oracle.forward(q, k, v, causal, scale)
    dq, dk, dv = oracle.backward(q, k, v, do, causal, scale)

    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = Hq // Hkv
    tk_rep = tk.repeat_interleave(G, dim=1)
    tv_rep = tv.repeat_interleave(G, dim=1)
    tout = torch.nn.functional.scaled_dot_product_attention(
        tq, tk_rep, tv_rep, is_causal=causal, scale=scale)
    tout.backward(torch.tensor(do))
    sc = (tq @ tk_rep.transpose(-1, -2)) * scale
    if causal:
        sc = sc.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), -math.inf)
    tlse = torch.logsumexp(sc, dim=-1)

    assert np.abs(out - tout.detach().numpy()).max() <= 1e-12
    assert np.abs(lse - tlse.detach().numpy()).max() <= 1e-12
    assert np.abs(dq - tq.grad.numpy()).max() <= 1e-12
    assert np.abs(dk - tk.grad.numpy()).max() <= 1e-12
    assert np.abs(dv - tv.grad.numpy()).max() <= 1e-12


# 6b. special cases with closed forms
def test_single_position_returns_v():
    q, k, v, do = rand_qkv(1, 2, 2, 1, 8)
    out, lse = oracle.forward(q, k, v, True)
    assert np.array_equal(out, v)
    dq, dk, dv = oracle.backward(q, k, v, do, True)
    assert np.abs(dq).max() == 0 and np.abs(dk).max() == 0
    assert np.array_equal(dv, do)


def test_zero_queries_give_prefix_means():
    _, k, v, _ = rand_qkv(1, 1, 1, 12, 4)
    q = np.zeros((1, 1, 12, 4))
    out, lse = oracle.forward(q, k, v, True)
    prefix_mean = np.cumsum(v[0, 0], axis=0) / np.arange(1, 13)[:, None]
    assert np.abs(out[0, 0] - prefix_mean).max() <= 1e-14
    assert np.abs(lse[0, 0] - np.log(np.arange(1, 13))).max() <= 1e-14


def test_equal_keys_non_causal_give_mean():
    q, _, v, _ = rand_qkv(1, 1, 1, 9, 4)
    k = np.tile(rand(1, 1, 1, 4), (1, 1, 9, 1))
    out, _ = oracle.forward(q, k, v, False)
    assert np.abs(out[0, 0] - v[0, 0].mean(axis=0)).max() <= 1e-14


def test_large_scale_is_hard_argmax():
    q, k, v, _ = rand_qkv(1, 1, 1, 16, 4)
    out, _ = oracle.forward(q, k, v, True, scale=1e4)
    s = q[0, 0] @ k[0, 0].T
    s[np.triu_indices(16, 1)] = -np.inf
    arg = s.argmax(axis=1)
    assert np.abs(out[0, 0] - v[0, 0][arg]).max() <= 1e-6


def test_two_position_closed_form():
    # scale 1, d = 1: row 1 has scores (0, ln 3) -> weights (1/4, 3/4)
    q = np.array([1.0, 1.0]).reshape(1, 1, 2, 1)
    k = np.array([0.0, math.log(3.0)]).reshape(1, 1, 2, 1)
    v = np.array([2.0, -6.0]).reshape(1, 1, 2, 1)
    g = np.array([0.5, 4.0]).reshape(1, 1, 2, 1)
    out, lse = oracle.forward(q, k, v, True, scale=1.0)
    assert out[0, 0, 0, 0] == pytest.approx(2.0, abs=1e-15)
    assert out[0, 0, 1, 0] == pytest.approx(0.25 * 2 + 0.75 * -6, abs=1e-14)
    assert lse[0, 0, 0] == pytest.approx(0.0, abs=1e-15)
    assert lse[0, 0, 1] == pytest.approx(math.log(4.0), abs=1e-14)
    dq, dk, dv = oracle.backward(q, k, v, g, True, scale=1.0)
    # row 1: dP = g1*v = (8, -24), D = g1*out1 = -16, dS = p*(dP - D) = (6, -6)
    assert dq[0, 0, 1, 0] == pytest.approx(6 * 0.0 + -6 * math.log(3.0), abs=1e-13)
    assert dq[0, 0, 0, 0] == pytest.approx(0.0, abs=1e-15)
    assert dk[0, 0, 0, 0] == pytest.approx(6 * 1.0, abs=1e-13)
    assert dk[0, 0, 1, 0] == pytest.approx(-6 * 1.0, abs=1e-13)
    assert dv[0, 0, 0, 0] == pytest.approx(1.0 * 0.5 + 0.25 * 4.0, abs=1e-14)
    assert dv[0, 0, 1, 0] == pytest.approx(0.75 * 4.0, abs=1e-14)


# 6c. grouped-query attention == multi-head attention on repeated K/V heads, with
#     dK/dV of a shared head the sum over its group
def test_gqa_equals_repeated_heads():
    q, k, v, do = rand_qkv(2, 8, 2, 23, 8)
    out, lse = oracle.forward(q, k, v, True)
    kr, vr = np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1)
    out_r, lse_r = oracle.forward(q, kr, vr, True)
    assert np.array_equal(out, out_r) and np.array_equal(lse, lse_r)
    dq, dk, dv = oracle.backward(q, k, v, do, True)
    dq_r, dk_r, dv_r = oracle.backward(q, kr, vr, do, True)
    assert np.abs(dq - dq_r).max() <= 1e-13
    assert np.abs(dk - dk_r.reshape(2, 2, 4, 23, 8).sum(axis=2)).max() <= 1e-12
    assert np.abs(dv - dv_r.reshape(2, 2, 4, 23, 8).sum(axis=2)).max() <= 1e-12


# 6d. the softmax Jacobian form used by the backward, checked entry by entry
def test_jacobian_vector_product_brute_force():
    p, _ = oracle.head_probs(rand(6, 3), rand(6, 3), True, 1.0)
    dp = rand(6, 6)
    ds = oa._jacobian_vjp(p, dp)
    for i in range(6):
        J = np.zeros((6, 6))
        for a in range(6):
            for c in range(6):
                J[a, c] = p[i, a] * ((a == c) - p[i, c])   # d p_a / d s_c
        assert np.abs(ds[i] - J.T @ dp[i]).max() <= 1e-15
        # the oracle's explicit Jacobian is the same matrix
        assert np.abs(oa.softmax_jacobian(p[i]) - J).max() <= 1e-15


# 6e. the explicit softmax Jacobian against central finite differences of a
#     library softmax (scipy), at random score rows including a masked entry
def test_softmax_jacobian_finite_differences():
    from scipy.special import softmax
    rng = np.random.default_rng(77)
    eps = 1e-6
    for n in (1, 2, 5, 9):
        s = rng.standard_normal(n) * 2.0
        if n > 2:
            s[-1] = -np.inf            # a masked key: its probability and derivatives are 0
        fin = np.isfinite(s)
        J_fd = np.zeros((n, n))
        for c in np.flatnonzero(fin):
            e = np.zeros(n)
            e[c] = eps
            J_fd[:, c] = (softmax(s + e) - softmax(s - e)) / (2 * eps)
        J = oa.softmax_jacobian(softmax(s))
        assert np.abs(J - J_fd).max() <= 1e-9, n
        assert np.abs(J.sum(axis=0)).max() <= 1e-15   # columns sum to 0 (probabilities sum to 1)


# 7. sampled-row and sampled-column evaluators agree with the dense oracle
@pytest.mark.parametrize("causal", [True, False])
def test_sampled_evaluators(causal):
    q, k, v, do = rand_qkv(2, 4, 2, 300, 8)
    out, lse = oracle.forward(q, k, v, causal)
    dq, dk, dv = oracle.backward(q, k, v, do, causal)
    idx = fa_inputs.sample_rows(300, 20, seed=5)
    for b, h in ((0, 0), (1, 3)):
        o_r, l_r, dq_r = oracle.rows(q, k, v, do, b, h, idx, causal)
        assert np.abs(o_r - out[b, h, idx]).max() <= 1e-13
        assert np.abs(l_r - lse[b, h, idx]).max() <= 1e-13
        assert np.abs(dq_r - dq[b, h, idx]).max() <= 1e-12
    for b, kvh in ((0, 1), (1, 0)):
        dk_c, dv_c = oracle.key_columns(q, k, v, do, b, kvh, idx, causal, row_block=64)
        assert np.abs(dk_c - dk[b, kvh, idx]).max() <= 1e-12
        assert np.abs(dv_c - dv[b, kvh, idx]).max() <= 1e-12


# 8. the teaching example of "FlashAttention 与 SDPA Backend" (section
#    可运行 online-softmax reference): fp32 [1,2,7,4], key tile width 3, tiled
#    vs dense within rtol=1e-5 / atol=1e-6 (the page printed a max-abs
#    difference of 1.192e-07 for its own fp32 run)
def test_teaching_example_fp32():
    import json, os
    fx = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "online_softmax_teaching_case.json")))
    rng = np.random.default_rng(71)
    shape = tuple(fx["shape"])
    q, k, v = (rng.standard_normal(shape).astype(np.float32) for _ in range(3))
    dense, _ = oracle.forward(*(x.astype(np.float64) for x in (q, k, v)), True)
    tiled, _, m, l = oracle.forward_tiled(*(x.astype(np.float64) for x in (q, k, v)),
                                          True, block_n=fx["tile_n"])
    assert m.shape == l.shape == shape[:3]
    diff = np.abs(dense.astype(np.float32) - tiled.astype(np.float32)).max()
    assert diff <= fx["atol"] + fx["rtol"] * np.abs(dense).max()


# 9. planted mistakes: each must break at least one of the pins above
def _pins_pass():
    try:
        test_causal_row_zero()
        test_two_position_closed_form()
        for causal in (True, False):
            test_matches_torch_sdpa_float64((1, 2, 2, 40, 8), causal)
        test_finite_differences(1, 2, 1, 5, 4, True)
        test_kv_offset_matches_torch_lower_right_bias((1, 2, 1, 5, 12, 4), True)
        test_softmax_jacobian_finite_differences()
    except Exception:   # a failed assertion, or NaNs tripping a comparison
        return False
    return True


def _softmax_rows_lse_without_max(s):
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=1, keepdims=True), np.zeros(s.shape[0]), e.sum(axis=1)


def test_planted_mistakes_are_caught(monkeypatch):
    assert _pins_pass()
    mutants = {
        "mask includes the diagonal": ("_causal_mask",
            lambda n, c, r0=0, offset=0: np.arange(c)[None, :] >= np.arange(r0, r0 + n)[:, None] + offset),
        "mask off by one the other way": ("_causal_mask",
            lambda n, c, r0=0, offset=0: np.arange(c)[None, :] > np.arange(r0, r0 + n)[:, None] + offset + 1),
        "kv_offset ignored (top-left alignment)": ("_causal_mask",
            lambda n, c, r0=0, offset=0: np.arange(c)[None, :] > np.arange(r0, r0 + n)[:, None]),
        "kv_offset with the wrong sign": ("_causal_mask",
            lambda n, c, r0=0, offset=0: np.arange(c)[None, :] > np.arange(r0, r0 + n)[:, None] - offset),
        "Jacobian term dropped": ("_jacobian_vjp", lambda p, dp: p * dp),
        "Jacobian sign flipped": ("_jacobian_vjp",
            lambda p, dp: p * dp + p * (p * dp).sum(axis=1, keepdims=True)),
        "explicit Jacobian sign flipped": ("softmax_jacobian",
            lambda p: np.diag(p) + np.outer(p, p)),
        "explicit Jacobian diagonal dropped": ("softmax_jacobian",
            lambda p: -np.outer(p, p)),
        "logsumexp missing the max term": ("_softmax_rows",
                                           _softmax_rows_lse_without_max),
    }
    for name, (attr, fn) in mutants.items():
        # some mutants mask whole rows; their NaNs are what the pins must catch
        with monkeypatch.context() as mp, np.errstate(invalid="ignore"):
            mp.setattr(oa, attr, fn)
            assert not _pins_pass(), f"planted mistake not caught: {name}"


def test_workload_recipes():
    w = fa_inputs.WORKLOADS["long_8k"]
    small = fa_inputs.Workload("t", "bf16", 1, 2, 2, 1100, 8, seed=3,
                               value_scale=0.5, spike_every=512, spike_scale=8.0)
    q, k, v, do = fa_inputs.make_inputs(small)
    assert q.dtype == torch.bfloat16 and k.shape == (1, 2, 1100, 8)
    ratio = k[..., ::512, :].float().abs().mean() / k.float().abs().mean()
    assert ratio > 5
    assert w.S == 8192 and w.d == 128 and w.Hq == w.Hkv == 32
    rows = fa_inputs.sample_rows(8192, 256, seed=0)
    assert len(rows) == 256 and {0, 127, 128, 511, 512, 8191} <= set(rows)


# 10. separate query and key/value lengths. Query row i stands at position
#     i + kv_offset, kv_offset = Skv - Sq ("Phase 14: Flash Attention 2 for
#     SM120", section "Causal Mask"), i.e. the causal mask is aligned to the
#     last key. PyTorch's `causal_lower_right` attention bias is an independent
#     definition of exactly that alignment.
def rand_qkv_kv(B, Hq, Hkv, Sq, Skv, d):
    rng = np.random.default_rng(B * 7919 + Hq * 131 + Sq * 17 + Skv * 3 + d)
    return (rand(B, Hq, Sq, d, rng=rng), rand(B, Hkv, Skv, d, rng=rng),
            rand(B, Hkv, Skv, d, rng=rng), rand(B, Hq, Sq, d, rng=rng))


KV_SHAPES = [(1, 2, 2, 1, 9, 8), (1, 2, 1, 5, 12, 4), (2, 4, 2, 17, 40, 8),
             (1, 2, 2, 33, 33, 8), (1, 1, 1, 3, 130, 4)]


@pytest.mark.parametrize("shape", KV_SHAPES)
@pytest.mark.parametrize("causal", [True, False])
def test_kv_offset_matches_torch_lower_right_bias(shape, causal):
    from torch.nn.attention.bias import causal_lower_right
    B, Hq, Hkv, Sq, Skv, d = shape
    q, k, v, do = rand_qkv_kv(*shape)
    scale = 0.7
    out, lse = oracle.forward(q, k, v, causal, scale)
    dq, dk, dv = oracle.backward(q, k, v, do, causal, scale)

    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = Hq // Hkv
    tk_rep = tk.repeat_interleave(G, dim=1)
    tv_rep = tv.repeat_interleave(G, dim=1)
    bias = causal_lower_right(Sq, Skv) if causal else None
    tout = torch.nn.functional.scaled_dot_product_attention(
        tq, tk_rep, tv_rep, attn_mask=bias, scale=scale)
    tout.backward(torch.tensor(do))
    sc = (tq @ tk_rep.transpose(-1, -2)) * scale
    if causal:
        sc = sc.masked_fill(~bias._materialize(), -math.inf)
    tlse = torch.logsumexp(sc, dim=-1)

    assert np.abs(out - tout.detach().numpy()).max() <= 1e-12
    assert np.abs(lse - tlse.detach().numpy()).max() <= 1e-12
    assert np.abs(dq - tq.grad.numpy()).max() <= 1e-12
    assert np.abs(dk - tk.grad.numpy()).max() <= 1e-12
    assert np.abs(dv - tv.grad.numpy()).max() <= 1e-12


@pytest.mark.parametrize("shape", [(1, 2, 1, 5, 12, 4), (2, 4, 2, 17, 40, 8)])
def test_query_chunk_is_the_tail_of_self_attention(shape):
    """A chunk of the last Sq queries against all Skv keys gives the last Sq
    rows of self-attention over Skv positions, forward and backward (with dO
    zero on the rows outside the chunk)."""
    B, Hq, Hkv, Sq, Skv, d = shape
    rng = np.random.default_rng(99)
    q_full = rand(B, Hq, Skv, d, rng=rng)
    k, v = rand(B, Hkv, Skv, d, rng=rng), rand(B, Hkv, Skv, d, rng=rng)
    do = rand(B, Hq, Sq, d, rng=rng)
    tail = slice(Skv - Sq, Skv)
    out_c, lse_c = oracle.forward(q_full[:, :, tail], k, v, True)
    out_f, lse_f = oracle.forward(q_full, k, v, True)
    assert np.abs(out_c - out_f[:, :, tail]).max() <= 1e-13
    assert np.abs(lse_c - lse_f[:, :, tail]).max() <= 1e-13
    do_full = np.zeros_like(q_full)
    do_full[:, :, tail] = do
    dq_c, dk_c, dv_c = oracle.backward(q_full[:, :, tail], k, v, do, True)
    dq_f, dk_f, dv_f = oracle.backward(q_full, k, v, do_full, True)
    assert np.abs(dq_c - dq_f[:, :, tail]).max() <= 1e-13
    assert np.abs(dk_c - dk_f).max() <= 1e-13
    assert np.abs(dv_c - dv_f).max() <= 1e-13


def test_single_query_sees_every_key():
    """Sq = 1 (one new token against a longer key/value sequence): the causal
    mask hides nothing, so the result is the unmasked one."""
    q, k, v, do = rand_qkv_kv(1, 2, 1, 1, 37, 8)
    for a, b in zip(oracle.forward(q, k, v, True), oracle.forward(q, k, v, False)):
        assert np.array_equal(a, b)
    for a, b in zip(oracle.backward(q, k, v, do, True), oracle.backward(q, k, v, do, False)):
        assert np.array_equal(a, b)


def test_causal_needs_keys_for_every_query():
    q, k, v, do = rand_qkv_kv(1, 1, 1, 9, 4, 4)
    with pytest.raises(ValueError):
        oracle.forward(q, k, v, True)
    out, lse = oracle.forward(q, k, v, False)      # unmasked: any lengths
    assert out.shape == (1, 1, 9, 4) and np.isfinite(lse).all()


@pytest.mark.parametrize("shape", KV_SHAPES)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("block_n", [1, 3, 64])
def test_tiled_matches_dense_kv_lengths(shape, causal, block_n):
    q, k, v, _ = rand_qkv_kv(*shape)
    out, lse = oracle.forward(q, k, v, causal)
    out_t, lse_t, _, _ = oracle.forward_tiled(q, k, v, causal, block_n=block_n)
    assert np.abs(out - out_t).max() <= 1e-12
    assert np.abs(lse - lse_t).max() <= 1e-12


@pytest.mark.parametrize("causal", [True, False])
def test_finite_differences_kv_lengths(causal):
    q, k, v, w = rand_qkv_kv(1, 2, 1, 3, 7, 4)
    scale = 0.8

    def F(q_, k_, v_):
        return float((w * oracle.forward(q_, k_, v_, causal, scale)[0]).sum())

    dq, dk, dv = oracle.backward(q, k, v, w, causal, scale)
    eps = 1e-6
    for x, g, pos in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args = [q, k, v]
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args[pos] = xp
            fp = F(*args)
            args[pos] = xm
            fm = F(*args)
            num[idx] = (fp - fm) / (2 * eps)
        assert np.abs(num - g).max() <= 1e-7 * max(1.0, np.abs(g).max())


@pytest.mark.parametrize("causal", [True, False])
def test_sampled_evaluators_kv_lengths(causal):
    q, k, v, do = rand_qkv_kv(1, 4, 2, 150, 420, 8)
    out, lse = oracle.forward(q, k, v, causal)
    dq, dk, dv = oracle.backward(q, k, v, do, causal)
    qidx = fa_inputs.sample_rows(150, 20, seed=6)
    kidx = fa_inputs.sample_rows(420, 30, seed=7)
    for h in (0, 3):
        o_r, l_r, dq_r = oracle.rows(q, k, v, do, 0, h, qidx, causal)
        assert np.abs(o_r - out[0, h, qidx]).max() <= 1e-13
        assert np.abs(l_r - lse[0, h, qidx]).max() <= 1e-13
        assert np.abs(dq_r - dq[0, h, qidx]).max() <= 1e-12
    for kvh in (0, 1):
        dk_c, dv_c = oracle.key_columns(q, k, v, do, 0, kvh, kidx, causal, row_block=64)
        assert np.abs(dk_c - dk[0, kvh, kidx]).max() <= 1e-12
        assert np.abs(dv_c - dv[0, kvh, kidx]).max() <= 1e-12


def test_kv_length_workload_recipes():
    w = fa_inputs.WORKLOADS["prefill_8k"]
    assert (w.S, w.kv_len, w.Hq, w.Hkv, w.d, w.causal) == (2048, 8192, 32, 8, 128, True)
    small = fa_inputs.Workload("t", "bf16", 1, 4, 2, 10, 8, seed=5, Skv=30)
    q, k, v, do = fa_inputs.make_inputs(small)
    assert q.shape == do.shape == (1, 4, 10, 8) and k.shape == v.shape == (1, 2, 30, 8)
    for name in ("long_8k_nc", "gqa_qwen3_nc"):
        nc, c = fa_inputs.WORKLOADS[name], fa_inputs.WORKLOADS[name[:-3]]
        assert not nc.causal and dataclasses.replace(nc, name=c.name, causal=True) == c
