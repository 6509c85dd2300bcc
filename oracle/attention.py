"""fp64 CPU oracle for scaled-dot-product attention with an optional causal
mask: forward (out, logsumexp) and backward (dQ, dK, dV).

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module. It shares no code with the CUDA path
and the CUDA path never calls it.

Inputs are numpy float64 arrays holding the values the GPU sees (bf16 / fp16 /
fp32 tensors widened exactly to double):

    q, dout : [B, Hq,  Sq,  d]
    k, v    : [B, Hkv, Skv, d]      Hq % Hkv == 0, G = Hq // Hkv

Sq and Skv are the query and key/value lengths (equal in self-attention).

Query head h reads key/value head h // G (grouped-query attention, as in
"Phase 14: Flash Attention 2 for SM120", section "GQA 支持"). dK and dV of a
key/value head are the sums over its G query heads.

What is computed (the plain definition, no tiling):

  * scores  s_ij = scale * <Q_i, K_j>; with causal masking s_ij = -inf for
    key position j > query position i ("Phase T14: 融合 Flash-Attention
    Kernel", section "什么是 flash-attention": standard attention
    O = softmax(causal(Q K^T / sqrt(d))) V, masked columns j > i; "FlashAttention
    与 SDPA Backend", section "先从 reference 语义出发"). When the key/value
    sequence is longer than the query sequence, query row i sits at position
    i + kv_offset with kv_offset = Skv - Sq, so the mask is j > i + kv_offset
    ("Phase 14: Flash Attention 2 for SM120", section "Causal Mask": the offset
    is kv_len - q_len, for a KV cache longer than Q). Causal masking needs
    Skv >= Sq: with fewer keys than queries the first rows would see no key at
    all and their softmax would be undefined.
  * P = row softmax of s, O = P V, and the natural-log logsumexp
    LSE_i = log sum_j exp(s_ij), the per-row statistic the forward keeps for
    the backward ("Phase T14", section "Key Design Decisions" item 2, L = m + log l).
  * backward through the softmax Jacobian written out:
    dV = P^T dO, dP = dO V^T, each row of dS = J_i^T dP_i with
    J_i = diag(P_i) - P_i P_i^T, dQ = scale * dS K, dK = scale * dS^T Q
    ("Phase T14", section "什么是 flash-attention", backward formulas, and
    item 3 of "Key Design Decisions" for the Jacobian form). The D shortcut
    (D_i = <dO_i, O_i>) is deliberately NOT used here; the tests check the
    identity D_i = sum_j P_ij dP_ij against this oracle instead.

`forward_tiled` restates the online-softmax recurrence (running max m,
running sum l, rescaled accumulator) as the pages give it, so that the tests
can check it against the plain definition.

Rows are processed a group at a time in `key_columns` only to bound memory;
each row is still the definition above.
"""
from __future__ import annotations

import numpy as np


def _check(q, k, v, causal=False):
    """Returns (B, Hq, Hkv, Sq, Skv, d)."""
    if q.ndim != 4 or k.shape != v.shape or q.shape[0] != k.shape[0] or \
            q.shape[3] != k.shape[3] or q.shape[1] % k.shape[1] != 0:
        raise ValueError(f"bad shapes q{q.shape} k{k.shape} v{v.shape}")
    if causal and k.shape[2] < q.shape[2]:
        raise ValueError("causal masking needs at least as many keys as queries")
    return q.shape[0], q.shape[1], k.shape[1], q.shape[2], k.shape[2], q.shape[3]


def _causal_mask(n_rows, n_cols, row0=0, offset=0):
    """True where key position j > query position i + offset (masked); the
    rows are query rows row0 .. row0 + n_rows - 1."""
    rows = np.arange(row0, row0 + n_rows)[:, None]
    cols = np.arange(n_cols)[None, :]
    return cols > rows + offset


def _softmax_rows(s):
    """Row softmax of s (entries may be -inf); returns (P, M, l) with
    P = exp(s - M) / l, M = row max, l = sum exp(s - M)."""
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    return e / l, m[:, 0], l[:, 0]


def head_probs(qh, kh, causal, scale):
    """Probabilities P [Sq, Skv] and LSE [Sq] of one (batch, query head)."""
    s = scale * (qh @ kh.T)
    if causal:
        s[_causal_mask(*s.shape, offset=kh.shape[0] - qh.shape[0])] = -np.inf
    p, m, l = _softmax_rows(s)
    return p, m + np.log(l)


def forward(q, k, v, causal=True, scale=None):
    """Dense forward: returns (out [B,Hq,Sq,d], lse [B,Hq,Sq]) in float64."""
    B, Hq, Hkv, Sq, _, d = _check(q, k, v, causal)
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    out = np.empty((B, Hq, Sq, d))
    lse = np.empty((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            p, lse[b, h] = head_probs(q[b, h], k[b, h // G], causal, scale)
            out[b, h] = p @ v[b, h // G]
    return out, lse


def softmax_jacobian(p_row):
    """Jacobian of softmax at probabilities p_row: J = diag(p) - p p^T."""
    return np.diag(p_row) - np.outer(p_row, p_row)


def _jacobian_vjp(p, dp):
    """Each row i of the result is J_i^T dp_i for J_i = softmax_jacobian(p_i),
    i.e. p_ij * dp_ij - p_ij * sum_k p_ik dp_ik (J is symmetric)."""
    return p * dp - p * (p * dp).sum(axis=1, keepdims=True)


def backward(q, k, v, dout, causal=True, scale=None):
    """Dense backward: returns (dq, dk, dv) in float64 (dk/dv summed over each
    key/value head's query-head group)."""
    B, Hq, Hkv, Sq, Skv, d = _check(q, k, v, causal)
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    dq = np.zeros((B, Hq, Sq, d))
    dk = np.zeros((B, Hkv, Skv, d))
    dv = np.zeros((B, Hkv, Skv, d))
    for b in range(B):
        for h in range(Hq):
            kvh = h // G
            p, _ = head_probs(q[b, h], k[b, kvh], causal, scale)
            dv[b, kvh] += p.T @ dout[b, h]
            dp = dout[b, h] @ v[b, kvh].T
            ds = _jacobian_vjp(p, dp)
            dq[b, h] = scale * (ds @ k[b, kvh])
            dk[b, kvh] += scale * (ds.T @ q[b, h])
    return dq, dk, dv


def forward_tiled(q, k, v, causal=True, scale=None, block_n=64):
    """Online-softmax forward over key/value tiles of width `block_n`.

    Restates the recurrence of "Phase T14", section "什么是 flash-attention",
    and the loop of "Phase 14: Flash Attention 2 for SM120", section "FA2 算法"
    (also "Flash Attention" on udemi.tech, Algorithm 1, and "FlashAttention 与
    SDPA Backend", section "Online softmax 的三个状态"): per query row keep a
    running max m, a running sum l and an accumulator acc; for each tile
    m_new = max(m, rowmax(s)), p = exp(s - m_new), l = l*exp(m - m_new) + sum p,
    acc = acc*exp(m - m_new) + p V_tile; finally out = acc / l and
    LSE = m + log l. Masked entries contribute p = 0.

    Query row i stands at position i + kv_offset, kv_offset = Skv - Sq
    ("Phase 14", section "Causal Mask").

    Returns (out, lse, m, l), all float64.
    """
    B, Hq, Hkv, Sq, Skv, d = _check(q, k, v, causal)
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    out = np.empty((B, Hq, Sq, d))
    lse = np.empty((B, Hq, Sq))
    m_all = np.empty((B, Hq, Sq))
    l_all = np.empty((B, Hq, Sq))
    query_pos = np.arange(Sq)[:, None] + (Skv - Sq)
    for b in range(B):
        for h in range(Hq):
            qh, kh, vh = q[b, h], k[b, h // G], v[b, h // G]
            m = np.full(Sq, -np.inf)
            l = np.zeros(Sq)
            acc = np.zeros((Sq, d))
            for start in range(0, Skv, block_n):
                end = min(start + block_n, Skv)
                s = scale * (qh @ kh[start:end].T)
                if causal:
                    key_pos = np.arange(start, end)[None, :]
                    s = np.where(key_pos > query_pos, -np.inf, s)
                m_new = np.maximum(m, s.max(axis=1))
                # a row with every key so far masked keeps m = -inf and l = 0
                finite = np.isfinite(m_new)
                m_safe = np.where(finite, m_new, 0.0)
                alpha = np.where(finite, np.exp(m - m_safe), 1.0)
                p = np.where(np.isfinite(s), np.exp(s - m_safe[:, None]), 0.0)
                l = l * alpha + p.sum(axis=1)
                acc = acc * alpha[:, None] + p @ vh[start:end]
                m = m_new
            out[b, h] = acc / l[:, None]
            lse[b, h] = m + np.log(l)
            m_all[b, h] = m
            l_all[b, h] = l
    return out, lse, m_all, l_all


def rows(q, k, v, dout, b, h, idx, causal=True, scale=None):
    """Forward and dQ of selected query rows of one (batch, query head).

    Row i needs only keys 0..i + kv_offset under causal masking (all keys
    otherwise), so this is O(Skv d) per row. Returns (out [n,d], lse [n],
    dq [n,d]).
    """
    _, Hq, Hkv, Sq, Skv, d = _check(q, k, v, causal)
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    kh, vh = k[b, h // G], v[b, h // G]
    out = np.empty((len(idx), d))
    lse = np.empty(len(idx))
    dq = np.empty((len(idx), d))
    for n, i in enumerate(idx):
        visible = i + 1 + (Skv - Sq) if causal else Skv
        s = scale * (kh[:visible] @ q[b, h, i])
        p, m, l = _softmax_rows(s[None, :])
        out[n] = p[0] @ vh[:visible]
        lse[n] = m[0] + np.log(l[0])
        dp = vh[:visible] @ dout[b, h, i]
        ds = _jacobian_vjp(p, dp[None, :])[0]
        dq[n] = scale * (ds @ kh[:visible])
    return out, lse, dq


def key_columns(q, k, v, dout, b, kvh, idx, causal=True, scale=None,
                row_block=512):
    """dK and dV of selected key positions of one (batch, key/value head),
    summed over the head's query-head group.

    Column j of dK needs dS_ij for every query row i, and each dS_ij needs the
    whole of row i (its softmax normaliser and sum_k P_ik dP_ik), so every row
    is evaluated; rows are taken `row_block` at a time to bound memory.
    Returns (dk [n,d], dv [n,d]).
    """
    _, Hq, Hkv, Sq, Skv, d = _check(q, k, v, causal)
    G = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    off = Skv - Sq
    idx = np.asarray(idx)
    kh, vh = k[b, kvh], v[b, kvh]
    dk = np.zeros((len(idx), d))
    dv = np.zeros((len(idx), d))
    for h in range(kvh * G, (kvh + 1) * G):
        for r0 in range(0, Sq, row_block):
            r1 = min(r0 + row_block, Sq)
            # keys beyond position r1 - 1 + kv_offset are masked for these rows
            ncol = r1 + off if causal else Skv
            sel = idx < ncol
            if not sel.any():
                continue
            s = scale * (q[b, h, r0:r1] @ kh[:ncol].T)
            if causal:
                s[_causal_mask(r1 - r0, ncol, r0, off)] = -np.inf
            p, _, _ = _softmax_rows(s)
            dp = dout[b, h, r0:r1] @ vh[:ncol].T
            ds = _jacobian_vjp(p, dp)
            cols = idx[sel]
            dk[sel] += scale * (ds[:, cols].T @ q[b, h, r0:r1])
            dv[sel] += p[:, cols].T @ dout[b, h, r0:r1]
    return dk, dv
