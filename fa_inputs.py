"""Seeded synthetic inputs for causal attention, shared by the CUDA path's tests,
the benchmark and the oracle's tests.

This module holds no attention arithmetic: it only names the workloads and
draws their Q, K, V and dO tensors on the CPU from a seeded torch generator,
rounded to the workload's storage dtype. Everything that consumes the tensors
(the CUDA path, the fp64 oracle) receives the same rounded values.

Workloads (shapes in [B, H, S, d] order, Q/dO with Hq heads, K/V with Hkv):

  tiny_fp32    fp32,  B=1 Hq=Hkv=2  S=128   d=64,  N(0,1), seed 0
  gpt2_small   bf16,  B=8 Hq=Hkv=12 S=1024  d=64,  N(0,1), seed 1
  gqa_qwen3    bf16,  B=4 Hq=32 Hkv=8 S=2048 d=128, N(0,1), seed 2
  long_8k      bf16,  B=1 Hq=Hkv=32 S=8192  d=128, 0.5*N(0,1) with every
               512th key (positions 0, 512, 1024, ...) scaled by 8, seed 3
  fp16_32k     fp16,  B=1 Hq=Hkv=8  S=32768 d=64,  N(0,1), seed 4, forward only
  gqa_qwen3_nc gqa_qwen3 without the causal mask (same draws)
  long_8k_nc   long_8k without the causal mask (same draws)
  prefill_8k   bf16,  B=1 Hq=32 Hkv=8 Sq=2048 Skv=8192 d=128, N(0,1), seed 5:
               a 2048-query chunk at the end of an 8192-position context
               (causal mask aligned to the last key, kv_offset = Skv - Sq)
  decode_8k    bf16,  B=16 Hq=32 Hkv=8 Sq=1 Skv=8192 d=128, N(0,1), seed 6,
               forward only: one new token per sequence over an 8192-key cache
  spec_32k     bf16,  B=2 Hq=32 Hkv=8 Sq=4 Skv=32768 d=128, N(0,1), seed 7,
               forward only: four new tokens over a 32768-key cache
  decode_8k_paged  decode_8k with its cache in 64-key blocks at seeded random
               places of a shared pool (make_paged, seed 64)

All use scale = 1/sqrt(d); all but the *_nc workloads use causal masking.
S is the query length; K and V have `kv_len` rows (S unless Skv is given).
"""
from __future__ import annotations

import dataclasses
import math

import torch

DTYPES = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str
    B: int
    Hq: int
    Hkv: int
    S: int
    d: int
    seed: int
    causal: bool = True
    backward: bool = True
    value_scale: float = 1.0      # multiplies every N(0,1) draw
    spike_every: int = 0          # if > 0: K rows at positions % spike_every == 0 ...
    spike_scale: float = 1.0      # ... are multiplied by this before rounding
    Skv: int = 0                  # key/value length; 0 means the same as S
    decode: bool = False          # few query rows: timed through the split-KV forward
    page_size: int = 0            # > 0: K/V in a paged cache of blocks of this many keys

    @property
    def kv_len(self) -> int:
        return self.Skv or self.S

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def describe(self) -> str:
        lens = f"S={self.S}" if self.kv_len == self.S else f"Sq={self.S} Skv={self.kv_len}"
        s = (f"{self.name}: {self.dtype} B={self.B} Hq={self.Hq} Hkv={self.Hkv} "
             f"{lens} d={self.d} causal={int(self.causal)} seed={self.seed}")
        if self.value_scale != 1.0:
            s += f" values={self.value_scale}*N(0,1)"
        if self.spike_every:
            s += f" K[j]*={self.spike_scale} for j%{self.spike_every}==0"
        return s


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_fp32", "fp32", 1, 2, 2, 128, 64, seed=0),
        Workload("gpt2_small", "bf16", 8, 12, 12, 1024, 64, seed=1),
        Workload("gqa_qwen3", "bf16", 4, 32, 8, 2048, 128, seed=2),
        Workload("long_8k", "bf16", 1, 32, 32, 8192, 128, seed=3,
                 value_scale=0.5, spike_every=512, spike_scale=8.0),
        Workload("fp16_32k", "fp16", 1, 8, 8, 32768, 64, seed=4, backward=False),
        Workload("gqa_qwen3_nc", "bf16", 4, 32, 8, 2048, 128, seed=2, causal=False),
        Workload("long_8k_nc", "bf16", 1, 32, 32, 8192, 128, seed=3, causal=False,
                 value_scale=0.5, spike_every=512, spike_scale=8.0),
        Workload("prefill_8k", "bf16", 1, 32, 8, 2048, 128, seed=5, Skv=8192),
        Workload("decode_8k", "bf16", 16, 32, 8, 1, 128, seed=6, Skv=8192, backward=False,
                 decode=True),
        Workload("spec_32k", "bf16", 2, 32, 8, 4, 128, seed=7, Skv=32768, backward=False,
                 decode=True),
        Workload("decode_8k_paged", "bf16", 16, 32, 8, 1, 128, seed=6, Skv=8192,
                 backward=False, decode=True, page_size=64),
    ]
}


def make_inputs(w: Workload, with_dout: bool = True):
    """Draw (q, k, v[, dout]) on the CPU for workload `w`.

    Draw order is Q, K, V, dO from one generator seeded with `w.seed`; each
    tensor is drawn in fp32, multiplied by `value_scale`, K gets its spike
    rows, and the result is rounded (round-to-nearest-even) to the storage
    dtype.
    """
    g = torch.Generator().manual_seed(w.seed)
    qshape = (w.B, w.Hq, w.S, w.d)
    kshape = (w.B, w.Hkv, w.kv_len, w.d)

    def draw(shape):
        t = torch.randn(shape, generator=g, dtype=torch.float32)
        if w.value_scale != 1.0:
            t.mul_(w.value_scale)
        return t

    q = draw(qshape)
    k = draw(kshape)
    if w.spike_every:
        k[:, :, :: w.spike_every, :] *= w.spike_scale
    v = draw(kshape)
    out = [q, k, v]
    if with_dout:
        out.append(draw(qshape))
    return tuple(t.to(w.torch_dtype) for t in out)


def make_custom(B, Hq, Hkv, S, d, dtype="bf16", seed=0, value_scale=1.0,
                with_dout=True, Skv=0):
    """Same recipe as `make_inputs` for an ad-hoc shape (edge-case tests);
    S is the query length, Skv the key/value length (0: same as S)."""
    w = Workload("custom", dtype, B, Hq, Hkv, S, d, seed=seed,
                 value_scale=value_scale, Skv=Skv)
    return make_inputs(w, with_dout=with_dout)


def make_paged(k, v, block_size: int, seed: int, spare_blocks: int = 3):
    """Scatter contiguous k, v [B, Hkv, Skv, d] into a paged cache.

    Returns (k_cache, v_cache, block_table, num_blocks): caches
    [num_blocks, Hkv, block_size, d] with the sequences' blocks at seeded random
    physical positions (plus `spare_blocks` unused blocks filled with large
    values that must never be read), and an int32 block table [B, max_blocks]
    whose entries past each sequence's last block are -1. A layout change only:
    no attention arithmetic.
    """
    B, Hkv, Skv, d = k.shape
    per_seq = -(-Skv // block_size)
    num_blocks = B * per_seq + spare_blocks
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_blocks, generator=g)
    table = torch.full((B, per_seq + 2), -1, dtype=torch.int32)
    k_cache = torch.full((num_blocks, Hkv, block_size, d), 1000.0, dtype=k.dtype)
    v_cache = torch.full((num_blocks, Hkv, block_size, d), 1000.0, dtype=v.dtype)
    for b in range(B):
        for lb in range(per_seq):
            pb = int(perm[b * per_seq + lb])
            table[b, lb] = pb
            t0, t1 = lb * block_size, min((lb + 1) * block_size, Skv)
            k_cache[pb, :, : t1 - t0] = k[b, :, t0:t1]
            v_cache[pb, :, : t1 - t0] = v[b, :, t0:t1]
    return k_cache, v_cache, table, num_blocks


def sample_rows(S: int, n: int, seed: int, tile: int = 128):
    """Sorted distinct row indices for sampled checks at long S.

    Always contains 0, S-1 and the tile boundaries tile-1/tile and
    2*tile-1/2*tile (plus 511/512 when S is large enough), the rest drawn
    uniformly from a seeded generator.
    """
    must = {0, S - 1}
    for t in (tile, 2 * tile, 512):
        if t < S:
            must.update({t - 1, t})
    rows = set(must)
    g = torch.Generator().manual_seed(seed)
    for r in torch.randperm(S, generator=g).tolist():
        if len(rows) >= n:
            break
        rows.add(r)
    return sorted(rows)
