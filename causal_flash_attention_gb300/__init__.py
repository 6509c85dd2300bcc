"""Causal flash attention on one NVIDIA GB300 (sm_103a): thin Python binding of
libfa (include/fa.h).

The functions with the C names (`fa_fwd`, `fa_bwd`, `fa_bwd_workspace_bytes`,
`fa_fwd_kv`, `fa_bwd_kv`, `fa_bwd_kv_workspace_bytes`, `fa_fwd_splitkv`,
`fa_fwd_splitkv_workspace_bytes`, `fa_fwd_splitkv_paged`, `fa_strerror`,
`fa_last_device_status`, `fa_version`) only marshal arguments:
shapes come from the tensors, pointers from `data_ptr()`, and the stream from
PyTorch's current stream. Every step of the computation runs in libfa's CUDA
kernels; there is no other code path. `attention_forward` / `attention_backward`
additionally allocate their outputs (and the backward workspace) with
PyTorch.

The library is built in-tree by `causal_flash_attention_gb300.build.build()`;
loading it raises if it has not been built.
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os

import torch

__all__ = [
    "FAError", "lib", "fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_strerror",
    "fa_last_device_status", "fa_version", "attention_forward", "attention_backward",
    "DTYPE_CODES", "fa_bwd_noalloc", "NOALLOC_SCRATCH_BYTES", "fa_fwd_kv", "fa_bwd_kv",
    "fa_bwd_kv_workspace_bytes", "fa_fwd_splitkv", "fa_fwd_splitkv_workspace_bytes",
    "decode_forward", "fa_fwd_splitkv_paged", "decode_forward_paged",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")
DTYPE_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
_lib = None


class FAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {fa_strerror(code)} (code {code})")


def lib() -> ctypes.CDLL:
    """Load libfa.so (once) and declare its C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with causal_flash_attention_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp]
    L.fa_fwd.restype = i32
    L.fa_bwd_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.fa_bwd_workspace_bytes.restype = sz
    L.fa_bwd.argtypes = [vp] * 9 + [i32, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp]
    L.fa_bwd.restype = i32
    L.fa_fwd_kv.argtypes = [vp, vp, vp, vp, vp] + [i32] * 7 + [f32, i32, vp]
    L.fa_fwd_kv.restype = i32
    L.fa_bwd_kv_workspace_bytes.argtypes = [i32] * 6
    L.fa_bwd_kv_workspace_bytes.restype = sz
    L.fa_bwd_kv.argtypes = [vp] * 9 + [i32] * 7 + [f32, i32, vp, sz, vp]
    L.fa_bwd_kv.restype = i32
    L.fa_fwd_splitkv.argtypes = [vp] * 5 + [i32] * 7 + [f32, i32, i32, vp, sz, vp]
    L.fa_fwd_splitkv.restype = i32
    L.fa_fwd_splitkv_workspace_bytes.argtypes = [i32] * 7
    L.fa_fwd_splitkv_workspace_bytes.restype = sz
    L.fa_fwd_splitkv_paged.argtypes = [vp] * 6 + [i32] * 10 + [f32, i32, i32, vp, sz, vp]
    L.fa_fwd_splitkv_paged.restype = i32
    L.fa_strerror.argtypes = [i32]
    L.fa_strerror.restype = ctypes.c_char_p
    L.fa_last_device_status.argtypes = [vp, ctypes.POINTER(i32)]
    L.fa_last_device_status.restype = i32
    L.fa_version.argtypes = []
    L.fa_version.restype = i32
    _lib = L
    return L


def fa_strerror(code: int) -> str:
    return lib().fa_strerror(int(code)).decode()


def fa_version() -> int:
    return int(lib().fa_version())


def _ptr(t):
    return None if t is None else t.data_ptr()


# the current stream's raw handle straight from PyTorch's C layer, where the
# build has it (a cheap call; torch.cuda.current_stream() builds a Stream object)
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_NULL_CONTEXT = contextlib.nullcontext()


def _stream(stream, t=None):
    """The CUDA stream handle for a call: `stream` itself, or PyTorch's current
    stream on t's device (the current device when t is None)."""
    if stream is None:
        if _raw_stream is not None and t is not None and t.is_cuda:
            return _raw_stream(t.get_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dims(q, k):
    """(B, Hq, Hkv, S, d) of a self-attention call (q and k of one length)."""
    B, Hq, Hkv, Sq, Skv, d = _dims_kv(q, k)
    if Sq != Skv:
        raise ValueError(f"q has {Sq} rows and k {Skv}: use the *_kv functions")
    return B, Hq, Hkv, Sq, d


def _dims_kv(q, k):
    """(B, Hq, Hkv, Sq, Skv, d) from q [B,Hq,Sq,d] and k [B,Hkv,Skv,d]."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be [B, H, S, d]")
    B, Hq, Sq, d = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    return int(B), int(Hq), int(Hkv), int(Sq), int(Skv), int(d)


def _on_device(t):
    """Make t's GPU the current device for the call (the library runs on the
    current device); nothing to switch when it already is."""
    if t is not None and t.is_cuda and t.get_device() != torch.cuda.current_device():
        return torch.cuda.device(t.device)
    return _NULL_CONTEXT


def _check_contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def fa_fwd(q, k, v, out, lse, causal=True, scale=None, stream=None):
    """Call fa_fwd on caller-provided tensors (out: like q; lse: float32 [B,Hq,S])."""
    _check_contig(q, k, v, out, lse)
    B, Hq, Hkv, S, d = _dims(q, k)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with _on_device(q):
        rc = lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S, d,
                          int(bool(causal)), scale, DTYPE_CODES.get(q.dtype, -1), _stream(stream, q))
    if rc != 0:
        raise FAError(rc, "fa_fwd")


def fa_bwd_workspace_bytes(B, Hq, Hkv, S, d) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, Hq, Hkv, S, d))


def fa_bwd(q, k, v, out, dout, lse, dq, dk, dv, workspace, causal=True, scale=None,
           stream=None):
    """Call fa_bwd on caller-provided tensors; `workspace` is a device tensor of at
    least fa_bwd_workspace_bytes(...) bytes."""
    _check_contig(q, k, v, out, dout, lse, dq, dk, dv)
    B, Hq, Hkv, S, d = _dims(q, k)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on_device(q):
        rc = lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq),
                          _ptr(dk), _ptr(dv), B, Hq, Hkv, S, d, int(bool(causal)), scale,
                          DTYPE_CODES.get(q.dtype, -1), _ptr(workspace), ws_bytes, _stream(stream, q))
    if rc != 0:
        raise FAError(rc, "fa_bwd")


def fa_fwd_kv(q, k, v, out, lse, causal=True, scale=None, stream=None):
    """Call fa_fwd_kv: q/out [B,Hq,Sq,d], k/v [B,Hkv,Skv,d], lse float32 [B,Hq,Sq];
    the causal mask is aligned to the last key (kv_offset = Skv - Sq)."""
    _check_contig(q, k, v, out, lse)
    B, Hq, Hkv, Sq, Skv, d = _dims_kv(q, k)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with _on_device(q):
        rc = lib().fa_fwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Skv,
                             d, int(bool(causal)), scale, DTYPE_CODES.get(q.dtype, -1),
                             _stream(stream, q))
    if rc != 0:
        raise FAError(rc, "fa_fwd_kv")


def fa_bwd_kv_workspace_bytes(B, Hq, Hkv, Sq, Skv, d) -> int:
    return int(lib().fa_bwd_kv_workspace_bytes(B, Hq, Hkv, Sq, Skv, d))


def fa_bwd_kv(q, k, v, out, dout, lse, dq, dk, dv, workspace, causal=True, scale=None,
              stream=None):
    """Call fa_bwd_kv (separate query and key/value lengths, as fa_fwd_kv)."""
    _check_contig(q, k, v, out, dout, lse, dq, dk, dv)
    B, Hq, Hkv, Sq, Skv, d = _dims_kv(q, k)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on_device(q):
        rc = lib().fa_bwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq),
                             _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Skv, d, int(bool(causal)), scale,
                             DTYPE_CODES.get(q.dtype, -1), _ptr(workspace), ws_bytes,
                             _stream(stream, q))
    if rc != 0:
        raise FAError(rc, "fa_bwd_kv")


def fa_fwd_splitkv_workspace_bytes(B, Hq, Hkv, Sq, Skv, d, n_splits=0) -> int:
    return int(lib().fa_fwd_splitkv_workspace_bytes(B, Hq, Hkv, Sq, Skv, d, n_splits))


def fa_fwd_splitkv(q, k, v, out, lse, causal=True, scale=None, n_splits=0, workspace=None,
                   stream=None):
    """Call fa_fwd_splitkv (few query rows against a long key/value sequence);
    `workspace` is a device tensor of at least fa_fwd_splitkv_workspace_bytes(...)
    bytes, or None when that size is 0."""
    _check_contig(q, k, v, out, lse)
    B, Hq, Hkv, Sq, Skv, d = _dims_kv(q, k)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on_device(q):
        rc = lib().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq,
                                  Skv, d, int(bool(causal)), scale, DTYPE_CODES.get(q.dtype, -1),
                                  int(n_splits), _ptr(workspace), ws_bytes, _stream(stream, q))
    if rc != 0:
        raise FAError(rc, "fa_fwd_splitkv")


def decode_forward(q, k, v, causal=True, scale=None, n_splits=0, stream=None):
    """Allocate out, lse and the split workspace with PyTorch and run
    fa_fwd_splitkv. Returns (out, lse)."""
    B, Hq, Hkv, Sq, Skv, d = _dims_kv(q, k)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    n = fa_fwd_splitkv_workspace_bytes(B, Hq, Hkv, Sq, Skv, d, n_splits)
    ws = torch.empty(n, dtype=torch.uint8, device=q.device) if n else None
    fa_fwd_splitkv(q, k, v, out, lse, causal, scale, n_splits, ws, stream)
    return out, lse


def fa_fwd_splitkv_paged(q, k_cache, v_cache, block_table, out, lse, Skv, causal=True,
                         scale=None, n_splits=0, workspace=None, stream=None):
    """Call fa_fwd_splitkv_paged: q [B,Hq,Sq,d]; k_cache/v_cache
    [num_blocks,Hkv,block_size,d]; block_table int32 [B,max_blocks]; every
    sequence holds Skv keys."""
    _check_contig(q, k_cache, v_cache, block_table, out, lse)
    if q.dim() != 4 or k_cache.dim() != 4 or block_table.dim() != 2:
        raise ValueError("q [B,Hq,Sq,d], caches [num_blocks,Hkv,block_size,d], table [B,max_blocks]")
    if block_table.dtype != torch.int32:
        raise ValueError("block_table must be int32")
    B, Hq, Sq, d = (int(x) for x in q.shape)
    num_blocks, Hkv, block_size = (int(x) for x in k_cache.shape[:3])
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _on_device(q):
        rc = lib().fa_fwd_splitkv_paged(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(out), _ptr(lse), B, Hq,
            Hkv, Sq, int(Skv), d, block_size, num_blocks, int(block_table.shape[1]),
            int(bool(causal)), scale, DTYPE_CODES.get(q.dtype, -1), int(n_splits), _ptr(workspace),
            ws_bytes, _stream(stream, q))
    if rc != 0:
        raise FAError(rc, "fa_fwd_splitkv_paged")


def decode_forward_paged(q, k_cache, v_cache, block_table, Skv, causal=True, scale=None,
                         n_splits=0, stream=None):
    """Allocate out, lse and the split workspace and run fa_fwd_splitkv_paged."""
    B, Hq, Sq, d = (int(x) for x in q.shape)
    Hkv = int(k_cache.shape[1])
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    n = fa_fwd_splitkv_workspace_bytes(B, Hq, Hkv, Sq, int(Skv), d, n_splits)
    ws = torch.empty(n, dtype=torch.uint8, device=q.device) if n else None
    fa_fwd_splitkv_paged(q, k_cache, v_cache, block_table, out, lse, Skv, causal, scale, n_splits,
                         ws, stream)
    return out, lse


def fa_last_device_status(stream=None) -> int:
    st = ctypes.c_int(0)
    rc = lib().fa_last_device_status(_stream(stream), ctypes.byref(st))
    if rc != 0:
        raise FAError(rc, "fa_last_device_status")
    return st.value


def attention_forward(q, k, v, causal=True, scale=None, stream=None):
    """Allocate out and lse with PyTorch and run fa_fwd (fa_fwd_kv when q and k
    have different lengths). Returns (out, lse)."""
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    if q.shape[2] == k.shape[2]:
        fa_fwd(q, k, v, out, lse, causal, scale, stream)
    else:
        fa_fwd_kv(q, k, v, out, lse, causal, scale, stream)
    return out, lse


def workspace_for(q, k):
    B, Hq, Hkv, Sq, Skv, d = _dims_kv(q, k)
    n = fa_bwd_kv_workspace_bytes(B, Hq, Hkv, Sq, Skv, d)
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def attention_backward(q, k, v, out, dout, lse, causal=True, scale=None, workspace=None,
                       stream=None):
    """Allocate dq, dk, dv (and a workspace unless given) and run fa_bwd
    (fa_bwd_kv when q and k have different lengths)."""
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = workspace_for(q, k)
    if q.shape[2] == k.shape[2]:
        fa_bwd(q, k, v, out, dout, lse, dq, dk, dv, workspace, causal, scale, stream)
    else:
        fa_bwd_kv(q, k, v, out, dout, lse, dq, dk, dv, workspace, causal, scale, stream)
    return dq, dk, dv


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024   # FA_NOALLOC_SCRATCH_BYTES in include/fa.h


def fa_bwd_noalloc(q, k, v, out, dout, lse, dq, dk, dv, causal=True, scale=None, stream=None):
    """Call fa_bwd_noalloc: fa_bwd without a workspace, for callers that cannot
    allocate device memory; the scratch is a fixed array inside libfa (see
    include/fa.h for its size, sharing and ordering rules)."""
    L = lib()
    fn = L.fa_bwd_noalloc
    if fn.argtypes is None:
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        fn.argtypes = [vp] * 9 + [i32, i32, i32, i32, i32, i32, ctypes.c_float, i32, vp]
        fn.restype = i32
    _check_contig(q, k, v, out, dout, lse, dq, dk, dv)
    B, Hq, Hkv, S, d = _dims(q, k)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with _on_device(q):   # the scratch array used is the current device's
        rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                _ptr(dv), B, Hq, Hkv, S, d, int(bool(causal)), scale,
                DTYPE_CODES.get(q.dtype, -1), _stream(stream, q))
    if rc != 0:
        raise FAError(rc, "fa_bwd_noalloc")
