"""The C ABI without a GPU: the library loads, exports every function that
include/fa.h declares, and rejects bad arguments on the host with the
documented codes before touching the device."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")

FA_OK, FA_ERR_SHAPE, FA_ERR_DTYPE, FA_ERR_NULL, FA_ERR_ALIGN, FA_ERR_WORKSPACE, \
    FA_ERR_CUDA, FA_ERR_SCALE, FA_ERR_TMA = 0, -1, -2, -3, -4, -5, -6, -7, -8


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_strerror",
              "fa_last_device_status", "fa_version"):
        assert n in names


def test_library_exports_every_declared_symbol(fa_lib):
    L = fa_lib.lib()
    for n in declared_functions():
        assert hasattr(L, n), f"libfa.so does not export {n}"


def test_error_codes_match_header():
    text = open(HEADER).read()
    for name, val in [("FA_OK", 0), ("FA_ERR_SHAPE", -1), ("FA_ERR_DTYPE", -2),
                      ("FA_ERR_NULL", -3), ("FA_ERR_ALIGN", -4), ("FA_ERR_WORKSPACE", -5),
                      ("FA_ERR_CUDA", -6), ("FA_ERR_SCALE", -7), ("FA_ERR_TMA", -8)]:
        assert re.search(rf"\b{name}\s*=\s*{val}\b", text), name


def test_strerror_and_version(fa_lib):
    for code in range(0, -9, -1):
        s = fa_lib.fa_strerror(code)
        assert s and s != "unknown error code"
    assert fa_lib.fa_strerror(-99) == "unknown error code"
    assert fa_lib.fa_version() >= 10000


def _fwd(L, q=16, k=16, v=16, out=16, lse=16, B=1, Hq=2, Hkv=1, S=128, d=64, causal=1,
         scale=0.125, dtype=2):
    return L.fa_fwd(q, k, v, out, lse, B, Hq, Hkv, S, d, causal, scale, dtype, None)


def _bwd(L, ptr=256, B=1, Hq=2, Hkv=1, S=128, d=64, scale=0.125, dtype=2, ws=256,
         ws_bytes=1 << 30, **over):
    ptrs = dict(q=ptr, k=ptr, v=ptr, out=ptr, dout=ptr, lse=ptr, dq=ptr, dk=ptr, dv=ptr)
    ptrs.update(over)
    return L.fa_bwd(ptrs["q"], ptrs["k"], ptrs["v"], ptrs["out"], ptrs["dout"], ptrs["lse"],
                    ptrs["dq"], ptrs["dk"], ptrs["dv"], B, Hq, Hkv, S, d, 1, scale, dtype,
                    ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=32), FA_ERR_SHAPE), (dict(d=96), FA_ERR_SHAPE), (dict(d=256), FA_ERR_SHAPE),
    (dict(S=0), FA_ERR_SHAPE), (dict(B=0), FA_ERR_SHAPE), (dict(Hq=3, Hkv=2), FA_ERR_SHAPE),
    (dict(Hkv=0), FA_ERR_SHAPE), (dict(dtype=3), FA_ERR_DTYPE), (dict(dtype=-1), FA_ERR_DTYPE),
    (dict(scale=0.0), FA_ERR_SCALE), (dict(scale=-1.0), FA_ERR_SCALE),
    (dict(scale=float("nan")), FA_ERR_SCALE), (dict(scale=float("inf")), FA_ERR_SCALE),
    (dict(q=None), FA_ERR_NULL), (dict(lse=None), FA_ERR_NULL), (dict(out=None), FA_ERR_NULL),
    (dict(q=8), FA_ERR_ALIGN), (dict(v=24), FA_ERR_ALIGN), (dict(lse=4), FA_ERR_ALIGN),
])
def test_fwd_rejects_bad_arguments(fa_lib, kw, code):
    assert _fwd(fa_lib.lib(), **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(d=48), FA_ERR_SHAPE), (dict(Hq=5, Hkv=2), FA_ERR_SHAPE), (dict(dtype=7), FA_ERR_DTYPE),
    (dict(dq=None), FA_ERR_NULL), (dict(dout=None), FA_ERR_NULL), (dict(dv=8), FA_ERR_ALIGN),
    (dict(ws=None), FA_ERR_WORKSPACE), (dict(ws_bytes=1024), FA_ERR_WORKSPACE),
    (dict(ws=16 + 256), FA_ERR_ALIGN), (dict(scale=0.0), FA_ERR_SCALE),
])
def test_bwd_rejects_bad_arguments(fa_lib, kw, code):
    assert _bwd(fa_lib.lib(), **kw) == code


def test_workspace_size_formula(fa_lib):
    def expect(B, Hq, S, d):
        up = lambda x, m: (x + m - 1) // m * m
        bh, sp = B * Hq, up(S, 128)
        return up(bh * sp * d * 4, 256) + 2 * up(bh * sp * 4, 256) + 256
    for B, Hq, Hkv, S, d in [(1, 2, 2, 128, 64), (8, 12, 12, 1024, 64), (4, 32, 8, 2048, 128),
                             (1, 32, 32, 8192, 128), (1, 1, 1, 1, 64), (3, 4, 2, 200, 128)]:
        assert fa_lib.fa_bwd_workspace_bytes(B, Hq, Hkv, S, d) == expect(B, Hq, S, d)
    assert fa_lib.fa_bwd_workspace_bytes(1, 3, 2, 128, 64) == 0
    assert fa_lib.fa_bwd_workspace_bytes(1, 1, 1, 128, 80) == 0


def test_status_requires_output_pointer(fa_lib):
    assert fa_lib.lib().fa_last_device_status(None, None) == FA_ERR_NULL


def test_package_fails_loudly_without_library(monkeypatch, tmp_path):
    import causal_flash_attention_gb300 as fa
    monkeypatch.setattr(fa, "_lib", None)
    monkeypatch.setattr(fa, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        fa.lib()


# separate query / key-value lengths (fa_fwd_kv, fa_bwd_kv)
def _fwd_kv(L, q=16, k=16, v=16, out=16, lse=16, B=1, Hq=2, Hkv=1, Sq=128, Skv=300, d=64,
            causal=1, scale=0.125, dtype=2):
    return L.fa_fwd_kv(q, k, v, out, lse, B, Hq, Hkv, Sq, Skv, d, causal, scale, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Sq=301, Skv=300), FA_ERR_SHAPE),              # causal: fewer keys than queries
    (dict(Sq=301, Skv=300, causal=0, q=None), FA_ERR_NULL),   # unmasked: any lengths
    (dict(Sq=0), FA_ERR_SHAPE), (dict(Skv=0), FA_ERR_SHAPE), (dict(Skv=-5), FA_ERR_SHAPE),
    (dict(d=80), FA_ERR_SHAPE), (dict(dtype=5), FA_ERR_DTYPE), (dict(scale=0.0), FA_ERR_SCALE),
    (dict(v=None), FA_ERR_NULL), (dict(k=8), FA_ERR_ALIGN), (dict(out=40), FA_ERR_ALIGN),
    (dict(Sq=1, Skv=(1 << 31) - 1), FA_ERR_SHAPE),
])
def test_fwd_kv_rejects_bad_arguments(fa_lib, kw, code):
    assert _fwd_kv(fa_lib.lib(), **kw) == code


def _bwd_kv(L, ptr=256, B=1, Hq=2, Hkv=1, Sq=128, Skv=300, d=64, causal=1, scale=0.125,
            dtype=2, ws=256, ws_bytes=1 << 30, **over):
    ptrs = dict(q=ptr, k=ptr, v=ptr, out=ptr, dout=ptr, lse=ptr, dq=ptr, dk=ptr, dv=ptr)
    ptrs.update(over)
    return L.fa_bwd_kv(ptrs["q"], ptrs["k"], ptrs["v"], ptrs["out"], ptrs["dout"], ptrs["lse"],
                       ptrs["dq"], ptrs["dk"], ptrs["dv"], B, Hq, Hkv, Sq, Skv, d, causal, scale,
                       dtype, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Sq=400, Skv=300), FA_ERR_SHAPE), (dict(Sq=400, Skv=300, causal=0, dk=None), FA_ERR_NULL),
    (dict(Skv=0), FA_ERR_SHAPE), (dict(dk=None), FA_ERR_NULL), (dict(dv=24), FA_ERR_ALIGN),
    (dict(ws=None), FA_ERR_WORKSPACE), (dict(ws_bytes=1024), FA_ERR_WORKSPACE),
    (dict(ws=16 + 256), FA_ERR_ALIGN),
])
def test_bwd_kv_rejects_bad_arguments(fa_lib, kw, code):
    assert _bwd_kv(fa_lib.lib(), **kw) == code


def test_backward_item_count_bound(fa_lib):
    """The backward's work items (batch x key/value heads x 128-key tiles) are
    claimed from a 32-bit counter that runs past the last item by one claim
    per CTA: sizes within 2^16 of 2^31 are rejected, smaller ones accepted."""
    H = 1 << 24
    assert fa_lib.fa_bwd_kv_workspace_bytes(1, H, H, 1, 128 * 128, 64) == 0       # 2^31 items
    assert fa_lib.fa_bwd_kv_workspace_bytes(1, H, H, 1, 128 * 127 + 1, 64) == 0   # 2^31 items
    assert fa_lib.fa_bwd_kv_workspace_bytes(1, H, H, 1, 128 * 127, 64) > 0        # 2^31 - 2^24


def test_kv_workspace_is_sized_by_the_query_length(fa_lib):
    up = lambda x, m: (x + m - 1) // m * m
    for B, Hq, Hkv, Sq, Skv, d in [(1, 32, 8, 2048, 8192, 128), (2, 4, 2, 1, 777, 64),
                                   (1, 2, 2, 300, 129, 128)]:
        bh, sp = B * Hq, up(Sq, 128)
        want = up(bh * sp * d * 4, 256) + 2 * up(bh * sp * 4, 256) + 256
        assert fa_lib.fa_bwd_kv_workspace_bytes(B, Hq, Hkv, Sq, Skv, d) == want
    assert fa_lib.fa_bwd_kv_workspace_bytes(1, 2, 2, 128, 0, 64) == 0
    assert fa_lib.fa_bwd_kv_workspace_bytes(1, 2, 2, 128, 128, 64) == \
        fa_lib.fa_bwd_workspace_bytes(1, 2, 2, 128, 64)


# split-KV forward (fa_fwd_splitkv)
def _splitkv(L, q=16, k=16, v=16, out=16, lse=16, B=1, Hq=8, Hkv=2, Sq=1, Skv=4096, d=128,
             causal=1, scale=0.125, dtype=2, n_splits=0, ws=256, ws_bytes=1 << 30):
    return L.fa_fwd_splitkv(q, k, v, out, lse, B, Hq, Hkv, Sq, Skv, d, causal, scale, dtype,
                            n_splits, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Sq=33, Hq=16, Hkv=4), FA_ERR_SHAPE),           # G * Sq = 132 > 128 rows
    (dict(Sq=32, Hq=16, Hkv=4, q=None), FA_ERR_NULL),     # G * Sq = 128 fits
    (dict(n_splits=-1), FA_ERR_SHAPE), (dict(Sq=5000), FA_ERR_SHAPE),
    (dict(Skv=0), FA_ERR_SHAPE), (dict(d=96), FA_ERR_SHAPE), (dict(dtype=4), FA_ERR_DTYPE),
    (dict(scale=-2.0), FA_ERR_SCALE), (dict(lse=None), FA_ERR_NULL), (dict(v=40), FA_ERR_ALIGN),
])
def test_splitkv_rejects_bad_arguments(fa_lib, kw, code):
    assert _splitkv(fa_lib.lib(), **kw) == code


def test_splitkv_workspace_plan(fa_lib):
    up = lambda x, m: (x + m - 1) // m * m
    ws = fa_lib.fa_fwd_splitkv_workspace_bytes

    def expect(B, Hq, Hkv, Sq, Skv, d, n_req):
        tiles = (Skv + 127) // 128
        want = n_req if n_req > 0 else 152 // (B * Hkv)
        want = max(1, min(want, tiles))
        per = -(-tiles // want)
        n = -(-tiles // per)
        if n == 1:
            return 0
        rows = B * Hkv * n * (Hq // Hkv) * Sq
        return up(rows * d * 4, 256) + up(rows * 4, 256)

    for args in [(16, 32, 8, 1, 8192, 128, 0), (1, 8, 2, 4, 4096, 64, 0), (2, 4, 4, 1, 100, 128, 0),
                 (1, 8, 1, 16, 65536, 128, 7), (1, 2, 2, 1, 300, 64, 1), (64, 32, 8, 1, 1024, 128, 0)]:
        assert ws(*args) == expect(*args), args
    assert ws(1, 8, 2, 1, 4096, 128, 0) > 0
    assert ws(1, 2, 2, 1, 128, 128, 0) == 0          # one key tile: one range, no workspace
    assert ws(1, 16, 4, 33, 4096, 128, 0) == 0       # invalid: G * Sq > 128


def _paged(L, q=16, kc=16, vc=16, table=16, out=16, lse=16, B=2, Hq=8, Hkv=2, Sq=1, Skv=1000,
           d=128, block_size=64, num_blocks=40, max_blocks=16, causal=1, scale=0.125, dtype=2,
           n_splits=0, ws=256, ws_bytes=1 << 30):
    return L.fa_fwd_splitkv_paged(q, kc, vc, table, out, lse, B, Hq, Hkv, Sq, Skv, d, block_size,
                                  num_blocks, max_blocks, causal, scale, dtype, n_splits, ws,
                                  ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(block_size=8), FA_ERR_SHAPE), (dict(block_size=48), FA_ERR_SHAPE),
    (dict(block_size=2048), FA_ERR_SHAPE), (dict(num_blocks=0), FA_ERR_SHAPE),
    (dict(max_blocks=15), FA_ERR_SHAPE),             # ceil(1000 / 64) = 16 entries needed
    (dict(max_blocks=16, table=None), FA_ERR_NULL), (dict(table=18), FA_ERR_ALIGN),
    (dict(kc=None), FA_ERR_NULL), (dict(vc=8), FA_ERR_ALIGN), (dict(dtype=0), FA_ERR_DTYPE),
    (dict(Sq=33, Hq=16, Hkv=4), FA_ERR_SHAPE), (dict(Sq=2000), FA_ERR_SHAPE),
    (dict(block_size=1024, max_blocks=1, q=None), FA_ERR_NULL),
])
def test_paged_rejects_bad_arguments(fa_lib, kw, code):
    assert _paged(fa_lib.lib(), **kw) == code
