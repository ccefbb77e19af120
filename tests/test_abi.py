"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function ``include/fa.h`` declares, and
reject bad arguments synchronously, before it touches the device.
"""

import ctypes
import json
import os
import re

import pytest

from attention_sm_flashattention_gb300 import _native
from oracle import attention as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_native.LIB_PATH):
        from attention_sm_flashattention_gb300 import build
        build.build()
    return _native.lib()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    syms = set(declared_symbols())
    for name in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_device_status", "fa_error_string"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    syms = declared_symbols()
    assert syms
    for name in syms:
        assert hasattr(lib, name), name
        assert name in _native.SIGNATURES, f"binding lacks a signature for {name}"


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert len(_native.error_string(code)) >= 2
    assert "unknown" in _native.error_string(12345)


FAKE = 1 << 20  # an aligned non-null address that is never dereferenced


def call_fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, Z=1, H=1, N=128, D=64, causal=0, scale=0.125):
    return lib.fa_fwd(q, k, v, o, lse, Z, H, N, D, causal, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), _native.FA_ERR_INVALID_ARG),
    (dict(lse=None), _native.FA_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), _native.FA_ERR_INVALID_ARG),      # not 16-byte aligned
    (dict(Z=0), _native.FA_ERR_INVALID_ARG),
    (dict(H=-1), _native.FA_ERR_INVALID_ARG),
    (dict(N=0), _native.FA_ERR_INVALID_ARG),
    (dict(causal=2), _native.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), _native.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), _native.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), _native.FA_ERR_INVALID_ARG),
    (dict(D=96), _native.FA_ERR_UNSUPPORTED),
    (dict(D=32), _native.FA_ERR_UNSUPPORTED),
    (dict(Z=1 << 14, H=1 << 10, N=256), _native.FA_ERR_UNSUPPORTED),  # rows >= 2^31
])
def test_fwd_rejects_bad_arguments(lib, kw, code):
    assert call_fwd(lib, **kw) == code


def call_bwd(lib, ws=FAKE, ws_bytes=1 << 40, dq=FAKE, D=64, N=128, scale=0.125):
    return lib.fa_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dq, FAKE, FAKE, ws, ws_bytes,
                      1, 1, N, D, 0, scale, None)


def test_bwd_rejects_bad_arguments(lib):
    assert call_bwd(lib, dq=None) == _native.FA_ERR_INVALID_ARG
    assert call_bwd(lib, D=80) == _native.FA_ERR_UNSUPPORTED
    assert call_bwd(lib, scale=-1.0) == _native.FA_ERR_INVALID_ARG


def test_workspace_size_rejects_bad_shapes(lib):
    assert lib.fa_bwd_ex_workspace_size(1, 4, 3, 128, 128, 64, 0) == 0    # H not a multiple of Hkv
    assert lib.fa_bwd_ex_workspace_size(1, 4, 2, 256, 128, 64, 1) == 0    # causal with Nq > Nk
    assert lib.fa_bwd_workspace_size(1, 1, 128, 48, 0) == 0


def test_workspace_is_two_padded_row_vectors(lib):
    # Delta and lse2 over Z*H query rows padded to whole 128-row tiles, each
    # rounded up to 256 bytes; nothing grows with N^2 or with D.
    def want(Z, H, Nq):
        vec = Z * H * ((Nq + 127) // 128 * 128) * 4
        return 2 * ((vec + 255) // 256 * 256)
    for Z, H, Hkv, Nq, Nk, D in ((1, 1, 1, 100, 100, 256), (2, 8, 2, 1000, 3000, 128), (3, 4, 4, 1, 1, 64),
                                 (128, 8, 8, 1024, 1024, 256)):
        assert lib.fa_bwd_ex_workspace_size(Z, H, Hkv, Nq, Nk, D, 0) == want(Z, H, Nq)
    assert lib.fa_bwd_workspace_size(128, 8, 1024, 128, 1) == want(128, 8, 1024)


def test_tile_count_matches_pages_and_oracle(lib):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "causal_tiles.json")))
    n = g["n_tiles"] * 128
    assert lib.fa_fwd_tile_count(n, 128, 0) == g["non_causal_tiles"]
    assert lib.fa_fwd_tile_count(n, 128, 1) == g["causal_tiles"]
    for N in (128, 256, 1024, 2048):
        t = N // 128
        assert lib.fa_fwd_tile_count(N, 64, 1) == orc.causal_tile_count(t, True)
        assert lib.fa_fwd_tile_count(N, 128, 0) == orc.causal_tile_count(t, False)
        # the dense forward tiles D = 256 by 128 keys too (each tile moves as two halves)
        assert lib.fa_fwd_tile_count(N, 256, 0) == orc.causal_tile_count(t, False)
        assert lib.fa_fwd_tile_count(N, 256, 1) == orc.causal_tile_count(t, True)
    # ragged N: count the (query tile, key tile) pairs that hold at least one
    # visible (query, key) pair, by brute force over the tile grid
    for N, D in ((100, 64), (300, 128), (130, 256), (1, 64)):
        bn = 128
        for causal in (0, 1):
            want = 0
            for qt in range((N + 127) // 128):
                for kt in range((N + bn - 1) // bn):
                    q_last = min(N, (qt + 1) * 128) - 1
                    if kt * bn < N and (not causal or kt * bn <= q_last):
                        want += 1
            assert lib.fa_fwd_tile_count(N, D, causal) == want, (N, D, causal)
    assert lib.fa_fwd_tile_count(0, 64, 0) == -1


def call_fwd_ex(lib, Z=1, H=4, Hkv=2, Nq=100, Nk=200, D=64, causal=0, scale=0.125, dtype=0):
    return lib.fa_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, Z, H, Hkv, Nq, Nk, D, causal, scale, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Hkv=3), _native.FA_ERR_INVALID_ARG),       # 4 query heads over 3 K/V heads
    (dict(Hkv=0), _native.FA_ERR_INVALID_ARG),
    (dict(Nk=0), _native.FA_ERR_INVALID_ARG),
    (dict(dtype=2), _native.FA_ERR_INVALID_ARG),
    (dict(causal=1, Nq=201), _native.FA_ERR_UNSUPPORTED),  # a query row would see no key
    (dict(D=80), _native.FA_ERR_UNSUPPORTED),
])
def test_fwd_ex_rejects_bad_arguments(lib, kw, code):
    assert call_fwd_ex(lib, **kw) == code


def test_flop_model_general_shapes(lib):
    # 4 D FLOPs per visible (query, key) pair per query head: count the pairs
    for Nq, Nk in ((1, 1), (3, 7), (100, 300), (128, 128)):
        for causal in (0, 1):
            pairs = sum(1 for i in range(Nq) for j in range(Nk) if not causal or j <= i + Nk - Nq)
            assert lib.fa_fwd_ex_flops(2, 3, Nq, Nk, 64, causal) == pytest.approx(6 * 4 * 64 * pairs)
            assert lib.fa_bwd_ex_flops(2, 3, Nq, Nk, 64, causal) == pytest.approx(2.5 * 6 * 4 * 64 * pairs)


def test_flop_model(lib):
    assert lib.fa_fwd_flops(128, 8, 1024, 128, 0) == pytest.approx(4 * 1024 * 1024 * 128 * 1024)
    assert lib.fa_fwd_flops(1, 1, 1024, 128, 1) == pytest.approx(2 * 1024 * 1025 * 128)
    assert lib.fa_bwd_flops(2, 3, 256, 64, 1) == pytest.approx(2.5 * lib.fa_fwd_flops(2, 3, 256, 64, 1))


def call_fwd_paged(lib, B=2, H=4, Hkv=2, Nq=1, D=128, num_pages=8, page_size=64, max_pages=4, causal=0,
                   scale=0.125, dtype=0, table=FAKE):
    return lib.fa_fwd_paged(FAKE, FAKE, FAKE, table, FAKE, FAKE, FAKE, B, H, Hkv, Nq, D, num_pages, page_size,
                            max_pages, causal, scale, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(table=None), _native.FA_ERR_INVALID_ARG),
    (dict(table=FAKE + 2), _native.FA_ERR_INVALID_ARG),   # int32 table not 4-byte aligned
    (dict(Hkv=3), _native.FA_ERR_INVALID_ARG),
    (dict(num_pages=0), _native.FA_ERR_INVALID_ARG),
    (dict(max_pages=0), _native.FA_ERR_INVALID_ARG),
    (dict(dtype=5), _native.FA_ERR_INVALID_ARG),
    (dict(page_size=48), _native.FA_ERR_UNSUPPORTED),     # not a power-of-two page of 16-128 rows
    (dict(page_size=8), _native.FA_ERR_UNSUPPORTED),
    (dict(D=256, page_size=128), _native.FA_ERR_UNSUPPORTED),  # D = 256 key tiles hold 64 keys
    (dict(D=96), _native.FA_ERR_UNSUPPORTED),
])
def test_fwd_paged_rejects_bad_arguments(lib, kw, code):
    assert call_fwd_paged(lib, **kw) == code


def test_reshape_and_cache_argument_checks(lib):
    f = lib.fa_reshape_and_cache
    assert f(None, None, None, None, None, 0, 2, 64, 4, 16, None) == _native.FA_OK   # nothing to write
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 3, 2, 96, 4, 16, None) == _native.FA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, None, FAKE, FAKE, 3, 2, 64, 4, 16, None) == _native.FA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE + 4, FAKE, FAKE, 3, 2, 64, 4, 16, None) == _native.FA_ERR_INVALID_ARG  # int64 slots
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 2, 64, 4, 16, None) == _native.FA_ERR_INVALID_ARG


def test_fwd_sparse_argument_checks(lib):
    def call(pages=FAKE, blocks=FAKE, count=FAKE, page_size=64, D=128, max_sel=4):
        return lib.fa_fwd_sparse(FAKE, FAKE, FAKE, pages, blocks, count, FAKE, FAKE, FAKE, 2, 4, 2, 1, D, 8,
                                 page_size, max_sel, 0, 0.125, 0, None)
    assert call(blocks=None) == _native.FA_ERR_INVALID_ARG
    assert call(count=FAKE + 2) == _native.FA_ERR_INVALID_ARG
    assert call(max_sel=0) == _native.FA_ERR_INVALID_ARG
    assert call(page_size=24) == _native.FA_ERR_UNSUPPORTED
    assert call(D=256, page_size=128) == _native.FA_ERR_UNSUPPORTED


def call_fwd_paged_split(lib, ws=FAKE, ws_bytes=1 << 30, splits=4, page_size=64, D=128, B=2, H=4, Nq=1):
    return lib.fa_fwd_paged_split(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, ws_bytes, B, H, 2, Nq, D, 8,
                                  page_size, 4, splits, 0, 0.125, 0, None)


@pytest.mark.parametrize("kw,code", [
    (dict(splits=0), _native.FA_ERR_INVALID_ARG),
    (dict(splits=257), _native.FA_ERR_INVALID_ARG),
    (dict(ws=None), _native.FA_ERR_WORKSPACE),
    (dict(ws=FAKE + 8), _native.FA_ERR_WORKSPACE),          # workspace not 16-byte aligned
    (dict(page_size=48), _native.FA_ERR_UNSUPPORTED),       # the paged checks still apply
    (dict(D=96), _native.FA_ERR_UNSUPPORTED),
])
def test_fwd_paged_split_rejects_bad_arguments(lib, kw, code):
    assert call_fwd_paged_split(lib, **kw) == code


def test_paged_split_workspace_is_per_slice_lse_then_o(lib):
    f = lib.fa_fwd_paged_split_workspace_size
    rows = 2 * 4 * 3                                         # B * H * Nq query rows
    lse_bytes = (rows * 5 * 4 + 255) // 256 * 256             # padded to 256 bytes so O stays aligned
    assert f(2, 4, 3, 128, 5) == lse_bytes + rows * 5 * 128 * 4
    assert f(2, 4, 3, 256, 1) == (rows * 4 + 255) // 256 * 256 + rows * 256 * 4
    for bad in [(0, 4, 3, 128, 5), (2, 4, 3, 96, 5), (2, 4, 3, 128, 0), (2, 4, 3, 128, 257)]:
        assert f(*bad) == 0


def test_paged_split_count_rejects_bad_arguments(lib):
    f = lib.fa_fwd_paged_split_count
    assert f(2, 6, 4, 1, 128, 64, 8, 0) == 1                  # H not a multiple of Hkv
    assert f(2, 8, 2, 1, 96, 64, 8, 0) == 1                   # unsupported D
    assert f(0, 8, 2, 1, 128, 64, 8, 0) == 1


def test_binding_constants_match_the_header():
    import re
    text = open(HEADER).read()
    codes = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define (FA_(?:OK|ERR_\w+))\s+\(?(-?\d+)\)?", text)}
    assert codes, "no status codes found in the header"
    for name, value in codes.items():
        assert getattr(_native, name) == value, name
    m = re.search(r"#define FA_NOALLOC_SCRATCH_BYTES \((\d+)ull << (\d+)\)", text)
    assert m and _native.FA_NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
