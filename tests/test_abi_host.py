"""Host-side checks of the C-ABI library: it loads, it exports every entry
point its header declares, and argument validation returns the documented
status codes before anything reaches the GPU (no compute call here)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "mxfp4.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxfp4_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import mxfp4_block_quantization_gb300 as m
    return m


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mxfp4_quantize", "mxfp4_quantize_grouped", "mxfp4_dequantize", "mxfp4_swap_w13",
              "mxfp4_scale_bytes", "mxfp4_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    L = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_size_helpers(lib):
    assert lib.mxfp4_scale_bytes(128, 256) == 1024
    assert lib.mxfp4_scale_bytes(4096, 7168) == 917504
    assert lib.mxfp4_scale_bytes(1000, 2880) == 94208
    assert lib.mxfp4_scale_bytes(1, 32) == 512
    assert lib.mxfp4_scale_bytes(0, 32) == 0 and lib.mxfp4_scale_bytes(4, 48) == 0
    # 131072 rows over 384 experts, K = 7168: floor((131072 + 127*384)/128) tiles
    assert lib.mxfp4_grouped_scale_bytes_bound(131072, 384, 7168) == 1405 * 128 * 224
    assert lib.mxfp4_version() >= 100
    assert "OFFSETS" in lib.mxfp4_status_string(lib.MXFP4_EOFFSETS)


A = 1 << 32   # fake, 16-byte aligned addresses: validation fails before any use


def q(lib, x, M, K, ldx, c, s):
    return lib._lib.mxfp4_quantize(x, M, K, ldx, c, s, None)


def test_quantize_validation(lib):
    assert q(lib, A, -1, 32, 32, 2 * A, 3 * A) == lib.MXFP4_EINVAL
    assert q(lib, A, 4, 48, 48, 2 * A, 3 * A) == lib.MXFP4_ESHAPE
    assert q(lib, A, 4, 64, 32, 2 * A, 3 * A) == lib.MXFP4_ESHAPE
    assert q(lib, None, 4, 64, 64, 2 * A, 3 * A) == lib.MXFP4_EINVAL
    assert q(lib, A + 8, 4, 64, 64, 2 * A, 3 * A) == lib.MXFP4_EALIGN
    assert q(lib, A, 4, 64, 68, 2 * A, 3 * A) == lib.MXFP4_EALIGN
    assert q(lib, A, 4, 64, 64, 2 * A, 3 * A + 4) == lib.MXFP4_EALIGN
    # codes overlapping x, scales overlapping codes
    assert q(lib, A, 4, 64, 64, A + 256, 3 * A) == lib.MXFP4_EALIAS
    assert q(lib, A, 4, 64, 64, 2 * A, 2 * A + 64) == lib.MXFP4_EALIAS
    # empty work is a no-op, even with NULL pointers
    assert q(lib, None, 0, 64, 64, None, None) == lib.MXFP4_OK
    assert q(lib, None, 5, 0, 0, None, None) == lib.MXFP4_OK


def test_grouped_validation(lib):
    g = lib._lib.mxfp4_quantize_grouped
    assert g(A, 10, 64, 2 * A, -1, 3 * A, 4 * A, 5 * A, None, None) == lib.MXFP4_EINVAL
    assert g(A, 10, 48, 2 * A, 2, 3 * A, 4 * A, 5 * A, None, None) == lib.MXFP4_ESHAPE
    assert g(A, 10, 64, None, 2, 3 * A, 4 * A, 5 * A, None, None) == lib.MXFP4_EINVAL
    assert g(A, 10, 64, 2 * A, 0, 3 * A, 4 * A, 5 * A, None, None) == lib.MXFP4_EINVAL
    assert g(A, 10, 64, 2 * A, 2, 3 * A + 4, 4 * A, 5 * A, None, None) == lib.MXFP4_EALIGN
    assert g(A, 10, 64, 2 * A + 2, 2, 3 * A, 4 * A, 5 * A, None, None) == lib.MXFP4_EALIGN
    # scale_row_offsets overlapping the offsets input
    assert g(A, 10, 64, 2 * A, 2, 3 * A, 4 * A, 2 * A + 4, None, None) == lib.MXFP4_EALIAS
    # status overlapping codes
    assert g(A, 10, 64, 2 * A, 2, 3 * A, 4 * A, 5 * A, 3 * A + 16, None) == lib.MXFP4_EALIAS
    # padded rows must fit int32
    assert g(A, 2 ** 31 - 10, 32, 2 * A, 2, 3 * A, 4 * A, 5 * A, None, None) == lib.MXFP4_ESHAPE


def test_dequantize_validation(lib):
    d = lib._lib.mxfp4_dequantize
    assert d(A, 2 * A, 4, 40, 3 * A, None) == lib.MXFP4_ESHAPE
    assert d(A, 2 * A, -4, 64, 3 * A, None) == lib.MXFP4_EINVAL
    assert d(A, None, 4, 64, 3 * A, None) == lib.MXFP4_EINVAL
    assert d(A, 2 * A, 4, 64, 3 * A + 2, None) == lib.MXFP4_EALIGN
    assert d(A, 2 * A, 4, 64, A + 64, None) == lib.MXFP4_EALIAS
    assert d(None, None, 0, 64, None, None) == lib.MXFP4_OK


def test_swap_validation(lib):
    s = lib._lib.mxfp4_swap_w13
    ok_args = [A, 2 * A, None, 2, 8, 64, 0, 3 * A, 4 * A, None, None, 0, None, None]

    def call(**kw):
        names = ["ci", "si", "b13", "E", "two_n", "K", "tiled", "co", "so", "b13o", "b2", "n2",
                 "b2o", "st"]
        a = dict(zip(names, ok_args))
        a.update(kw)
        return s(*[a[n] for n in names])

    assert call(two_n=7) == lib.MXFP4_ESHAPE
    assert call(K=48) == lib.MXFP4_ESHAPE
    assert call(tiled=2) == lib.MXFP4_EINVAL
    assert call(E=-1) == lib.MXFP4_EINVAL
    assert call(co=None) == lib.MXFP4_EINVAL
    assert call(b13=5 * A) == lib.MXFP4_EINVAL              # bias without output
    assert call(co=3 * A + 8) == lib.MXFP4_EALIGN
    assert call(co=A + 64) == lib.MXFP4_EALIAS               # out overlaps codes_in
    assert call(so=3 * A + 128) == lib.MXFP4_EALIAS          # scales_out overlaps codes_out
    assert call(E=0) == lib.MXFP4_OK                          # nothing to do


def test_binding_rejects_cpu_tensors(lib):
    import torch
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        lib.quantize(x)


def test_grouped_gather_validation(lib):
    g = lib._lib.mxfp4_quantize_grouped_gather
    # x, n_src, K, ldx, idx, total, off, E, codes, scales, sro, status, stream
    ok = [A, 50, 64, 64, 2 * A, 10, 3 * A, 2, 4 * A, 5 * A, 6 * A, None, None]

    def call(**kw):
        names = ["x", "n", "K", "ldx", "idx", "tot", "off", "E", "c", "s", "sro", "st", "strm"]
        a = dict(zip(names, ok))
        a.update(kw)
        return g(*[a[n] for n in names])

    assert call(K=48, ldx=48) == lib.MXFP4_ESHAPE
    assert call(ldx=32) == lib.MXFP4_ESHAPE
    assert call(idx=None) == lib.MXFP4_EINVAL
    assert call(n=0) == lib.MXFP4_EINVAL
    assert call(idx=2 * A + 2) == lib.MXFP4_EALIGN
    assert call(ldx=68) == lib.MXFP4_EALIGN
    assert call(c=2 * A + 16) == lib.MXFP4_EALIAS            # codes overlap the indices
    assert call(sro=A + 64) == lib.MXFP4_EALIAS              # offsets out overlap x
    # the call may use the tail of codes as its workspace: nothing else may
    # share those bytes
    assert call(c=3 * A) == lib.MXFP4_EALIAS                 # codes overlap the offsets
    assert call(st=4 * A + 64) == lib.MXFP4_EALIAS           # status inside the codes
    assert call(sro=4 * A + 256) == lib.MXFP4_EALIAS         # offsets out inside the codes


def test_grouped_scatter_validation(lib):
    g = lib._lib.mxfp4_quantize_grouped_scatter
    # x, T, K, ldx, dest, top_k, total, off, E, codes, scales, sro, status, stream
    ok = [A, 50, 64, 64, 2 * A, 8, 400, 3 * A, 2, 4 * A, 5 * A, 6 * A, None, None]

    def call(**kw):
        names = ["x", "T", "K", "ldx", "dst", "k", "tot", "off", "E", "c", "s", "sro", "st",
                 "strm"]
        a = dict(zip(names, ok))
        a.update(kw)
        return g(*[a[n] for n in names])

    assert call(K=48, ldx=48) == lib.MXFP4_ESHAPE
    assert call(ldx=32) == lib.MXFP4_ESHAPE
    assert call(k=0) == lib.MXFP4_EINVAL
    assert call(k=lib.MXFP4_SCATTER_MAX_TOP_K + 1) == lib.MXFP4_EINVAL
    assert call(dst=None) == lib.MXFP4_EINVAL
    assert call(c=None) == lib.MXFP4_EINVAL
    assert call(E=0) == lib.MXFP4_EINVAL                     # rows but no segments
    assert call(dst=2 * A + 2) == lib.MXFP4_EALIGN
    assert call(ldx=68) == lib.MXFP4_EALIGN
    assert call(c=2 * A + 16) == lib.MXFP4_EALIAS            # codes overlap the routes
    assert call(sro=A + 64) == lib.MXFP4_EALIAS              # offsets out overlap x
    assert call(s=4 * A + 64) == lib.MXFP4_EALIAS            # scales overlap codes
    # no tokens: dest_rows and x may be NULL (pad rows are still written)
    assert call(T=0, x=None, dst=None, off=None) == lib.MXFP4_EINVAL


def test_grouped_scatter_ws_validation(lib):
    f = lib._lib.mxfp4_quantize_grouped_scatter_ws
    need = lib.mxfp4_scatter_workspace_bytes(50, 400, 2, 64)
    # token of every padded row (floor((R + 127E)/128)*128 ints), then T rows of 4 words
    assert need == 4 * ((400 + 254) // 128 * 128) + 50 * 4 * 4
    assert lib.mxfp4_scatter_workspace_bytes(50, 400, 2, 7168) == 4 * 640 + 50 * 56 * 4
    assert lib.mxfp4_scatter_workspace_bytes(50, 400, 2, 48) == 0
    assert lib.mxfp4_scatter_workspace_bytes(50, 400, -1, 64) == 0
    # x, T, K, ldx, dest, top_k, total, off, E, ws, ws_bytes, codes, scales, sro, status, stream
    ok = [A, 50, 64, 64, 2 * A, 8, 400, 3 * A, 2, 8 * A, need, 4 * A, 5 * A, 6 * A, None, None]

    def call(**kw):
        names = ["x", "T", "K", "ldx", "dst", "k", "tot", "off", "E", "ws", "wsb", "c", "s",
                 "sro", "st", "strm"]
        a = dict(zip(names, ok))
        a.update(kw)
        return f(*[a[n] for n in names])

    assert call(ws=None) == lib.MXFP4_EINVAL
    assert call(wsb=need - 16) == lib.MXFP4_EINVAL
    assert call(ws=8 * A + 8) == lib.MXFP4_EALIGN
    assert call(ws=4 * A + 16) == lib.MXFP4_EALIAS            # workspace overlaps the codes
    assert call(ws=2 * A) == lib.MXFP4_EALIAS                 # workspace overlaps the routes
    assert call(k=0) == lib.MXFP4_EINVAL
    assert call(K=48, ldx=48) == lib.MXFP4_ESHAPE
    assert call(T=(1 << 31) // 4 + 1) == lib.MXFP4_ESHAPE
    assert lib._lib.mxfp4_quantize_grouped_scatter_ws_f16(*ok[:2], 48, 48, *ok[4:]) == \
        lib.MXFP4_ESHAPE


def test_nvfp4_grouped_scatter_validation(lib):
    f = lib._lib.mxfp4_quantize_nvfp4_grouped_scatter
    # x, T, K, ldx, dest, top_k, total, off, E, g, codes, scales, sro, status, stream
    ok = [A, 50, 64, 64, 2 * A, 8, 400, 3 * A, 2, 9 * A, 4 * A, 5 * A, 6 * A, None, None]

    def call(**kw):
        names = ["x", "T", "K", "ldx", "dst", "k", "tot", "off", "E", "g", "c", "s", "sro",
                 "st", "strm"]
        a = dict(zip(names, ok))
        a.update(kw)
        return f(*[a[n] for n in names])

    assert call(K=40, ldx=40) == lib.MXFP4_ESHAPE          # K % 16 != 0
    assert call(ldx=48) == lib.MXFP4_ESHAPE                 # ldx < K
    assert call(k=0) == lib.MXFP4_EINVAL
    assert call(k=lib.MXFP4_SCATTER_MAX_TOP_K + 1) == lib.MXFP4_EINVAL
    assert call(g=None) == lib.MXFP4_EINVAL
    assert call(dst=None) == lib.MXFP4_EINVAL
    assert call(E=0) == lib.MXFP4_EINVAL
    assert call(g=9 * A + 2) == lib.MXFP4_EALIGN
    assert call(x=A + 8) == lib.MXFP4_EALIGN
    assert call(c=2 * A + 16) == lib.MXFP4_EALIAS            # codes overlap the routes
    assert call(s=9 * A - 64) == lib.MXFP4_EALIAS            # scales overlap the global scales
    assert lib._lib.mxfp4_quantize_nvfp4_grouped_scatter_f16(
        *ok[:2], 40, 40, *ok[4:]) == lib.MXFP4_ESHAPE


def test_nvfp4_grouped_scatter_ws_validation(lib):
    f = lib._lib.mxfp4_quantize_nvfp4_grouped_scatter_ws
    need = lib.mxfp4_nvfp4_scatter_workspace_bytes(400, 2, 64)
    # PT = floor((400 + 254) / 128) * 128 = 640 padded rows: the row map (4 B) and a staged
    # row of ceil(64/64) = 1 scale word, padded to 4 words (16 B), per padded row
    assert need == 640 * (4 + 16)
    assert lib.mxfp4_nvfp4_scatter_workspace_bytes(400, 2, 7168) == 640 * (4 + 448)
    assert lib.mxfp4_nvfp4_scatter_workspace_bytes(400, 2, 40) == 0
    # x, T, K, ldx, dest, top_k, total, off, E, g, ws, ws_bytes, codes, scales, sro, st, stream
    ok = [A, 50, 64, 64, 2 * A, 8, 400, 3 * A, 2, 9 * A, 8 * A, need, 4 * A, 5 * A, 6 * A,
          None, None]

    def call(**kw):
        names = ["x", "T", "K", "ldx", "dst", "k", "tot", "off", "E", "g", "ws", "wsb", "c", "s",
                 "sro", "st", "strm"]
        a = dict(zip(names, ok))
        a.update(kw)
        return f(*[a[n] for n in names])

    assert call(ws=None) == lib.MXFP4_EINVAL
    assert call(wsb=need - 16) == lib.MXFP4_EINVAL
    assert call(ws=8 * A + 8) == lib.MXFP4_EALIGN
    assert call(ws=4 * A + 16) == lib.MXFP4_EALIAS            # workspace overlaps the codes
    assert call(K=40, ldx=40) == lib.MXFP4_ESHAPE


def test_quantize_f16_validation(lib):
    f = lib._lib.mxfp4_quantize_f16
    assert f(A, 4, 48, 48, 2 * A, 3 * A, None) == lib.MXFP4_ESHAPE
    assert f(A + 8, 4, 64, 64, 2 * A, 3 * A, None) == lib.MXFP4_EALIGN
    assert f(A, 4, 64, 64, A + 64, 3 * A, None) == lib.MXFP4_EALIAS
    assert f(None, 0, 64, 64, None, None, None) == lib.MXFP4_OK


def test_nvfp4_validation(lib):
    q = lib._lib.mxfp4_quantize_nvfp4
    d = lib._lib.mxfp4_dequantize_nvfp4
    assert lib.mxfp4_nvfp4_scale_bytes(1000, 2880) == 1024 * 180
    assert lib.mxfp4_nvfp4_scale_bytes(4, 24) == 0
    assert q(A, 4, 24, 24, 9 * A, 2 * A, 3 * A, None) == lib.MXFP4_ESHAPE
    assert q(A, 4, 64, 64, None, 2 * A, 3 * A, None) == lib.MXFP4_EINVAL
    assert q(A, 4, 64, 64, 9 * A + 2, 2 * A, 3 * A, None) == lib.MXFP4_EALIGN
    assert q(A, 4, 64, 64, 9 * A, A + 64, 3 * A, None) == lib.MXFP4_EALIAS
    assert q(A, 4, 64, 64, 3 * A + 4, 2 * A, 3 * A, None) == lib.MXFP4_EALIAS
    assert q(None, 0, 64, 64, None, None, None, None) == lib.MXFP4_OK
    assert d(A, 2 * A, 9 * A, 4, 24, 3 * A, None) == lib.MXFP4_ESHAPE
    assert d(A, 2 * A, None, 4, 64, 3 * A, None) == lib.MXFP4_EINVAL
    assert d(A, 2 * A, 9 * A, 4, 64, A + 32, None) == lib.MXFP4_EALIAS


def test_binding_rejects_mixed_devices(lib):
    import torch
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        lib._device_of(x, torch.zeros(1, device="meta"))


def test_debug_library_exports_both_headers(lib):
    import os
    L = ctypes.CDLL(lib.DEBUG_LIB_PATH)
    debug_h = os.path.join(ROOT, "include", "mxfp4_debug.h")
    text = re.sub(r"/\*.*?\*/", "", open(debug_h).read(), flags=re.S)
    names = declared_functions() + re.findall(r"\b(mxfp4_\w+)\s*\(", text)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert not hasattr(ctypes.CDLL(lib.LIB_PATH), "mxfp4_debug_bounds_violations")


def test_nvfp4_grouped_validation(lib):
    f = lib._lib.mxfp4_quantize_nvfp4_grouped
    # x, total, K, off, E, g, codes, scales, sro, status, stream
    ok = [A, 300, 64, 3 * A, 3, 7 * A, 4 * A, 5 * A, 6 * A, None, None]

    def call(**kw):
        names = ["x", "tot", "K", "off", "E", "g", "c", "s", "sro", "st", "strm"]
        a = dict(zip(names, ok))
        a.update(kw)
        return f(*[a[n] for n in names])

    assert call(K=40) == lib.MXFP4_ESHAPE
    assert call(g=None) == lib.MXFP4_EINVAL
    assert call(E=0) == lib.MXFP4_EINVAL
    assert call(x=A + 8) == lib.MXFP4_EALIGN
    assert call(g=7 * A + 2) == lib.MXFP4_EALIGN
    assert call(c=A + 64) == lib.MXFP4_EALIAS                # codes overlap x
    assert call(sro=7 * A) == lib.MXFP4_EALIAS               # offsets out overlap the scales in
    assert lib.mxfp4_nvfp4_grouped_scale_bytes_bound(300, 3, 64) == (300 + 381) // 128 * 128 * 4
    assert lib.mxfp4_nvfp4_grouped_scale_bytes_bound(300, 3, 40) == 0


def test_nvfp4_f16_forms_share_the_validation(lib):
    q = lib._lib.mxfp4_quantize_nvfp4_f16
    assert q(A, 4, 24, 24, 9 * A, 2 * A, 3 * A, None) == lib.MXFP4_ESHAPE
    assert q(A, 4, 64, 64, None, 2 * A, 3 * A, None) == lib.MXFP4_EINVAL
    assert q(A + 8, 4, 64, 64, 9 * A, 2 * A, 3 * A, None) == lib.MXFP4_EALIGN
    assert q(A, 4, 64, 64, 9 * A, A + 64, 3 * A, None) == lib.MXFP4_EALIAS
    assert q(None, 0, 64, 64, None, None, None, None) == lib.MXFP4_OK
    f = lib._lib.mxfp4_quantize_nvfp4_grouped_f16
    assert f(A, 300, 40, 3 * A, 3, 7 * A, 4 * A, 5 * A, 6 * A, None, None) == lib.MXFP4_ESHAPE
    assert f(A, 300, 64, 3 * A, 3, None, 4 * A, 5 * A, 6 * A, None, None) == lib.MXFP4_EINVAL
    assert f(A, 300, 64, 3 * A, 3, 7 * A + 2, 4 * A, 5 * A, 6 * A, None,
             None) == lib.MXFP4_EALIGN
    assert f(A, 300, 64, 3 * A, 3, 7 * A, A + 64, 5 * A, 6 * A, None, None) == lib.MXFP4_EALIAS


def test_f16_grouped_forms_share_the_validation(lib):
    L = lib._lib
    # K % 32 != 0 is refused by every FP16 grouped form, before any launch
    assert L.mxfp4_quantize_grouped_f16(A, 10, 48, 2 * A, 1, 3 * A, 4 * A, 5 * A, None,
                                        None) == lib.MXFP4_ESHAPE
    assert L.mxfp4_quantize_grouped_gather_f16(A, 10, 48, 48, 2 * A, 10, 3 * A, 1, 4 * A, 5 * A,
                                               6 * A, None, None) == lib.MXFP4_ESHAPE
    assert L.mxfp4_quantize_grouped_scatter_f16(A, 10, 48, 48, 2 * A, 1, 10, 3 * A, 1, 4 * A,
                                                5 * A, 6 * A, None, None) == lib.MXFP4_ESHAPE
    assert L.mxfp4_quantize_grouped_scatter_f16(A, 10, 64, 64, 2 * A, 0, 10, 3 * A, 1, 4 * A,
                                                5 * A, 6 * A, None, None) == lib.MXFP4_EINVAL


def test_gather_ws_validation(lib):
    f = lib._lib.mxfp4_quantize_grouped_gather_ws
    ws_need = lib.mxfp4_gather_workspace_bytes(50, 10, 2, 64)
    # inverse map 4 * (33T + 1 + 2R): counts, overflow counter, 32-row buckets, overflow
    # rows and tokens; the token of each of the floor((R + 127E)/128)*128 padded rows; then,
    # from the next 16-byte boundary, T rows of ceil(K/128) scale words padded to 4 words
    inv = 4 * (33 * 50 + 1 + 2 * 10)
    tok = 4 * ((10 + 127 * 2) // 128 * 128)
    assert inv == 6684 and tok == 1024 and ws_need == 7712 + 50 * 4 * 4
    assert lib.mxfp4_gather_workspace_bytes(50, 10, 2, 0) == 6688     # the map alone, rounded
    assert lib.mxfp4_gather_workspace_bytes(50, 10, 2, 7168) == 7712 + 50 * 56 * 4
    assert lib.mxfp4_gather_workspace_bytes(50, 10, 2, 160) == 7712 + 50 * 4 * 4  # 2 words -> 4
    assert lib.mxfp4_gather_workspace_bytes(50, 10, 2, 48) == 0
    assert lib.mxfp4_gather_workspace_bytes(50, 10, -1, 64) == 0
    assert lib.mxfp4_gather_workspace_bytes(-1, 10, 2, 64) == 0
    # x, n_src, K, ldx, idx, total, off, E, ws, ws_bytes, codes, scales, sro, status, stream
    ok = [A, 50, 64, 64, 2 * A, 10, 3 * A, 2, 8 * A, ws_need, 4 * A, 5 * A, 6 * A, None, None]

    def call(**kw):
        names = ["x", "n", "K", "ldx", "idx", "tot", "off", "E", "ws", "wsb", "c", "s", "sro",
                 "st", "strm"]
        a = dict(zip(names, ok))
        a.update(kw)
        return f(*[a[n] for n in names])

    assert call(ws=None) == lib.MXFP4_EINVAL
    assert call(wsb=ws_need - 16) == lib.MXFP4_EINVAL
    assert call(ws=8 * A + 8) == lib.MXFP4_EALIGN
    assert call(ws=4 * A + 16) == lib.MXFP4_EALIAS            # workspace overlaps the codes
    assert call(ws=2 * A) == lib.MXFP4_EALIAS                 # workspace overlaps the indices
    assert call(K=48, ldx=48) == lib.MXFP4_ESHAPE
    assert call(n=(1 << 31) // 4 + 1, ldx=64) == lib.MXFP4_ESHAPE


def test_noalloc_gather_rejects_oversized_scratch(lib):
    """Sizes whose inverse map would not fit the library's fixed scratch are
    refused with MXFP4_ESCRATCH before any device work (no GPU needed)."""
    f = lib._lib.mxfp4_quantize_grouped_gather_noalloc
    assert lib.mxfp4_gather_workspace_bytes(10_000_000, 1, 1, 0) > lib.MXFP4_NOALLOC_SCRATCH_BYTES
    rc = f(A, 10_000_000, 64, 64, 2 * A, 1, 3 * A, 1, 4 * A, 5 * A, 6 * A, None, None)
    assert rc == lib.MXFP4_ESCRATCH
    assert "MXFP4_ESCRATCH" in lib.mxfp4_status_string(rc)
    assert f(A, -1, 64, 64, 2 * A, 1, 3 * A, 1, 4 * A, 5 * A, 6 * A, None, None) == lib.MXFP4_EINVAL


def test_noalloc_gather_checks_shapes_before_its_scratch_size(lib):
    """The call without allocation reports the same errors as the workspace
    call in the same order, so a shape fault or an int32 overflow is
    MXFP4_ESHAPE even when the sizes would not fit the scratch either, and
    MXFP4_ESCRATCH is left for a well-formed call that is too large."""
    f = lib._lib.mxfp4_quantize_grouped_gather_noalloc
    big = 10_000_000                                   # map far beyond the scratch
    # x, n_src, K, ldx, idx, total, off, E, codes, scales, sro, status, stream
    ok = [A, big, 64, 64, 2 * A, 1, 3 * A, 1, 4 * A, 5 * A, 6 * A, None, None]

    def call(**kw):
        names = ["x", "n", "K", "ldx", "idx", "tot", "off", "E", "c", "s", "sro", "st", "strm"]
        a = dict(zip(names, ok))
        a.update(kw)
        return f(*[a[n] for n in names])

    assert call() == lib.MXFP4_ESCRATCH
    assert call(K=48, ldx=48) == lib.MXFP4_ESHAPE             # K % 32 != 0
    assert call(ldx=32) == lib.MXFP4_ESHAPE                   # ldx < K
    assert call(n=(1 << 31) // 4 + 1) == lib.MXFP4_ESHAPE     # token ids must stay int32
    assert call(tot=(1 << 31) - 100, E=2) == lib.MXFP4_ESHAPE  # padded rows overflow int32
    assert call(off=None) == lib.MXFP4_EINVAL
    assert call(E=0) == lib.MXFP4_EINVAL                      # rows but no expert
    assert call(n=0) == lib.MXFP4_EINVAL                      # rows but no source row
    # the workspace call gives the same codes for the same faults
    g = lib._lib.mxfp4_quantize_grouped_gather_ws
    assert g(A, big, 48, 48, 2 * A, 1, 3 * A, 1, 8 * A, 1 << 40, 4 * A, 5 * A, 6 * A, None,
             None) == lib.MXFP4_ESHAPE
    assert g(A, (1 << 31) // 4 + 1, 64, 64, 2 * A, 1, 3 * A, 1, 8 * A, 1 << 40, 4 * A, 5 * A,
             6 * A, None, None) == lib.MXFP4_ESHAPE


def test_gather_workspace_bytes_is_zero_beyond_the_call_limits(lib):
    """The size query returns 0 (no valid call) where the calls themselves
    would refuse the shape, instead of a truncated size."""
    assert lib.mxfp4_gather_workspace_bytes(50, 10, 2, 1 << 40) == 0
    assert lib.mxfp4_gather_workspace_bytes(50, 10, 2, 1 << 38) == 0
    assert lib.mxfp4_gather_workspace_bytes(50, 10, 2, 1 << 20) > 0
    assert lib.mxfp4_gather_workspace_bytes((1 << 31) // 4 + 1, 10, 2, 64) == 0


def test_route_validation(lib):
    """mxfp4_moe_route refuses bad arguments before any device work."""
    f = lib._lib.mxfp4_moe_route
    ws_need = lib.mxfp4_route_workspace_bytes(300, 4, 13)
    # 1200 routes: 5 chunks of 256 x (E + 1) counts and flags, and a 16-byte ticket
    assert ws_need == (5 * 14 + 4) * 4
    assert lib.mxfp4_route_workspace_bytes(16384, 8, 384) == (512 * 385 + 4) * 4
    assert lib.mxfp4_route_workspace_bytes(10, 8, lib.MXFP4_ROUTE_MAX_EXPERTS + 1) == 0
    assert lib.mxfp4_route_workspace_bytes(10, 0, 4) == 0
    # ids, T, top_k, E, ws, ws_bytes, offsets, dest, rows, status, stream
    ok = [A, 300, 4, 13, 8 * A, ws_need, 2 * A, 3 * A, 4 * A, 5 * A, None]

    def call(**kw):
        names = ["ids", "T", "k", "E", "ws", "wsb", "off", "dest", "rows", "st", "strm"]
        a = dict(zip(names, ok))
        a.update(kw)
        return f(*[a[n] for n in names])

    assert call(T=-1) == lib.MXFP4_EINVAL
    assert call(k=0) == lib.MXFP4_EINVAL
    assert call(E=0) == lib.MXFP4_EINVAL
    assert call(E=lib.MXFP4_ROUTE_MAX_EXPERTS + 1) == lib.MXFP4_ESHAPE
    assert call(T=(1 << 30), k=2) == lib.MXFP4_ESHAPE
    assert call(ids=None) == lib.MXFP4_EINVAL
    assert call(off=None) == lib.MXFP4_EINVAL
    assert call(dest=None) == lib.MXFP4_EINVAL
    assert call(ws=None) == lib.MXFP4_EINVAL
    assert call(wsb=ws_need - 4) == lib.MXFP4_EINVAL
    assert call(ws=8 * A + 8) == lib.MXFP4_EALIGN
    assert call(dest=3 * A + 2) == lib.MXFP4_EALIGN
    assert call(dest=A + 16) == lib.MXFP4_EALIAS          # dest_rows overlaps the ids
    assert call(rows=3 * A + 64) == lib.MXFP4_EALIAS      # row_index overlaps dest_rows
    assert call(st=2 * A + 4) == lib.MXFP4_EALIAS         # status inside the offsets


def test_size_queries_return_zero_instead_of_wrapping(lib):
    """Every size query answers 0 for sizes whose byte count would not fit in
    int64, or whose k tiles the calls cannot count, instead of a wrapped or
    truncated size; ordinary sizes are unchanged."""
    big_rows, big_k = 1 << 62, 1 << 40
    assert lib.mxfp4_scale_bytes(big_rows, 1024) == 0
    assert lib.mxfp4_scale_bytes(1 << 40, 1 << 30) == 0            # rows x cols overflows
    assert lib.mxfp4_grouped_scale_bytes_bound(big_rows, 4, 1024) == 0
    assert lib.mxfp4_grouped_scale_bytes_bound(1 << 40, 4, 1 << 30) == 0
    assert lib.mxfp4_nvfp4_scale_bytes(big_rows, 1024) == 0
    assert lib.mxfp4_nvfp4_scale_bytes(1 << 40, 1 << 30) == 0
    assert lib.mxfp4_nvfp4_grouped_scale_bytes_bound(1 << 40, 4, 1 << 30) == 0
    assert lib.mxfp4_scatter_workspace_bytes(100, 400, 2, big_k) == 0
    assert lib.mxfp4_nvfp4_scatter_workspace_bytes(400, 2, big_k) == 0
    assert lib.mxfp4_gather_workspace_bytes(100, 400, 2, big_k) == 0
    # ordinary sizes: 4096 x 7168 -> 4096 rows x 224 (MXFP4) / 448 (NVFP4) scale bytes
    assert lib.mxfp4_scale_bytes(4096, 7168) == 4096 * 224
    assert lib.mxfp4_nvfp4_scale_bytes(4096, 7168) == 4096 * 448
    assert lib.mxfp4_grouped_scale_bytes_bound(131072, 384, 7168) == \
        (131072 + 127 * 384) // 128 * 128 * 224
