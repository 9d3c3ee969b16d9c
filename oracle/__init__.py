"""CPU oracle of MXFP4 block quantization — TEST INFRASTRUCTURE ONLY.

Plain, slow, single-threaded C (``mxfp4_oracle.c``) behind numpy wrappers.
Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the GPU library never does, and the two
share no code.  Each wrapper names the step of the method it runs; the C file
cites the pages for every step.

Pins: see the CPU tests (``tests/test_oracle_*.py``).  The relative-L2 and
saturation reports computed from oracle outputs have no independent pin
(parity unpinned).
"""
import ctypes
import os
import threading

import numpy as np

from . import build as _build

_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_bf16_to_double.restype = ctypes.c_double
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_double_to_bf16_rne.restype = ctypes.c_uint16
        L.orc_double_to_bf16_rne.argtypes = [ctypes.c_double]
        L.orc_block_absmax.restype = ctypes.c_float
        L.orc_block_absmax.argtypes = [_u16p, _i64]
        L.orc_e8m0_scale.restype = ctypes.c_uint8
        L.orc_e8m0_scale.argtypes = [ctypes.c_float]
        L.orc_e2m1_encode.restype = ctypes.c_uint8
        L.orc_e2m1_encode.argtypes = [ctypes.c_uint16, ctypes.c_uint8]
        L.orc_e2m1_decode.restype = ctypes.c_double
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.orc_e8m0_scale_many.restype = None
        L.orc_e8m0_scale_many.argtypes = [_u16p, _i64, _u8p]
        L.orc_e2m1_encode_many.restype = None
        L.orc_e2m1_encode_many.argtypes = [_u16p, _i64, ctypes.c_uint8, _u8p]
        L.orc_dequant_value_many.restype = None
        L.orc_dequant_value_many.argtypes = [_u8p, _u8p, _i64, _u16p]
        L.orc_scale_bytes.restype = ctypes.c_size_t
        L.orc_scale_bytes.argtypes = [_i64, _i64]
        L.orc_quantize_flat.restype = None
        L.orc_quantize_flat.argtypes = [_u16p, _i64, _i64, _i64, _u8p, _u8p]
        L.orc_tile_scales.restype = None
        L.orc_tile_scales.argtypes = [_u8p, _i64, _i64, _u8p]
        L.orc_untile_scales.restype = None
        L.orc_untile_scales.argtypes = [_u8p, _i64, _i64, _u8p]
        L.orc_quantize.restype = None
        L.orc_quantize.argtypes = [_u16p, _i64, _i64, _i64, _u8p, _u8p]
        L.orc_quantize_grouped.restype = ctypes.c_int
        L.orc_quantize_grouped.argtypes = [_u16p, _i64, _i64, _i32p, ctypes.c_int32,
                                           _u8p, _u8p, _i32p]
        L.orc_f16_to_double.restype = ctypes.c_double
        L.orc_f16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_e2m1_encode_f16_many.restype = None
        L.orc_e2m1_encode_f16_many.argtypes = [_u16p, _i64, ctypes.c_uint8, _u8p]
        L.orc_f16_to_double_many.restype = None
        L.orc_f16_to_double_many.argtypes = [_u16p, _i64, _f64p]
        L.orc_quantize_f16.restype = None
        L.orc_quantize_f16.argtypes = [_u16p, _i64, _i64, _i64, _u8p, _u8p]
        L.orc_quantize_flat_f16.restype = None
        L.orc_quantize_flat_f16.argtypes = [_u16p, _i64, _i64, _i64, _u8p, _u8p]
        L.orc_e4m3_to_double.restype = ctypes.c_double
        L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_from_double.restype = ctypes.c_uint8
        L.orc_e4m3_from_double.argtypes = [ctypes.c_double]
        L.orc_e4m3_from_double_many.restype = None
        L.orc_e4m3_from_double_many.argtypes = [_f64p, _i64, _u8p]
        L.orc_nvfp4_scale_bytes.restype = ctypes.c_size_t
        L.orc_nvfp4_scale_bytes.argtypes = [_i64, _i64]
        L.orc_nvfp4_quantize_flat.restype = None
        L.orc_nvfp4_quantize_flat.argtypes = [_u16p, _i64, _i64, _i64, ctypes.c_float, _u8p, _u8p]
        L.orc_nvfp4_quantize.restype = None
        L.orc_nvfp4_quantize.argtypes = [_u16p, _i64, _i64, _i64, ctypes.c_float, _u8p, _u8p]
        L.orc_moe_route.restype = ctypes.c_int
        L.orc_moe_route.argtypes = [_i32p, _i64, ctypes.c_int32, ctypes.c_int32, _i32p, _i32p,
                                    _i32p]
        L.orc_nvfp4_dequantize.restype = None
        L.orc_nvfp4_dequantize.argtypes = [_u8p, _u8p, _i64, _i64, ctypes.c_float, _u16p]
        L.orc_e8m0_scale_legacy.restype = ctypes.c_uint8
        L.orc_e8m0_scale_legacy.argtypes = [ctypes.c_float]
        L.orc_quantize_flat_legacy.restype = None
        L.orc_quantize_flat_legacy.argtypes = [_u16p, _i64, _i64, _i64, _u8p, _u8p]
        L.orc_nvfp4_quantize_grouped.restype = ctypes.c_int
        L.orc_nvfp4_quantize_grouped.argtypes = [_u16p, _i64, _i64, _i32p, ctypes.c_int32, _f32p,
                                                 _u8p, _u8p, _i32p]
        L.orc_quantize_grouped_f16.restype = ctypes.c_int
        L.orc_quantize_grouped_f16.argtypes = [_u16p, _i64, _i64, _i32p, ctypes.c_int32,
                                               _u8p, _u8p, _i32p]
        L.orc_quantize_grouped_gather_f16.restype = ctypes.c_int
        L.orc_quantize_grouped_gather_f16.argtypes = [_u16p, _i64, _i64, _i64, _i32p, _i64,
                                                      _i32p, ctypes.c_int32, _u8p, _u8p, _i32p]
        L.orc_quantize_grouped_scatter_f16.restype = ctypes.c_int
        L.orc_quantize_grouped_scatter_f16.argtypes = [_u16p, _i64, _i64, _i64, _i32p,
                                                       ctypes.c_int32, _i64, _i32p,
                                                       ctypes.c_int32, _u8p, _u8p, _i32p]
        L.orc_nvfp4_quantize_f16.restype = None
        L.orc_nvfp4_quantize_f16.argtypes = [_u16p, _i64, _i64, _i64, ctypes.c_float, _u8p, _u8p]
        L.orc_nvfp4_quantize_grouped_f16.restype = ctypes.c_int
        L.orc_nvfp4_quantize_grouped_f16.argtypes = [_u16p, _i64, _i64, _i32p, ctypes.c_int32,
                                                     _f32p, _u8p, _u8p, _i32p]
        for name in ("orc_nvfp4_quantize_grouped_scatter",
                     "orc_nvfp4_quantize_grouped_scatter_f16"):
            getattr(L, name).restype = ctypes.c_int
            getattr(L, name).argtypes = [_u16p, _i64, _i64, _i64, _i32p, ctypes.c_int32, _i64,
                                         _i32p, ctypes.c_int32, _f32p, _u8p, _u8p, _i32p]
        L.orc_quantize_grouped_scatter.restype = ctypes.c_int
        L.orc_quantize_grouped_scatter.argtypes = [_u16p, _i64, _i64, _i64, _i32p, ctypes.c_int32,
                                                   _i64, _i32p, ctypes.c_int32, _u8p, _u8p, _i32p]
        L.orc_quantize_grouped_gather.restype = ctypes.c_int
        L.orc_quantize_grouped_gather.argtypes = [_u16p, _i64, _i64, _i64, _i32p, _i64, _i32p,
                                                  ctypes.c_int32, _u8p, _u8p, _i32p]
        L.orc_dequantize.restype = None
        L.orc_dequantize.argtypes = [_u8p, _u8p, _i64, _i64, _u16p]
        L.orc_swap_halves.restype = None
        L.orc_swap_halves.argtypes = [_u8p, _u8p, _i64, _i64, _i64]
        L.orc_swap_bias_bf16.restype = None
        L.orc_swap_bias_bf16.argtypes = [_f32p, _u16p, _i64, _i64]
        L.orc_cast_bf16.restype = None
        L.orc_cast_bf16.argtypes = [_f32p, _u16p, _i64]
        L.orc_swap_w13.restype = None
        L.orc_swap_w13.argtypes = [_u8p, _u8p, _f32p, ctypes.c_int32, _i64, _i64,
                                   ctypes.c_int32, _u8p, _u8p, _u16p, _f32p, _i64, _u16p]
        _lib = L
    return _lib


def _p(a, t):
    return a.ctypes.data_as(t) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- scalars
def bf16_to_double(b: int) -> float:
    return lib().orc_bf16_to_double(int(b))


def double_to_bf16(d: float) -> int:
    """Round a double to the nearest BF16 (ties to even); returns the bits."""
    return int(lib().orc_double_to_bf16_rne(float(d)))


def e8m0_scale(vecmax: float) -> int:
    """Step 2: scale exponent of a block whose absmax is ``vecmax`` (float32)."""
    return int(lib().orc_e8m0_scale(float(np.float32(vecmax))))


def e2m1_encode(xbits: int, s: int) -> int:
    """Step 3: nibble of one BF16 element under scale exponent ``s``."""
    return int(lib().orc_e2m1_encode(int(xbits), int(s)))


def e2m1_decode(nib: int) -> float:
    return lib().orc_e2m1_decode(int(nib))


def scale_bytes(M: int, K: int) -> int:
    return int(lib().orc_scale_bytes(int(M), int(K)))


# ----------------------------------------------------------------- vectors
def e8m0_scale_many(vbits: np.ndarray) -> np.ndarray:
    """Step 2 over BF16 bit patterns taken as vecMax."""
    v = _c(vbits, np.uint16).ravel()
    s = np.empty(v.size, np.uint8)
    lib().orc_e8m0_scale_many(_p(v, _u16p), v.size, _p(s, _u8p))
    return s


def e2m1_encode_many(xbits: np.ndarray, s: int) -> np.ndarray:
    """Step 3 over many BF16 elements sharing scale exponent ``s``."""
    x = _c(xbits, np.uint16).ravel()
    out = np.empty(x.size, np.uint8)
    lib().orc_e2m1_encode_many(_p(x, _u16p), x.size, int(s), _p(out, _u8p))
    return out


def dequant_value_many(nib: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Step 7 per element: BF16 bits of e2m1(nib) * 2^(s-127)."""
    n = _c(nib, np.uint8).ravel()
    sc = _c(np.broadcast_to(s, n.shape), np.uint8).ravel()
    y = np.empty(n.size, np.uint16)
    lib().orc_dequant_value_many(_p(n, _u8p), _p(sc, _u8p), n.size, _p(y, _u16p))
    return y


# ---------------------------------------------------------------- matrices
def quantize_flat(xbits: np.ndarray):
    """Steps 1-4: (codes [M, K/2], flat scales [M, K/32]) of a BF16 [M, K]."""
    x = _c(xbits, np.uint16)
    M, K = x.shape
    codes = np.zeros((M, K // 2), np.uint8)
    flat = np.zeros((M, K // 32), np.uint8)
    if M and K:
        lib().orc_quantize_flat(_p(x, _u16p), M, K, K, _p(codes, _u8p), _p(flat, _u8p))
    return codes, flat


def e8m0_scale_legacy(vecmax: float) -> int:
    """The pre-fix scale biased_exp(vecMax/6) (comparison only)."""
    return int(lib().orc_e8m0_scale_legacy(float(vecmax)))


def quantize_flat_legacy(xbits: np.ndarray):
    """Steps 1-4 with the pre-fix scale (comparison only): (codes, flat)."""
    x = _c(xbits, np.uint16)
    M, K = x.shape
    codes = np.zeros((M, K // 2), np.uint8)
    flat = np.zeros((M, K // 32), np.uint8)
    if M and K:
        lib().orc_quantize_flat_legacy(_p(x, _u16p), M, K, K, _p(codes, _u8p), _p(flat, _u8p))
    return codes, flat


def tile(flat: np.ndarray) -> np.ndarray:
    """Step 5: flat [M, sK] scales -> tiled bytes (zero padding)."""
    f = _c(flat, np.uint8)
    M, sK = f.shape
    out = np.zeros(scale_bytes(M, sK * 32), np.uint8)
    if out.size:
        lib().orc_tile_scales(_p(f, _u8p), M, sK, _p(out, _u8p))
    return out


def untile(tiled: np.ndarray, M: int, sK: int) -> np.ndarray:
    """Inverse of step 5: tiled bytes -> flat [M, sK]."""
    t = _c(tiled, np.uint8).ravel()
    out = np.zeros((M, sK), np.uint8)
    if M and sK:
        lib().orc_untile_scales(_p(t, _u8p), M, sK, _p(out, _u8p))
    return out


def quantize(xbits: np.ndarray):
    """Steps 1-5: (codes [M, K/2], tiled scales) of a BF16 [M, K] (bits)."""
    x = _c(xbits, np.uint16)
    M, K = x.shape
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros(scale_bytes(M, K), np.uint8)
    if M and K:
        lib().orc_quantize(_p(x, _u16p), M, K, K, _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def grouped_scale_bytes_bound(total_rows: int, E: int, K: int) -> int:
    tiles = (total_rows + 127 * E) // 128
    return tiles * 128 * ((K // 32 + 3) // 4 * 4)


def quantize_grouped(xbits: np.ndarray, offsets: np.ndarray, f16: bool = False):
    """Step 6: (rc, codes, scales, scale_row_offsets); rc is 0 or -6."""
    x = _c(xbits, np.uint16)
    off = _c(offsets, np.int32)
    total, K = x.shape
    E = off.size - 1
    codes = np.zeros((total, K // 2), np.uint8)
    scales = np.zeros(max(grouped_scale_bytes_bound(total, E, K), 1), np.uint8)
    sro = np.zeros(E + 1, np.int32)
    fn = lib().orc_quantize_grouped_f16 if f16 else lib().orc_quantize_grouped
    rc = fn(_p(x, _u16p), total, K, _p(off, _i32p), E, _p(codes, _u8p), _p(scales, _u8p),
            _p(sro, _i32p))
    return rc, codes, scales, sro


def f16_to_double_many(hbits: np.ndarray) -> np.ndarray:
    h = _c(hbits, np.uint16).ravel()
    out = np.empty(h.size, np.float64)
    lib().orc_f16_to_double_many(_p(h, _u16p), h.size, out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def e2m1_encode_f16_many(hbits: np.ndarray, s: int) -> np.ndarray:
    """Step 3 over many FP16 elements sharing scale exponent ``s``."""
    x = _c(hbits, np.uint16).ravel()
    out = np.empty(x.size, np.uint8)
    lib().orc_e2m1_encode_f16_many(_p(x, _u16p), x.size, int(s), _p(out, _u8p))
    return out


def quantize_f16(hbits: np.ndarray):
    """Steps 1-5 on FP16 input [M, K] (bit patterns): (codes, tiled scales)."""
    x = _c(hbits, np.uint16)
    M, K = x.shape
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros(scale_bytes(M, K), np.uint8)
    if M and K:
        lib().orc_quantize_f16(_p(x, _u16p), M, K, K, _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def quantize_flat_f16(hbits: np.ndarray):
    x = _c(hbits, np.uint16)
    M, K = x.shape
    codes = np.zeros((M, K // 2), np.uint8)
    flat = np.zeros((M, K // 32), np.uint8)
    if M and K:
        lib().orc_quantize_flat_f16(_p(x, _u16p), M, K, K, _p(codes, _u8p), _p(flat, _u8p))
    return codes, flat


def quantize_grouped_gather(xbits: np.ndarray, row_index: np.ndarray, offsets: np.ndarray,
                            f16: bool = False):
    """Step 6 on rows x[row_index]: (rc, codes, scales, scale_row_offsets);
    rc is 0, -6 (bad offsets) or -7 (an index out of range, zero row)."""
    x = _c(xbits, np.uint16)
    idx = _c(row_index, np.int32)
    off = _c(offsets, np.int32)
    n_src, K = x.shape
    total = idx.size
    E = off.size - 1
    codes = np.zeros((total, K // 2), np.uint8)
    scales = np.zeros(max(grouped_scale_bytes_bound(total, E, K), 1), np.uint8)
    sro = np.zeros(E + 1, np.int32)
    fn = lib().orc_quantize_grouped_gather_f16 if f16 else lib().orc_quantize_grouped_gather
    rc = fn(_p(x, _u16p), n_src, K, K, _p(idx, _i32p), total, _p(off, _i32p), E,
            _p(codes, _u8p), _p(scales, _u8p), _p(sro, _i32p))
    return rc, codes, scales, sro


def quantize_grouped_scatter(xbits: np.ndarray, dest_rows: np.ndarray, offsets: np.ndarray,
                             total_rows: int, codes=None, scales=None, f16: bool = False):
    """Step 6 with the dispatch as a scatter: route j of token t is row
    dest_rows[t, j] of the expert-sorted batch (-1: not dispatched).
    Returns (rc, codes, scales, scale_row_offsets); rc is 0, -6 (bad offsets)
    or -7 (an entry outside [-1, total_rows), skipped).  `codes` / `scales`,
    when given, are the buffers' previous contents (rows that no route
    targets keep them); by default they start zeroed."""
    x = _c(xbits, np.uint16)
    dst = _c(dest_rows, np.int32)
    off = _c(offsets, np.int32)
    T, K = x.shape
    top_k = dst.shape[1] if dst.ndim == 2 else 1
    assert dst.size == T * top_k
    E = off.size - 1
    codes = (np.zeros((total_rows, K // 2), np.uint8) if codes is None
             else np.array(codes, np.uint8, copy=True).reshape(total_rows, K // 2))
    nsb = max(grouped_scale_bytes_bound(total_rows, E, K), 1)
    scales = (np.zeros(nsb, np.uint8) if scales is None
              else np.array(scales, np.uint8, copy=True).ravel())
    assert scales.size >= grouped_scale_bytes_bound(total_rows, E, K)
    sro = np.zeros(E + 1, np.int32)
    fn = lib().orc_quantize_grouped_scatter_f16 if f16 else lib().orc_quantize_grouped_scatter
    rc = fn(_p(x, _u16p), T, K, K, _p(dst, _i32p), top_k, total_rows, _p(off, _i32p), E,
            _p(codes, _u8p), _p(scales, _u8p), _p(sro, _i32p))
    return rc, codes, scales, sro


def dequantize(codes: np.ndarray, tiled: np.ndarray, M: int, K: int) -> np.ndarray:
    """Step 7: BF16 bits [M, K] from codes and tiled scales."""
    c = _c(codes, np.uint8)
    t = _c(tiled, np.uint8).ravel()
    y = np.zeros((M, K), np.uint16)
    if M and K:
        lib().orc_dequantize(_p(c, _u8p), _p(t, _u8p), M, K, _p(y, _u16p))
    return y


def swap_halves(a: np.ndarray) -> np.ndarray:
    """Step 8 on bytes: a [E, 2N, row_bytes] uint8 -> rows (r + N) mod 2N."""
    x = _c(a, np.uint8)
    E, two_n, rb = x.shape
    out = np.zeros_like(x)
    lib().orc_swap_halves(_p(x, _u8p), _p(out, _u8p), E, two_n, rb)
    return out


def swap_bias_bf16(b: np.ndarray) -> np.ndarray:
    """Step 8 on a w13 bias [E, 2N] FP32 -> [b3, b1] as BF16 bits."""
    x = _c(b, np.float32)
    E, two_n = x.shape
    out = np.zeros(x.shape, np.uint16)
    lib().orc_swap_bias_bf16(_p(x, _f32p), _p(out, _u16p), E, two_n)
    return out


def cast_bf16(b: np.ndarray) -> np.ndarray:
    """FP32 -> BF16 bits (round to nearest, ties to even)."""
    x = _c(b, np.float32)
    out = np.zeros(x.shape, np.uint16)
    lib().orc_cast_bf16(_p(x, _f32p), _p(out, _u16p), x.size)
    return out


def swap_w13(codes, scales, w13_bias, E, two_n, K, scales_tiled, w2_bias=None):
    """Step 8: (codes_out, scales_out, w13_bias_bf16 | None, w2_bias_bf16 | None)."""
    c = _c(codes, np.uint8)
    s = _c(scales, np.uint8)
    b13 = _c(w13_bias, np.float32) if w13_bias is not None else None
    b2 = _c(w2_bias, np.float32) if w2_bias is not None else None
    c_out = np.zeros_like(c)
    s_out = np.zeros_like(s)
    b13_out = np.zeros(b13.shape, np.uint16) if b13 is not None else None
    b2_out = np.zeros(b2.shape, np.uint16) if b2 is not None else None
    lib().orc_swap_w13(_p(c, _u8p), _p(s, _u8p), _p(b13, _f32p), E, two_n, K,
                       int(scales_tiled), _p(c_out, _u8p), _p(s_out, _u8p),
                       _p(b13_out, _u16p), _p(b2, _f32p),
                       b2.size if b2 is not None else 0, _p(b2_out, _u16p))
    return c_out, s_out, b13_out, b2_out


def quantize_rows_into(xbits: np.ndarray, row0: int, row1: int, codes: np.ndarray,
                       scales: np.ndarray) -> None:
    """Step 1-5 over rows [row0, row1) of a full matrix, writing into the full
    outputs (row0 must be a multiple of 128).  Lets the CPU baseline spread the
    unchanged single-threaded routine over several host threads."""
    x = xbits
    M, K = x.shape
    assert row0 % 128 == 0 and x.flags.c_contiguous
    n_k_tiles = (K // 32 + 3) // 4
    xs = x[row0:row1]
    cs = codes[row0:row1]
    off = (row0 // 128) * n_k_tiles * 512
    lib().orc_quantize(xs.ctypes.data_as(_u16p), row1 - row0, K, K,
                       cs.ctypes.data_as(_u8p),
                       scales[off:].ctypes.data_as(_u8p))


# --------------------------------------------------- dispatch permutation
def moe_route(topk_ids: np.ndarray, num_experts: int):
    """The dispatch permutation from the router's expert ids [T, top_k]:
    (rc, offsets [E+1], dest_rows [T, top_k], row_index [rows]); rc 0 or -7."""
    ids = _c(topk_ids, np.int32)
    T = ids.shape[0]
    top_k = ids.shape[1] if ids.ndim == 2 else 1
    off = np.zeros(num_experts + 1, np.int32)
    dest = np.zeros((T, top_k), np.int32)
    rows = np.zeros(max(ids.size, 1), np.int32)
    rc = lib().orc_moe_route(_p(ids, _i32p), T, top_k, num_experts, _p(off, _i32p),
                             _p(dest, _i32p), _p(rows, _i32p))
    return rc, off, dest, rows[:int(off[-1])]


# ------------------------------------------- the same routines on host threads
# Full-size comparisons run the unchanged single-threaded routines above on
# independent parts of one problem, one host thread per part (the C calls
# release the GIL): 128-row bands of a dense matrix (every scale chunk belongs
# to one band), or contiguous ranges of experts of a grouped batch (each
# range is a grouped problem of its own whose padded scale rows start where
# the earlier experts' end).  The results equal the single calls byte for
# byte; the CPU tests check that on shapes with ragged and empty parts.
def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _run_parts(fn, parts):
    errors = []

    def run(args):
        try:
            fn(*args)
        except BaseException as e:  # re-raised on the calling thread
            errors.append(e)

    ths = [threading.Thread(target=run, args=(a,)) for a in parts]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    if errors:
        raise errors[0]


def _row_bands(M: int, threads: int):
    tiles = (M + 127) // 128
    per = max(1, (tiles + threads - 1) // threads)
    return [(t * 128, min(M, (t + per) * 128)) for t in range(0, tiles, per)]


def _expert_ranges(off: np.ndarray, threads: int):
    """Contiguous expert ranges [e0, e1) of about equal row counts."""
    E = off.size - 1
    cuts = np.searchsorted(off, np.linspace(0, off[-1], threads + 1)[1:-1], side="left")
    bounds = sorted({0, E, *[int(min(max(c, 1), E - 1)) for c in cuts]}) if E > 1 else [0, E]
    return [(a, b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]


def quantize_threads(xbits: np.ndarray, threads: int = 0):
    """quantize() of a whole matrix, the routine run on 128-row bands."""
    x = _c(xbits, np.uint16)
    M, K = x.shape
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros(scale_bytes(M, K), np.uint8)
    if M and K:
        _run_parts(lambda a, b: quantize_rows_into(x, a, b, codes, scales),
                   _row_bands(M, threads or host_threads()))
    return codes, scales


def dequantize_threads(codes: np.ndarray, tiled: np.ndarray, M: int, K: int,
                       threads: int = 0) -> np.ndarray:
    """dequantize() of a whole matrix, the routine run on 128-row bands."""
    c = _c(codes, np.uint8).reshape(M, K // 2)
    t = _c(tiled, np.uint8).ravel()
    y = np.zeros((M, K), np.uint16)
    chunk_row = (K // 32 + 3) // 4 * 512          # scale bytes of one 128-row band
    if M and K:
        def band(a, b):
            lib().orc_dequantize(_p(c[a:b], _u8p), _p(t[a // 128 * chunk_row:], _u8p), b - a, K,
                                 _p(y[a:b], _u16p))
        _run_parts(band, _row_bands(M, threads or host_threads()))
    return y


def _grouped_threads(single, call, xbits, offsets, cols, g, threads):
    x = _c(xbits, np.uint16)
    off32 = _c(offsets, np.int32)
    off = off32.astype(np.int64)
    total, K = x.shape
    E = off.size - 1
    if E < 1 or off[0] != 0 or off[-1] != total or np.any(np.diff(off) < 0):
        return single()                          # the single call reports the bad offsets
    pk = (cols + 3) // 4 * 4
    padded = np.concatenate([[0], np.cumsum((np.diff(off) + 127) // 128 * 128)])
    codes = np.zeros((total, K // 2), np.uint8)
    scales = np.zeros(max(int(padded[-1]) * pk, 1), np.uint8)
    sro = np.zeros(E + 1, np.int32)
    rcs = []

    def rng(e0, e1):
        a, b = int(off[e0]), int(off[e1])
        sub = (off32[e0:e1 + 1] - off32[e0]).astype(np.int32)
        sub_sro = np.zeros(e1 - e0 + 1, np.int32)
        rcs.append(call(x[a:b], b - a, K, sub, e1 - e0, None if g is None else g[e0:e1],
                        codes[a:b], scales[int(padded[e0]) * pk:], sub_sro))
        sro[e0:e1] = sub_sro[:-1] + int(padded[e0])

    _run_parts(rng, _expert_ranges(off, threads or host_threads()))
    sro[E] = int(padded[E])
    return (0 if all(r == 0 for r in rcs) else min(rcs)), codes, scales, sro


def quantize_grouped_threads(xbits: np.ndarray, offsets: np.ndarray, threads: int = 0):
    """quantize_grouped() with ranges of experts on host threads; the scale
    buffer ends at the last padded row (the bound's slack is not returned)."""
    def call(x, n, K, sub, E, _g, c, s, sro):
        return lib().orc_quantize_grouped(_p(x, _u16p), n, K, _p(sub, _i32p), E, _p(c, _u8p),
                                          _p(s, _u8p), _p(sro, _i32p))
    K = xbits.shape[1]
    return _grouped_threads(lambda: quantize_grouped(xbits, offsets), call, xbits, offsets,
                            K // 32, None, threads)


def nvfp4_quantize_grouped_threads(xbits: np.ndarray, offsets: np.ndarray, g: np.ndarray,
                                   threads: int = 0):
    """nvfp4_quantize_grouped() with ranges of experts on host threads; the
    scale buffer ends at the last padded row."""
    gs = _c(np.asarray(g, np.float32), np.float32)

    def call(x, n, K, sub, E, g_sub, c, s, sro):
        g_sub = np.ascontiguousarray(g_sub, np.float32)
        return lib().orc_nvfp4_quantize_grouped(_p(x, _u16p), n, K, _p(sub, _i32p), E,
                                                _p(g_sub, _f32p), _p(c, _u8p), _p(s, _u8p),
                                                _p(sro, _i32p))
    K = xbits.shape[1]
    return _grouped_threads(lambda: nvfp4_quantize_grouped(xbits, offsets, gs), call, xbits,
                            offsets, K // 16, gs, threads)


# ------------------------------------------------------------------ NVFP4
def e4m3_to_double(b: int) -> float:
    return lib().orc_e4m3_to_double(int(b))


def e4m3_from_double_many(d: np.ndarray) -> np.ndarray:
    """Nearest FP8 E4M3 (ties to even, saturating at 448) of float64 values."""
    x = _c(d, np.float64).ravel()
    out = np.empty(x.size, np.uint8)
    lib().orc_e4m3_from_double_many(x.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), x.size,
                                    _p(out, _u8p))
    return out


def nvfp4_scale_bytes(M: int, K: int) -> int:
    return int(lib().orc_nvfp4_scale_bytes(int(M), int(K)))


def nvfp4_quantize_flat(xbits: np.ndarray, g: float):
    """NVFP4 steps on BF16 [M, K]: (codes [M, K/2], flat E4M3 scales [M, K/16])."""
    x = _c(xbits, np.uint16)
    M, K = x.shape
    codes = np.zeros((M, K // 2), np.uint8)
    flat = np.zeros((M, K // 16), np.uint8)
    if M and K:
        lib().orc_nvfp4_quantize_flat(_p(x, _u16p), M, K, K, float(np.float32(g)),
                                      _p(codes, _u8p), _p(flat, _u8p))
    return codes, flat


def nvfp4_quantize(xbits: np.ndarray, g: float, f16: bool = False):
    """NVFP4 on BF16 [M, K]: (codes [M, K/2], 128x4-tiled E4M3 scales)."""
    x = _c(xbits, np.uint16)
    M, K = x.shape
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros(nvfp4_scale_bytes(M, K), np.uint8)
    if M and K:
        fn = lib().orc_nvfp4_quantize_f16 if f16 else lib().orc_nvfp4_quantize
        fn(_p(x, _u16p), M, K, K, float(np.float32(g)), _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def nvfp4_grouped_scale_bytes_bound(total_rows: int, E: int, K: int) -> int:
    tiles = (total_rows + 127 * E) // 128
    return tiles * 128 * ((K // 16 + 3) // 4 * 4)


def nvfp4_quantize_grouped(xbits: np.ndarray, offsets: np.ndarray, g: np.ndarray,
                           f16: bool = False):
    """NVFP4 experts quant: (rc, codes, scales, scale_row_offsets); rc 0 or -6.
    g: float32 [E] global scales, one per segment."""
    x = _c(xbits, np.uint16)
    off = _c(offsets, np.int32)
    gs = _c(np.asarray(g, np.float32), np.float32)
    total, K = x.shape
    E = off.size - 1
    assert gs.size == E
    codes = np.zeros((total, K // 2), np.uint8)
    scales = np.zeros(max(nvfp4_grouped_scale_bytes_bound(total, E, K), 1), np.uint8)
    sro = np.zeros(E + 1, np.int32)
    fn = lib().orc_nvfp4_quantize_grouped_f16 if f16 else lib().orc_nvfp4_quantize_grouped
    rc = fn(_p(x, _u16p), total, K, _p(off, _i32p), E, _p(gs, _f32p), _p(codes, _u8p),
            _p(scales, _u8p), _p(sro, _i32p))
    return rc, codes, scales, sro


def nvfp4_quantize_grouped_scatter(xbits: np.ndarray, dest_rows: np.ndarray, offsets: np.ndarray,
                                   total_rows: int, g: np.ndarray, codes=None, scales=None,
                                   f16: bool = False):
    """The NVFP4 experts quant with the dispatch as a scatter (route j of
    token t is row dest_rows[t, j], -1: not dispatched), segment e with global
    scale g[e].  Returns (rc, codes, scales, scale_row_offsets); rc 0, -6 or
    -7.  `codes` / `scales`, when given, are the buffers' previous contents
    (rows that no route targets keep them)."""
    x = _c(xbits, np.uint16)
    dst = _c(dest_rows, np.int32)
    off = _c(offsets, np.int32)
    gs = _c(np.asarray(g, np.float32), np.float32)
    T, K = x.shape
    top_k = dst.shape[1] if dst.ndim == 2 else 1
    assert dst.size == T * top_k
    E = off.size - 1
    assert gs.size == E
    codes = (np.zeros((total_rows, K // 2), np.uint8) if codes is None
             else np.array(codes, np.uint8, copy=True).reshape(total_rows, K // 2))
    nsb = max(nvfp4_grouped_scale_bytes_bound(total_rows, E, K), 1)
    scales = (np.zeros(nsb, np.uint8) if scales is None
              else np.array(scales, np.uint8, copy=True).ravel())
    assert scales.size >= nvfp4_grouped_scale_bytes_bound(total_rows, E, K)
    sro = np.zeros(E + 1, np.int32)
    fn = (lib().orc_nvfp4_quantize_grouped_scatter_f16 if f16
          else lib().orc_nvfp4_quantize_grouped_scatter)
    rc = fn(_p(x, _u16p), T, K, K, _p(dst, _i32p), top_k, total_rows, _p(off, _i32p), E,
            _p(gs, _f32p), _p(codes, _u8p), _p(scales, _u8p), _p(sro, _i32p))
    return rc, codes, scales, sro


def nvfp4_dequantize(codes: np.ndarray, tiled: np.ndarray, M: int, K: int, g: float) -> np.ndarray:
    c = _c(codes, np.uint8)
    t = _c(tiled, np.uint8).ravel()
    y = np.zeros((M, K), np.uint16)
    if M and K:
        lib().orc_nvfp4_dequantize(_p(c, _u8p), _p(t, _u8p), M, K, float(np.float32(g)), _p(y, _u16p))
    return y
