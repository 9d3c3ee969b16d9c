"""GB300 (sm_103a) MXFP4 block quantization.

Thin Python binding of ``libmxfp4_gb300.so`` (C ABI declared in
``include/mxfp4.h``).  The functions named ``mxfp4_*`` mirror the C entry
points one to one and only marshal arguments (device pointers, sizes, the
current CUDA stream); every step of the computation runs in the library's
CUDA kernels.  ``quantize``, ``quantize_grouped``, ``dequantize`` and
``swap_w13`` are conveniences that allocate the outputs with torch and call
the matching entry point.  PyTorch supplies device memory and streams only.

There is no CPU path: importing this package fails when the library has not
been built (``python mxfp4_block_quantization_gb300/_build.py``), and every
call rejects tensors that are not on a CUDA device.

Method sources (vLLM pull-request summary pages): PR #43557 "Fix the E8M0
scale computation in the MXFP4 MoE CUTLASS kernel" (scale rule, tiled scale
layout, experts quant); PR #51038 "[Bugfix][Quantization] Fix MXFP4
conversion for FlashInfer CUTLASS" ([w1; w3] -> [w3; w1] swap, BF16 bias);
PR #46915 "Fix the SM90 MXFP4 MoE test weight/scale interleave" (FP4 -> BF16
table read back).
"""
import contextlib
import ctypes
import functools
import os

import torch

__all__ = [
    "MXFP4Error", "LIB_PATH", "mxfp4_scale_bytes", "mxfp4_grouped_scale_bytes_bound",
    "mxfp4_quantize", "mxfp4_quantize_grouped", "mxfp4_dequantize", "mxfp4_swap_w13",
    "mxfp4_status_string", "mxfp4_version", "quantize", "quantize_grouped", "dequantize",
    "swap_w13", "MXFP4_OK", "MXFP4_EINVAL", "MXFP4_EALIGN", "MXFP4_ESHAPE", "MXFP4_EALIAS",
    "MXFP4_ECUDA", "MXFP4_EOFFSETS", "MXFP4_EINDEX", "mxfp4_quantize_grouped_gather",
    "quantize_grouped_gather", "mxfp4_quantize_grouped_scatter", "quantize_grouped_scatter",
    "mxfp4_scatter_workspace_bytes", "mxfp4_quantize_grouped_scatter_ws",
    "mxfp4_quantize_grouped_scatter_ws_f16",
    "MXFP4_SCATTER_MAX_TOP_K", "mxfp4_quantize_f16", "mxfp4_quantize_grouped_f16",
    "mxfp4_quantize_grouped_gather_f16", "mxfp4_quantize_grouped_scatter_f16",
    "mxfp4_gather_workspace_bytes", "mxfp4_quantize_grouped_gather_ws",
    "mxfp4_quantize_grouped_gather_ws_f16", "mxfp4_quantize_grouped_gather_noalloc",
    "MXFP4_ESCRATCH", "MXFP4_NOALLOC_SCRATCH_BYTES", "mxfp4_nvfp4_scale_bytes",
    "mxfp4_quantize_nvfp4", "mxfp4_dequantize_nvfp4", "quantize_nvfp4", "dequantize_nvfp4",
    "mxfp4_nvfp4_grouped_scale_bytes_bound", "mxfp4_quantize_nvfp4_grouped",
    "quantize_nvfp4_grouped", "mxfp4_quantize_nvfp4_f16", "mxfp4_quantize_nvfp4_grouped_f16",
    "mxfp4_quantize_nvfp4_grouped_scatter", "mxfp4_quantize_nvfp4_grouped_scatter_f16",
    "quantize_nvfp4_grouped_scatter", "mxfp4_nvfp4_scatter_workspace_bytes",
    "mxfp4_quantize_nvfp4_grouped_scatter_ws", "mxfp4_quantize_nvfp4_grouped_scatter_ws_f16",
    "MXFP4_ROUTE_MAX_EXPERTS", "mxfp4_route_workspace_bytes", "mxfp4_moe_route", "moe_route",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmxfp4_gb300.so")
# The bounds-checking build (same results; every global access checked and
# counted when out of range); see _load() and mxfp4_debug_bounds_violations.
DEBUG_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmxfp4_gb300_debug.so")

MXFP4_SCATTER_MAX_TOP_K = 32
MXFP4_ROUTE_MAX_EXPERTS = 8192
MXFP4_NOALLOC_SCRATCH_BYTES = 4 << 20
MXFP4_OK = 0
MXFP4_EINVAL = -1
MXFP4_EALIGN = -2
MXFP4_ESHAPE = -3
MXFP4_EALIAS = -4
MXFP4_ECUDA = -5
MXFP4_EOFFSETS = -6
MXFP4_EINDEX = -7
MXFP4_ESCRATCH = -8


class MXFP4Error(RuntimeError):
    """A non-zero status returned by the library."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {mxfp4_status_string(code)} ({code})")


def _load(path=LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with "
            "`python mxfp4_block_quantization_gb300/_build.py` (nvcc, sm_103a)")
    L = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    L.mxfp4_scale_bytes.restype = ctypes.c_size_t
    L.mxfp4_scale_bytes.argtypes = [i64, i64]
    L.mxfp4_grouped_scale_bytes_bound.restype = ctypes.c_size_t
    L.mxfp4_grouped_scale_bytes_bound.argtypes = [i64, i32, i64]
    L.mxfp4_quantize.restype = ctypes.c_int
    L.mxfp4_quantize.argtypes = [vp, i64, i64, i64, vp, vp, vp]
    L.mxfp4_quantize_f16.restype = ctypes.c_int
    L.mxfp4_quantize_f16.argtypes = [vp, i64, i64, i64, vp, vp, vp]
    L.mxfp4_quantize_grouped.restype = ctypes.c_int
    L.mxfp4_quantize_grouped.argtypes = [vp, i64, i64, vp, i32, vp, vp, vp, vp, vp]
    L.mxfp4_quantize_grouped_f16.restype = ctypes.c_int
    L.mxfp4_quantize_grouped_f16.argtypes = [vp, i64, i64, vp, i32, vp, vp, vp, vp, vp]
    L.mxfp4_quantize_grouped_gather_f16.restype = ctypes.c_int
    L.mxfp4_quantize_grouped_gather_f16.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, vp, vp,
                                                    vp, vp, vp]
    L.mxfp4_quantize_grouped_scatter_f16.restype = ctypes.c_int
    L.mxfp4_quantize_grouped_scatter_f16.argtypes = [vp, i64, i64, i64, vp, i32, i64, vp, i32,
                                                     vp, vp, vp, vp, vp]
    L.mxfp4_gather_workspace_bytes.restype = ctypes.c_size_t
    L.mxfp4_gather_workspace_bytes.argtypes = [i64, i64, i32, i64]
    for name in ("mxfp4_quantize_grouped_gather_ws", "mxfp4_quantize_grouped_gather_ws_f16"):
        getattr(L, name).restype = ctypes.c_int
        getattr(L, name).argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, vp, ctypes.c_size_t,
                                     vp, vp, vp, vp, vp]
    L.mxfp4_quantize_grouped_gather_noalloc.restype = ctypes.c_int
    L.mxfp4_quantize_grouped_gather_noalloc.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, vp,
                                                        vp, vp, vp, vp]
    L.mxfp4_quantize_grouped_gather.restype = ctypes.c_int
    L.mxfp4_quantize_grouped_gather.argtypes = [vp, i64, i64, i64, vp, i64, vp, i32, vp, vp, vp,
                                                vp, vp]
    L.mxfp4_quantize_grouped_scatter.restype = ctypes.c_int
    L.mxfp4_quantize_grouped_scatter.argtypes = [vp, i64, i64, i64, vp, i32, i64, vp, i32, vp,
                                                 vp, vp, vp, vp]
    L.mxfp4_scatter_workspace_bytes.restype = ctypes.c_size_t
    L.mxfp4_scatter_workspace_bytes.argtypes = [i64, i64, i32, i64]
    for name in ("mxfp4_quantize_grouped_scatter_ws", "mxfp4_quantize_grouped_scatter_ws_f16"):
        getattr(L, name).restype = ctypes.c_int
        getattr(L, name).argtypes = [vp, i64, i64, i64, vp, i32, i64, vp, i32, vp,
                                     ctypes.c_size_t, vp, vp, vp, vp, vp]
    L.mxfp4_dequantize.restype = ctypes.c_int
    L.mxfp4_dequantize.argtypes = [vp, vp, i64, i64, vp, vp]
    L.mxfp4_swap_w13.restype = ctypes.c_int
    L.mxfp4_swap_w13.argtypes = [vp, vp, vp, i32, i64, i64, i32, vp, vp, vp, vp, i64, vp, vp]
    L.mxfp4_nvfp4_scale_bytes.restype = ctypes.c_size_t
    L.mxfp4_nvfp4_scale_bytes.argtypes = [i64, i64]
    for name in ("mxfp4_quantize_nvfp4", "mxfp4_quantize_nvfp4_f16"):
        getattr(L, name).restype = ctypes.c_int
        getattr(L, name).argtypes = [vp, i64, i64, i64, vp, vp, vp, vp]
    L.mxfp4_nvfp4_grouped_scale_bytes_bound.restype = ctypes.c_size_t
    L.mxfp4_nvfp4_grouped_scale_bytes_bound.argtypes = [i64, i32, i64]
    for name in ("mxfp4_quantize_nvfp4_grouped", "mxfp4_quantize_nvfp4_grouped_f16"):
        getattr(L, name).restype = ctypes.c_int
        getattr(L, name).argtypes = [vp, i64, i64, vp, i32, vp, vp, vp, vp, vp, vp]
    for name in ("mxfp4_quantize_nvfp4_grouped_scatter",
                 "mxfp4_quantize_nvfp4_grouped_scatter_f16"):
        getattr(L, name).restype = ctypes.c_int
        getattr(L, name).argtypes = [vp, i64, i64, i64, vp, i32, i64, vp, i32, vp, vp, vp, vp, vp,
                                     vp]
    for name in ("mxfp4_quantize_nvfp4_grouped_scatter_ws",
                 "mxfp4_quantize_nvfp4_grouped_scatter_ws_f16"):
        getattr(L, name).restype = ctypes.c_int
        getattr(L, name).argtypes = [vp, i64, i64, i64, vp, i32, i64, vp, i32, vp, vp,
                                     ctypes.c_size_t, vp, vp, vp, vp, vp]
    L.mxfp4_nvfp4_scatter_workspace_bytes.restype = ctypes.c_size_t
    L.mxfp4_nvfp4_scatter_workspace_bytes.argtypes = [i64, i32, i64]
    L.mxfp4_dequantize_nvfp4.restype = ctypes.c_int
    L.mxfp4_dequantize_nvfp4.argtypes = [vp, vp, vp, i64, i64, vp, vp]
    L.mxfp4_route_workspace_bytes.restype = ctypes.c_size_t
    L.mxfp4_route_workspace_bytes.argtypes = [i64, i32, i32]
    L.mxfp4_moe_route.restype = ctypes.c_int
    L.mxfp4_moe_route.argtypes = [vp, i64, i32, i32, vp, ctypes.c_size_t, vp, vp, vp, vp, vp]
    L.mxfp4_status_string.restype = ctypes.c_char_p
    L.mxfp4_status_string.argtypes = [ctypes.c_int]
    L.mxfp4_version.restype = ctypes.c_int
    L.mxfp4_version.argtypes = []
    if hasattr(L, "mxfp4_debug_bounds_violations"):
        L.mxfp4_debug_bounds_violations.restype = ctypes.c_int64
        L.mxfp4_debug_bounds_violations.argtypes = []
    return L


_lib = _load()


# ------------------------------------------------------------------ helpers
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# The current stream's raw handle without building a torch Stream object (a
# measurable share of a call's host time); the public path where torch lacks it.
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device):
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _raw_current_stream is not None:
        return ctypes.c_void_p(_raw_current_stream(device.index))
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda(name, t, dtype=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (this library has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _need_bytes(name, t, nbytes):
    """``t`` (if given) must be contiguous and hold at least ``nbytes`` bytes:
    the library sees only its pointer and reads or writes the whole extent
    the call's sizes imply, so a short or strided buffer is refused here,
    before anything is launched.  ``nbytes`` <= 0 (sizes the library itself
    rejects) checks contiguity only."""
    if t is None:
        return
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name} holds {have} bytes; this call needs {nbytes}")


def _check(rc, where):
    if rc != MXFP4_OK:
        raise MXFP4Error(rc, where)


def _device_of(*tensors):
    """The one CUDA device all given tensors live on (the library launches on
    the current device, so every call switches to it)."""
    dev = None
    for t in tensors:
        if t is None:
            continue
        if dev is None:
            dev = t.device
        elif t.device != dev:
            devs = sorted({str(u.device) for u in tensors if u is not None})
            raise ValueError(f"all tensors must be on the same CUDA device, got {devs}")
    if dev is None:
        raise ValueError("no tensor given")
    return dev


def _switch(device):
    """The library launches on the current device: make ``device`` current for
    the call, or do nothing when it already is (the usual case, and a
    measurable share of a call's host time)."""
    if device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(device)


# ------------------------------------------------------- C entry points
@functools.lru_cache(maxsize=1024)
def mxfp4_scale_bytes(M: int, K: int) -> int:
    return int(_lib.mxfp4_scale_bytes(int(M), int(K)))


@functools.lru_cache(maxsize=1024)
def mxfp4_grouped_scale_bytes_bound(total_rows: int, E: int, K: int) -> int:
    return int(_lib.mxfp4_grouped_scale_bytes_bound(int(total_rows), int(E), int(K)))


def mxfp4_status_string(code: int) -> str:
    return _lib.mxfp4_status_string(int(code)).decode()


def mxfp4_version() -> int:
    return int(_lib.mxfp4_version())


def mxfp4_quantize(x, codes, scales, stream=None) -> None:
    """BF16 ``x`` [M, K] (row stride may exceed K) -> ``codes`` uint8 [M, K/2]
    and ``scales`` uint8 [mxfp4_scale_bytes(M, K)] (128x4 tiled)."""
    _need_cuda("x", x, torch.bfloat16)
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    M, K = x.shape
    _need_bytes("codes", codes, M * (K // 2))
    _need_bytes("scales", scales, mxfp4_scale_bytes(M, K))
    with _switch(_device_of(x, codes, scales)):
        _check(_lib.mxfp4_quantize(_ptr(x), M, K, x.stride(0), _ptr(codes), _ptr(scales),
                                   _stream(stream, x.device)), "mxfp4_quantize")


def mxfp4_quantize_f16(x, codes, scales, stream=None) -> None:
    """FP16 ``x`` [M, K] (row stride may exceed K) -> the same codes and tiled
    scales as mxfp4_quantize produces for BF16 input."""
    _need_cuda("x", x, torch.float16)
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    M, K = x.shape
    _need_bytes("codes", codes, M * (K // 2))
    _need_bytes("scales", scales, mxfp4_scale_bytes(M, K))
    with _switch(_device_of(x, codes, scales)):
        _check(_lib.mxfp4_quantize_f16(_ptr(x), M, K, x.stride(0), _ptr(codes), _ptr(scales),
                                       _stream(stream, x.device)), "mxfp4_quantize_f16")


def _need_grouped_outputs(expert_offsets, codes, scales, scale_row_offsets, status, rows, K,
                          scale_bound):
    """The buffers of a grouped call over ``rows`` expert-sorted rows."""
    E = expert_offsets.numel() - 1
    _need_bytes("expert_offsets", expert_offsets, 4 * (E + 1))
    _need_bytes("codes", codes, rows * (K // 2))
    _need_bytes("scales", scales, scale_bound(rows, E, K) if E >= 0 and rows >= 0 else 0)
    _need_bytes("scale_row_offsets", scale_row_offsets, 4 * (E + 1))
    _need_bytes("status", status, 4)


def _grouped(x, expert_offsets, codes, scales, scale_row_offsets, status, stream, f16):
    name = "mxfp4_quantize_grouped" + ("_f16" if f16 else "")
    _need_cuda("x", x, torch.float16 if f16 else torch.bfloat16)
    _need_cuda("expert_offsets", expert_offsets, torch.int32)
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    _need_cuda("scale_row_offsets", scale_row_offsets, torch.int32)
    _need_cuda("status", status, torch.int32)
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D tensor")
    total, K = x.shape
    E = expert_offsets.numel() - 1
    _need_grouped_outputs(expert_offsets, codes, scales, scale_row_offsets, status, total, K,
                          mxfp4_grouped_scale_bytes_bound)
    with _switch(_device_of(x, expert_offsets, codes, scales, scale_row_offsets, status)):
        _check(getattr(_lib, name)(_ptr(x), total, K, _ptr(expert_offsets), E, _ptr(codes),
                                   _ptr(scales), _ptr(scale_row_offsets), _ptr(status),
                                   _stream(stream, x.device)), name)


def mxfp4_quantize_grouped(x, expert_offsets, codes, scales, scale_row_offsets, status=None,
                           stream=None) -> None:
    """Per-expert quantize of contiguous BF16 rows ``x`` [total_rows, K]
    delimited by int32 ``expert_offsets`` [E+1] (device)."""
    _grouped(x, expert_offsets, codes, scales, scale_row_offsets, status, stream, False)


def mxfp4_quantize_grouped_f16(x, expert_offsets, codes, scales, scale_row_offsets, status=None,
                               stream=None) -> None:
    """mxfp4_quantize_grouped for FP16 ``x``."""
    _grouped(x, expert_offsets, codes, scales, scale_row_offsets, status, stream, True)


def _gather(x, row_index, expert_offsets, codes, scales, scale_row_offsets, status, stream, f16):
    name = "mxfp4_quantize_grouped_gather" + ("_f16" if f16 else "")
    _need_cuda("x", x, torch.float16 if f16 else torch.bfloat16)
    _need_cuda("row_index", row_index, torch.int32)
    _need_cuda("expert_offsets", expert_offsets, torch.int32)
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    _need_cuda("scale_row_offsets", scale_row_offsets, torch.int32)
    _need_cuda("status", status, torch.int32)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    if not row_index.is_contiguous():
        raise ValueError("row_index must be contiguous")
    n_src, K = x.shape
    E = expert_offsets.numel() - 1
    _need_grouped_outputs(expert_offsets, codes, scales, scale_row_offsets, status,
                          row_index.numel(), K, mxfp4_grouped_scale_bytes_bound)
    with _switch(_device_of(x, row_index, expert_offsets, codes, scales,
                                      scale_row_offsets, status)):
        _check(getattr(_lib, name)(
            _ptr(x), n_src, K, x.stride(0), _ptr(row_index), row_index.numel(),
            _ptr(expert_offsets), E, _ptr(codes), _ptr(scales), _ptr(scale_row_offsets),
            _ptr(status), _stream(stream, x.device)), name)


def mxfp4_quantize_grouped_gather(x, row_index, expert_offsets, codes, scales, scale_row_offsets,
                                  status=None, stream=None) -> None:
    """Grouped quantize of the rows ``x[row_index]`` (int32 device indices)
    without materialising the gathered BF16 matrix."""
    _gather(x, row_index, expert_offsets, codes, scales, scale_row_offsets, status, stream, False)


def mxfp4_quantize_grouped_gather_f16(x, row_index, expert_offsets, codes, scales,
                                      scale_row_offsets, status=None, stream=None) -> None:
    """mxfp4_quantize_grouped_gather for FP16 ``x``."""
    _gather(x, row_index, expert_offsets, codes, scales, scale_row_offsets, status, stream, True)


@functools.lru_cache(maxsize=1024)
def mxfp4_gather_workspace_bytes(num_src_rows: int, total_rows: int, E: int, K: int) -> int:
    return int(_lib.mxfp4_gather_workspace_bytes(int(num_src_rows), int(total_rows), int(E),
                                                 int(K)))


def _gather_ws(x, row_index, expert_offsets, workspace, codes, scales, scale_row_offsets, status,
               stream, f16):
    name = "mxfp4_quantize_grouped_gather_ws" + ("_f16" if f16 else "")
    _need_cuda("x", x, torch.float16 if f16 else torch.bfloat16)
    _need_cuda("row_index", row_index, torch.int32)
    _need_cuda("expert_offsets", expert_offsets, torch.int32)
    _need_cuda("workspace", workspace)
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    _need_cuda("scale_row_offsets", scale_row_offsets, torch.int32)
    _need_cuda("status", status, torch.int32)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    if not row_index.is_contiguous() or not workspace.is_contiguous():
        raise ValueError("row_index and workspace must be contiguous")
    n_src, K = x.shape
    E = expert_offsets.numel() - 1
    _need_grouped_outputs(expert_offsets, codes, scales, scale_row_offsets, status,
                          row_index.numel(), K, mxfp4_grouped_scale_bytes_bound)
    with _switch(_device_of(x, row_index, expert_offsets, workspace, codes, scales,
                                      scale_row_offsets, status)):
        _check(getattr(_lib, name)(
            _ptr(x), n_src, K, x.stride(0), _ptr(row_index), row_index.numel(),
            _ptr(expert_offsets), E, _ptr(workspace), workspace.numel() * workspace.element_size(),
            _ptr(codes), _ptr(scales), _ptr(scale_row_offsets), _ptr(status),
            _stream(stream, x.device)), name)


def mxfp4_quantize_grouped_gather_ws(x, row_index, expert_offsets, workspace, codes, scales,
                                     scale_row_offsets, status=None, stream=None) -> None:
    """mxfp4_quantize_grouped_gather through the scatter path: the inverse
    map is built in ``workspace`` (device, >= mxfp4_gather_workspace_bytes)."""
    _gather_ws(x, row_index, expert_offsets, workspace, codes, scales, scale_row_offsets, status,
               stream, False)


def mxfp4_quantize_grouped_gather_noalloc(x, row_index, expert_offsets, codes, scales,
                                          scale_row_offsets, status=None, stream=None) -> None:
    """mxfp4_quantize_grouped_gather_ws with the library's fixed scratch
    buffer (no workspace, no allocation); calls must not overlap on the GPU."""
    _need_cuda("x", x, torch.bfloat16)
    _need_cuda("row_index", row_index, torch.int32)
    _need_cuda("expert_offsets", expert_offsets, torch.int32)
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    _need_cuda("scale_row_offsets", scale_row_offsets, torch.int32)
    _need_cuda("status", status, torch.int32)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    if not row_index.is_contiguous():
        raise ValueError("row_index must be contiguous")
    n_src, K = x.shape
    E = expert_offsets.numel() - 1
    _need_grouped_outputs(expert_offsets, codes, scales, scale_row_offsets, status,
                          row_index.numel(), K, mxfp4_grouped_scale_bytes_bound)
    with _switch(_device_of(x, row_index, expert_offsets, codes, scales,
                                      scale_row_offsets, status)):
        _check(_lib.mxfp4_quantize_grouped_gather_noalloc(
            _ptr(x), n_src, K, x.stride(0), _ptr(row_index), row_index.numel(),
            _ptr(expert_offsets), E, _ptr(codes), _ptr(scales), _ptr(scale_row_offsets),
            _ptr(status), _stream(stream, x.device)), "mxfp4_quantize_grouped_gather_noalloc")


def mxfp4_quantize_grouped_gather_ws_f16(x, row_index, expert_offsets, workspace, codes, scales,
                                         scale_row_offsets, status=None, stream=None) -> None:
    """mxfp4_quantize_grouped_gather_ws for FP16 ``x``."""
    _gather_ws(x, row_index, expert_offsets, workspace, codes, scales, scale_row_offsets, status,
               stream, True)


def _scatter(x, dest_rows, expert_offsets, total_rows, codes, scales, scale_row_offsets, status,
             stream, f16, workspace=None):
    name = ("mxfp4_quantize_grouped_scatter" + ("_ws" if workspace is not None else "") +
            ("_f16" if f16 else ""))
    _need_cuda("x", x, torch.float16 if f16 else torch.bfloat16)
    _need_cuda("workspace", workspace, torch.uint8)
    _need_cuda("dest_rows", dest_rows, torch.int32)
    _need_cuda("expert_offsets", expert_offsets, torch.int32)
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    _need_cuda("scale_row_offsets", scale_row_offsets, torch.int32)
    _need_cuda("status", status, torch.int32)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    if dest_rows.dim() != 2 or dest_rows.shape[0] != x.shape[0] or not dest_rows.is_contiguous():
        raise ValueError("dest_rows must be a contiguous [num_tokens, top_k] tensor")
    T, K = x.shape
    E = expert_offsets.numel() - 1
    _need_grouped_outputs(expert_offsets, codes, scales, scale_row_offsets, status,
                          int(total_rows), K, mxfp4_grouped_scale_bytes_bound)
    _need_bytes("workspace", workspace, 0)
    ws = () if workspace is None else (_ptr(workspace), workspace.numel())
    with _switch(_device_of(x, dest_rows, expert_offsets, codes, scales,
                                      scale_row_offsets, status, workspace)):
        _check(getattr(_lib, name)(
            _ptr(x), T, K, x.stride(0), _ptr(dest_rows), dest_rows.shape[1], int(total_rows),
            _ptr(expert_offsets), E, *ws, _ptr(codes), _ptr(scales), _ptr(scale_row_offsets),
            _ptr(status), _stream(stream, x.device)), name)


def mxfp4_quantize_grouped_scatter(x, dest_rows, expert_offsets, total_rows: int, codes, scales,
                                   scale_row_offsets, status=None, stream=None) -> None:
    """Grouped quantize with the dispatch given token -> rows: route j of
    token t is row ``dest_rows[t, j]`` (int32 device [T, top_k], -1 = not
    dispatched) of the ``total_rows``-row expert-sorted batch.  Each token
    row is read and quantized once; rows no route targets are not written."""
    _scatter(x, dest_rows, expert_offsets, total_rows, codes, scales, scale_row_offsets, status,
             stream, False)


def mxfp4_quantize_grouped_scatter_f16(x, dest_rows, expert_offsets, total_rows: int, codes,
                                       scales, scale_row_offsets, status=None,
                                       stream=None) -> None:
    """mxfp4_quantize_grouped_scatter for FP16 ``x``."""
    _scatter(x, dest_rows, expert_offsets, total_rows, codes, scales, scale_row_offsets, status,
             stream, True)


@functools.lru_cache(maxsize=1024)
def mxfp4_scatter_workspace_bytes(num_tokens: int, total_rows: int, E: int, K: int) -> int:
    return int(_lib.mxfp4_scatter_workspace_bytes(int(num_tokens), int(total_rows), int(E),
                                                  int(K)))


def mxfp4_quantize_grouped_scatter_ws(x, dest_rows, expert_offsets, total_rows: int, workspace,
                                      codes, scales, scale_row_offsets, status=None,
                                      stream=None) -> None:
    """mxfp4_quantize_grouped_scatter with identical results, staging each
    token's scale words once in ``workspace`` (uint8 device, >=
    mxfp4_scatter_workspace_bytes) and writing the tiled scales whole."""
    _scatter(x, dest_rows, expert_offsets, total_rows, codes, scales, scale_row_offsets, status,
             stream, False, workspace)


def mxfp4_quantize_grouped_scatter_ws_f16(x, dest_rows, expert_offsets, total_rows: int,
                                          workspace, codes, scales, scale_row_offsets,
                                          status=None, stream=None) -> None:
    """mxfp4_quantize_grouped_scatter_ws for FP16 ``x``."""
    _scatter(x, dest_rows, expert_offsets, total_rows, codes, scales, scale_row_offsets, status,
             stream, True, workspace)


@functools.lru_cache(maxsize=1024)
def mxfp4_route_workspace_bytes(num_tokens: int, top_k: int, E: int) -> int:
    return int(_lib.mxfp4_route_workspace_bytes(int(num_tokens), int(top_k), int(E)))


def mxfp4_moe_route(topk_ids, num_experts: int, workspace, expert_offsets, dest_rows,
                    row_index=None, status=None, stream=None) -> None:
    """The dispatch permutation from the router's expert ids ``topk_ids``
    [num_tokens, top_k] (int32, -1: not dispatched): ``expert_offsets``
    [E+1], ``dest_rows`` [num_tokens, top_k] and, if given, ``row_index``
    [num_tokens * top_k] (the token of every row), in order of expert, then
    of entry.  ``workspace``: >= mxfp4_route_workspace_bytes bytes."""
    for name, t in (("topk_ids", topk_ids), ("expert_offsets", expert_offsets),
                    ("dest_rows", dest_rows), ("row_index", row_index), ("status", status)):
        _need_cuda(name, t, torch.int32)
    _need_cuda("workspace", workspace)
    for name, t in (("topk_ids", topk_ids), ("dest_rows", dest_rows)):
        if t.dim() != 2 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [num_tokens, top_k] tensor")
    if dest_rows.shape != topk_ids.shape:
        raise ValueError("dest_rows must have the shape of topk_ids")
    T, top_k = topk_ids.shape
    _need_bytes("workspace", workspace, 0)
    _need_bytes("expert_offsets", expert_offsets, 4 * (int(num_experts) + 1))
    _need_bytes("row_index", row_index, 4 * T * top_k)
    _need_bytes("status", status, 4)
    with _switch(_device_of(topk_ids, workspace, expert_offsets, dest_rows,
                                      row_index, status)):
        _check(_lib.mxfp4_moe_route(_ptr(topk_ids), T, top_k, int(num_experts), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _ptr(expert_offsets), _ptr(dest_rows), _ptr(row_index),
                                    _ptr(status), _stream(stream, topk_ids.device)),
               "mxfp4_moe_route")


def mxfp4_dequantize(codes, scales, M: int, K: int, y, stream=None) -> None:
    """``codes`` [M, K/2] + tiled ``scales`` -> BF16 ``y`` [M, K] (contiguous)."""
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    _need_cuda("y", y, torch.bfloat16)
    M, K = int(M), int(K)
    _need_bytes("codes", codes, M * (K // 2))
    _need_bytes("scales", scales, mxfp4_scale_bytes(M, K))
    _need_bytes("y", y, 2 * M * K)
    with _switch(_device_of(codes, scales, y)):
        _check(_lib.mxfp4_dequantize(_ptr(codes), _ptr(scales), int(M), int(K), _ptr(y),
                                     _stream(stream, y.device)), "mxfp4_dequantize")


def mxfp4_swap_w13(codes_in, scales_in, w13_bias_in, E: int, two_n: int, K: int,
                   scales_tiled: int, codes_out, scales_out, w13_bias_out=None,
                   w2_bias_in=None, w2_bias_out=None, stream=None) -> None:
    """[w1; w3] -> [w3; w1] of codes, scales (flat or tiled per expert) and
    FP32 biases (cast to BF16); the w2 bias is cast only."""
    for n, t, d in (("codes_in", codes_in, torch.uint8), ("scales_in", scales_in, torch.uint8),
                    ("codes_out", codes_out, torch.uint8), ("scales_out", scales_out, torch.uint8),
                    ("w13_bias_in", w13_bias_in, torch.float32),
                    ("w13_bias_out", w13_bias_out, torch.bfloat16),
                    ("w2_bias_in", w2_bias_in, torch.float32),
                    ("w2_bias_out", w2_bias_out, torch.bfloat16)):
        _need_cuda(n, t, d)
    dev = _device_of(codes_in, scales_in, codes_out, scales_out, w13_bias_in, w13_bias_out,
                     w2_bias_in, w2_bias_out)
    n2 = w2_bias_in.numel() if w2_bias_in is not None else 0
    E, two_n, K = int(E), int(two_n), int(K)
    code_bytes = E * two_n * (K // 2)
    scale_bytes = (E * mxfp4_scale_bytes(two_n, K) if scales_tiled else E * two_n * (K // 32))
    _need_bytes("codes_in", codes_in, code_bytes)
    _need_bytes("codes_out", codes_out, code_bytes)
    _need_bytes("scales_in", scales_in, scale_bytes)
    _need_bytes("scales_out", scales_out, scale_bytes)
    _need_bytes("w13_bias_in", w13_bias_in, 4 * E * two_n)
    if w13_bias_in is not None:
        _need_bytes("w13_bias_out", w13_bias_out, 2 * E * two_n)
    _need_bytes("w2_bias_in", w2_bias_in, 4 * n2)
    if w2_bias_in is not None:
        _need_bytes("w2_bias_out", w2_bias_out, 2 * n2)
    with _switch(dev):
        _check(_lib.mxfp4_swap_w13(_ptr(codes_in), _ptr(scales_in), _ptr(w13_bias_in), int(E),
                                   int(two_n), int(K), int(scales_tiled), _ptr(codes_out),
                                   _ptr(scales_out), _ptr(w13_bias_out), _ptr(w2_bias_in), n2,
                                   _ptr(w2_bias_out), _stream(stream, dev)), "mxfp4_swap_w13")


@functools.lru_cache(maxsize=1024)
def mxfp4_nvfp4_scale_bytes(M: int, K: int) -> int:
    return int(_lib.mxfp4_nvfp4_scale_bytes(int(M), int(K)))


def _nvfp4(x, global_scale, codes, scales, stream, f16) -> None:
    name = "mxfp4_quantize_nvfp4" + ("_f16" if f16 else "")
    _need_cuda("x", x, torch.float16 if f16 else torch.bfloat16)
    _need_cuda("global_scale", global_scale, torch.float32)
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    M, K = x.shape
    _need_bytes("global_scale", global_scale, 4)
    _need_bytes("codes", codes, M * (K // 2))
    _need_bytes("scales", scales, mxfp4_nvfp4_scale_bytes(M, K))
    with _switch(_device_of(x, global_scale, codes, scales)):
        _check(getattr(_lib, name)(_ptr(x), M, K, x.stride(0), _ptr(global_scale), _ptr(codes),
                                   _ptr(scales), _stream(stream, x.device)), name)


def mxfp4_quantize_nvfp4(x, global_scale, codes, scales, stream=None) -> None:
    """NVFP4: BF16 ``x`` [M, K] with float32 ``global_scale`` (1 element,
    device) -> codes [M, K/2] + tiled E4M3 scales."""
    _nvfp4(x, global_scale, codes, scales, stream, False)


def mxfp4_quantize_nvfp4_f16(x, global_scale, codes, scales, stream=None) -> None:
    """NVFP4 of FP16 ``x``; everything else as mxfp4_quantize_nvfp4."""
    _nvfp4(x, global_scale, codes, scales, stream, True)


@functools.lru_cache(maxsize=1024)
def mxfp4_nvfp4_grouped_scale_bytes_bound(total_rows: int, E: int, K: int) -> int:
    return int(_lib.mxfp4_nvfp4_grouped_scale_bytes_bound(int(total_rows), int(E), int(K)))


def _nvfp4_grouped(x, expert_offsets, global_scales, codes, scales, scale_row_offsets, status,
                   stream, f16) -> None:
    name = "mxfp4_quantize_nvfp4_grouped" + ("_f16" if f16 else "")
    _need_cuda("x", x, torch.float16 if f16 else torch.bfloat16)
    _need_cuda("expert_offsets", expert_offsets, torch.int32)
    _need_cuda("global_scales", global_scales, torch.float32)
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    _need_cuda("scale_row_offsets", scale_row_offsets, torch.int32)
    _need_cuda("status", status, torch.int32)
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D tensor")
    total, K = x.shape
    E = expert_offsets.numel() - 1
    if global_scales.numel() != E:
        raise ValueError("global_scales needs one entry per expert")
    _need_bytes("global_scales", global_scales, 4 * E)
    _need_grouped_outputs(expert_offsets, codes, scales, scale_row_offsets, status, total, K,
                          mxfp4_nvfp4_grouped_scale_bytes_bound)
    with _switch(_device_of(x, expert_offsets, global_scales, codes, scales,
                                      scale_row_offsets, status)):
        _check(getattr(_lib, name)(
            _ptr(x), total, K, _ptr(expert_offsets), E, _ptr(global_scales), _ptr(codes),
            _ptr(scales), _ptr(scale_row_offsets), _ptr(status), _stream(stream, x.device)), name)


def mxfp4_quantize_nvfp4_grouped(x, expert_offsets, global_scales, codes, scales,
                                 scale_row_offsets, status=None, stream=None) -> None:
    """NVFP4 experts quant: segment e of the contiguous BF16 ``x`` with global
    scale ``global_scales[e]`` (float32 device [E])."""
    _nvfp4_grouped(x, expert_offsets, global_scales, codes, scales, scale_row_offsets, status,
                   stream, False)


def mxfp4_quantize_nvfp4_grouped_f16(x, expert_offsets, global_scales, codes, scales,
                                     scale_row_offsets, status=None, stream=None) -> None:
    """NVFP4 experts quant of FP16 ``x``; everything else as the BF16 form."""
    _nvfp4_grouped(x, expert_offsets, global_scales, codes, scales, scale_row_offsets, status,
                   stream, True)


def _nvfp4_scatter(x, dest_rows, expert_offsets, total_rows, global_scales, codes, scales,
                   scale_row_offsets, status, stream, f16, workspace=None) -> None:
    name = ("mxfp4_quantize_nvfp4_grouped_scatter" + ("_ws" if workspace is not None else "") +
            ("_f16" if f16 else ""))
    _need_cuda("x", x, torch.float16 if f16 else torch.bfloat16)
    _need_cuda("workspace", workspace, torch.uint8)
    _need_cuda("dest_rows", dest_rows, torch.int32)
    _need_cuda("expert_offsets", expert_offsets, torch.int32)
    _need_cuda("global_scales", global_scales, torch.float32)
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    _need_cuda("scale_row_offsets", scale_row_offsets, torch.int32)
    _need_cuda("status", status, torch.int32)
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    if dest_rows.dim() != 2 or dest_rows.shape[0] != x.shape[0] or not dest_rows.is_contiguous():
        raise ValueError("dest_rows must be a contiguous [num_tokens, top_k] tensor")
    T, K = x.shape
    E = expert_offsets.numel() - 1
    if global_scales.numel() != E:
        raise ValueError("global_scales needs one entry per expert")
    _need_bytes("global_scales", global_scales, 4 * E)
    _need_grouped_outputs(expert_offsets, codes, scales, scale_row_offsets, status,
                          int(total_rows), K, mxfp4_nvfp4_grouped_scale_bytes_bound)
    _need_bytes("workspace", workspace, 0)
    ws = () if workspace is None else (_ptr(workspace), workspace.numel())
    with _switch(_device_of(x, dest_rows, expert_offsets, global_scales, codes, scales,
                                      scale_row_offsets, status, workspace)):
        _check(getattr(_lib, name)(
            _ptr(x), T, K, x.stride(0), _ptr(dest_rows), dest_rows.shape[1], int(total_rows),
            _ptr(expert_offsets), E, _ptr(global_scales), *ws, _ptr(codes), _ptr(scales),
            _ptr(scale_row_offsets), _ptr(status), _stream(stream, x.device)), name)


def mxfp4_quantize_nvfp4_grouped_scatter(x, dest_rows, expert_offsets, total_rows: int,
                                         global_scales, codes, scales, scale_row_offsets,
                                         status=None, stream=None) -> None:
    """NVFP4 experts quant with the dispatch as a scatter: route j of token t
    is row ``dest_rows[t, j]`` (-1 = not dispatched); segment e uses
    ``global_scales[e]``.  Rows no route targets are not written."""
    _nvfp4_scatter(x, dest_rows, expert_offsets, total_rows, global_scales, codes, scales,
                   scale_row_offsets, status, stream, False)


def mxfp4_quantize_nvfp4_grouped_scatter_f16(x, dest_rows, expert_offsets, total_rows: int,
                                             global_scales, codes, scales, scale_row_offsets,
                                             status=None, stream=None) -> None:
    """mxfp4_quantize_nvfp4_grouped_scatter for FP16 ``x``."""
    _nvfp4_scatter(x, dest_rows, expert_offsets, total_rows, global_scales, codes, scales,
                   scale_row_offsets, status, stream, True)


@functools.lru_cache(maxsize=1024)
def mxfp4_nvfp4_scatter_workspace_bytes(total_rows: int, E: int, K: int) -> int:
    return int(_lib.mxfp4_nvfp4_scatter_workspace_bytes(int(total_rows), int(E), int(K)))


def mxfp4_quantize_nvfp4_grouped_scatter_ws(x, dest_rows, expert_offsets, total_rows: int,
                                            global_scales, workspace, codes, scales,
                                            scale_row_offsets, status=None, stream=None) -> None:
    """mxfp4_quantize_nvfp4_grouped_scatter with identical results, each
    route's scale bytes staged by padded row in ``workspace`` (uint8 device, >=
    mxfp4_nvfp4_scatter_workspace_bytes) and tiled by a second kernel."""
    _nvfp4_scatter(x, dest_rows, expert_offsets, total_rows, global_scales, codes, scales,
                   scale_row_offsets, status, stream, False, workspace)


def mxfp4_quantize_nvfp4_grouped_scatter_ws_f16(x, dest_rows, expert_offsets, total_rows: int,
                                                global_scales, workspace, codes, scales,
                                                scale_row_offsets, status=None,
                                                stream=None) -> None:
    """mxfp4_quantize_nvfp4_grouped_scatter_ws for FP16 ``x``."""
    _nvfp4_scatter(x, dest_rows, expert_offsets, total_rows, global_scales, codes, scales,
                   scale_row_offsets, status, stream, True, workspace)


def mxfp4_dequantize_nvfp4(codes, scales, global_scale, M: int, K: int, y, stream=None) -> None:
    _need_cuda("codes", codes, torch.uint8)
    _need_cuda("scales", scales, torch.uint8)
    _need_cuda("global_scale", global_scale, torch.float32)
    _need_cuda("y", y, torch.bfloat16)
    M, K = int(M), int(K)
    _need_bytes("global_scale", global_scale, 4)
    _need_bytes("codes", codes, M * (K // 2))
    _need_bytes("scales", scales, mxfp4_nvfp4_scale_bytes(M, K))
    _need_bytes("y", y, 2 * M * K)
    with _switch(_device_of(codes, scales, global_scale, y)):
        _check(_lib.mxfp4_dequantize_nvfp4(_ptr(codes), _ptr(scales), _ptr(global_scale), int(M),
                                           int(K), _ptr(y), _stream(stream, y.device)),
               "mxfp4_dequantize_nvfp4")


# --------------------------------------------------- allocating wrappers
def quantize(x, stream=None):
    """BF16 or FP16 ``x`` [M, K] -> (codes uint8 [M, K/2], scales uint8 [scale_bytes])."""
    M, K = x.shape
    codes = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device)
    scales = torch.empty(mxfp4_scale_bytes(M, K), dtype=torch.uint8, device=x.device)
    if x.dtype == torch.float16:
        mxfp4_quantize_f16(x, codes, scales, stream)
    else:
        mxfp4_quantize(x, codes, scales, stream)
    return codes, scales


def quantize_grouped(x, expert_offsets, stream=None):
    """Returns (codes, scales, scale_row_offsets int32 [E+1], status int32 [1])."""
    total, K = x.shape
    E = expert_offsets.numel() - 1
    dev = x.device
    codes = torch.empty((total, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty(max(mxfp4_grouped_scale_bytes_bound(total, E, K), 16), dtype=torch.uint8,
                         device=dev)
    sro = torch.empty(E + 1, dtype=torch.int32, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    _grouped(x, expert_offsets, codes, scales, sro, status, stream, x.dtype == torch.float16)
    return codes, scales, sro, status


def quantize_grouped_gather(x, row_index, expert_offsets, stream=None, via_scatter=True):
    """Returns (codes, scales, scale_row_offsets, status) of x[row_index]
    (BF16 or FP16 x).  By default through the scatter path, with a workspace
    allocated here; via_scatter=False calls the entry point without a
    workspace, which borrows the tail of its codes output as one when that
    fits and otherwise runs the per-row gather kernel (same results)."""
    K = x.shape[1]
    total = row_index.numel()
    E = expert_offsets.numel() - 1
    dev = x.device
    f16 = x.dtype == torch.float16
    codes = torch.empty((total, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty(max(mxfp4_grouped_scale_bytes_bound(total, E, K), 16), dtype=torch.uint8,
                         device=dev)
    sro = torch.empty(E + 1, dtype=torch.int32, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    if via_scatter:
        ws = torch.empty(max(mxfp4_gather_workspace_bytes(x.shape[0], total, E, K), 16),
                         dtype=torch.uint8, device=dev)
        _gather_ws(x, row_index, expert_offsets, ws, codes, scales, sro, status, stream, f16)
    else:
        _gather(x, row_index, expert_offsets, codes, scales, sro, status, stream, f16)
    return codes, scales, sro, status


def quantize_grouped_scatter(x, dest_rows, expert_offsets, total_rows=None, stream=None,
                             staged=True):
    """Returns (codes, scales, scale_row_offsets, status) of the expert-sorted
    batch that ``dest_rows`` dispatches ``x`` into.  ``total_rows`` defaults
    to ``dest_rows.numel()`` (every route dispatched); rows that no route
    targets come back zero.  By default each token's scale words are staged
    in a workspace allocated here (same results); staged=False stores every
    route's scale words directly."""
    K = x.shape[1]
    total = dest_rows.numel() if total_rows is None else int(total_rows)
    E = expert_offsets.numel() - 1
    dev = x.device
    codes = torch.zeros((total, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.zeros(max(mxfp4_grouped_scale_bytes_bound(total, E, K), 16), dtype=torch.uint8,
                         device=dev)
    sro = torch.empty(E + 1, dtype=torch.int32, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    ws = None
    if staged:
        ws = torch.empty(max(mxfp4_scatter_workspace_bytes(x.shape[0], total, E, K), 16),
                         dtype=torch.uint8, device=dev)
    _scatter(x, dest_rows, expert_offsets, total, codes, scales, sro, status, stream,
             x.dtype == torch.float16, ws)
    return codes, scales, sro, status


def moe_route(topk_ids, num_experts: int, stream=None):
    """Returns (expert_offsets, dest_rows, row_index, status) of the router's
    expert ids ``topk_ids`` [num_tokens, top_k]: the inputs of the grouped,
    scatter and gather calls (row_index holds expert_offsets[-1] valid rows;
    the rest of it is not written)."""
    dev = topk_ids.device
    T, top_k = topk_ids.shape
    off = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    dest = torch.empty((T, top_k), dtype=torch.int32, device=dev)
    rows = torch.empty(max(T * top_k, 1), dtype=torch.int32, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    ws = torch.empty(max(mxfp4_route_workspace_bytes(T, top_k, num_experts), 16),
                     dtype=torch.uint8, device=dev)
    mxfp4_moe_route(topk_ids, num_experts, ws, off, dest, rows, status, stream)
    return off, dest, rows, status


def dequantize(codes, scales, M: int, K: int, stream=None):
    y = torch.empty((M, K), dtype=torch.bfloat16, device=codes.device)
    mxfp4_dequantize(codes, scales, M, K, y, stream)
    return y


def swap_w13(codes, scales, w13_bias=None, w2_bias=None, scales_tiled=True, stream=None):
    """codes uint8 [E, 2N, K/2]; scales tiled (E x scale_bytes(2N, K)) or flat
    [E, 2N, K/32].  Returns (codes, scales, w13_bias_bf16, w2_bias_bf16)."""
    E, two_n, half_k = codes.shape
    K = half_k * 2
    codes_out = torch.empty_like(codes)
    scales_out = torch.empty_like(scales)
    b13 = torch.empty(w13_bias.shape, dtype=torch.bfloat16, device=codes.device) \
        if w13_bias is not None else None
    b2 = torch.empty(w2_bias.shape, dtype=torch.bfloat16, device=codes.device) \
        if w2_bias is not None else None
    mxfp4_swap_w13(codes, scales, w13_bias, E, two_n, K, 1 if scales_tiled else 0, codes_out,
                   scales_out, b13, w2_bias, b2, stream)
    return codes_out, scales_out, b13, b2


def quantize_nvfp4(x, global_scale, stream=None):
    """Returns (codes uint8 [M, K/2], E4M3 scales uint8 [nvfp4_scale_bytes])
    of BF16 or FP16 ``x``."""
    M, K = x.shape
    codes = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device)
    scales = torch.empty(mxfp4_nvfp4_scale_bytes(M, K), dtype=torch.uint8, device=x.device)
    _nvfp4(x, global_scale, codes, scales, stream, x.dtype == torch.float16)
    return codes, scales


def quantize_nvfp4_grouped(x, expert_offsets, global_scales, stream=None):
    """Returns (codes, scales, scale_row_offsets, status) of the NVFP4 experts
    quant of the expert-sorted ``x`` (BF16 or FP16)."""
    total, K = x.shape
    E = expert_offsets.numel() - 1
    dev = x.device
    codes = torch.empty((total, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty(max(mxfp4_nvfp4_grouped_scale_bytes_bound(total, E, K), 16),
                         dtype=torch.uint8, device=dev)
    sro = torch.empty(E + 1, dtype=torch.int32, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    _nvfp4_grouped(x, expert_offsets, global_scales, codes, scales, sro, status, stream,
                   x.dtype == torch.float16)
    return codes, scales, sro, status


def quantize_nvfp4_grouped_scatter(x, dest_rows, expert_offsets, global_scales, total_rows=None,
                                   stream=None, staged=True):
    """Returns (codes, scales, scale_row_offsets, status) of the NVFP4 experts
    quant of the batch ``dest_rows`` dispatches ``x`` (BF16 or FP16) into;
    rows no route targets come back zero.  By default the scale bytes are
    staged in a workspace allocated here (same results); staged=False stores
    each route's scale words straight into the tiled layout."""
    K = x.shape[1]
    total = dest_rows.numel() if total_rows is None else int(total_rows)
    E = expert_offsets.numel() - 1
    dev = x.device
    codes = torch.zeros((total, K // 2), dtype=torch.uint8, device=dev)
    scales = torch.zeros(max(mxfp4_nvfp4_grouped_scale_bytes_bound(total, E, K), 16),
                         dtype=torch.uint8, device=dev)
    sro = torch.empty(E + 1, dtype=torch.int32, device=dev)
    status = torch.empty(1, dtype=torch.int32, device=dev)
    ws = None
    if staged:
        ws = torch.empty(max(mxfp4_nvfp4_scatter_workspace_bytes(total, E, K), 16),
                         dtype=torch.uint8, device=dev)
    _nvfp4_scatter(x, dest_rows, expert_offsets, total, global_scales, codes, scales, sro, status,
                   stream, x.dtype == torch.float16, ws)
    return codes, scales, sro, status


def dequantize_nvfp4(codes, scales, global_scale, M: int, K: int, stream=None):
    y = torch.empty((M, K), dtype=torch.bfloat16, device=codes.device)
    mxfp4_dequantize_nvfp4(codes, scales, global_scale, M, K, y, stream)
    return y
