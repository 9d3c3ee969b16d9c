"""The gather entry point that allocates nothing (its scratch is a fixed
device buffer inside the library), through the C ABI: two calls in a row,
each compared byte for byte with the per-row gather entry point on the same
inputs.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _outputs(mx, total, K, E):
    codes = torch.full((total, K // 2), 0xA5, dtype=torch.uint8, device="cuda")
    scales = torch.full((mx.mxfp4_grouped_scale_bytes_bound(total, E, K),), 0xA5,
                        dtype=torch.uint8, device="cuda")
    sro = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    st = torch.empty(1, dtype=torch.int32, device="cuda")
    return codes, scales, sro, st


def _call(fn, x, idx, off, out):
    vp = ctypes.c_void_p
    codes, scales, sro, st = out
    s = vp(torch.cuda.current_stream().cuda_stream)
    return fn(vp(x.data_ptr()), x.shape[0], x.shape[1], x.stride(0), vp(idx.data_ptr()),
              idx.numel(), vp(off.data_ptr()), off.numel() - 1, vp(codes.data_ptr()),
              vp(scales.data_ptr()), vp(sro.data_ptr()), vp(st.data_ptr()), s)


def test_noalloc_gather_two_calls_match_the_gather_entry_point():
    assert torch.cuda.is_available()
    import mxfp4_block_quantization_gb300 as mx
    L = mx._lib
    # the third case's staged scale words do not fit the scratch: the call then
    # stores the tiled scale words from the scatter kernel itself.  The last
    # case repeats the first, small staged one after that large call has
    # left its contents in the shared array, so what must start at zero is
    # shown to be cleared by the call itself.
    for seed, tokens, top_k, E, K in ((21, 300, 4, 11, 288), (22, 2048, 8, 64, 1024),
                                      (23, 16384, 4, 32, 7168), (21, 300, 4, 11, 288)):
        g = W.moe_grouped(seed=seed, tokens=tokens, top_k=top_k, num_experts=E, K=K,
                          device="cuda")
        total = g.row_index.numel()
        scratch = mx.MXFP4_NOALLOC_SCRATCH_BYTES
        assert (mx.mxfp4_gather_workspace_bytes(tokens, total, E, K) <= scratch) == (tokens < 16384)
        assert mx.mxfp4_gather_workspace_bytes(tokens, total, E, 0) <= scratch
        ref = _outputs(mx, total, K, E)
        assert _call(L.mxfp4_quantize_grouped_gather, g.x_tokens, g.row_index, g.offsets,
                     ref) == mx.MXFP4_OK
        got = _outputs(mx, total, K, E)
        assert _call(L.mxfp4_quantize_grouped_gather_noalloc, g.x_tokens, g.row_index,
                     g.offsets, got) == mx.MXFP4_OK
        torch.cuda.synchronize()
        assert int(got[3].item()) == int(ref[3].item()) == mx.MXFP4_OK
        for a, b in zip(got, ref):
            assert torch.equal(a, b), seed
        # out-of-range indices: zero rows and MXFP4_EINDEX in both modes
        bad = g.row_index.clone()
        bad[::97] = -1
        bad[5] = tokens
        ref = _outputs(mx, total, K, E)
        _call(L.mxfp4_quantize_grouped_gather, g.x_tokens, bad, g.offsets, ref)
        got = _outputs(mx, total, K, E)
        assert _call(L.mxfp4_quantize_grouped_gather_noalloc, g.x_tokens, bad, g.offsets,
                     got) == mx.MXFP4_OK
        torch.cuda.synchronize()
        assert int(got[3].item()) == int(ref[3].item()) == mx.MXFP4_EINDEX
        for a, b in zip(got, ref):
            assert torch.equal(a, b), seed


def test_noalloc_gather_python_wrapper_matches_the_c_call():
    """The binding's wrapper (device guard, dtype checks, status handling)
    gives the bytes of the raw C call, and raises on a refused call."""
    assert torch.cuda.is_available()
    import mxfp4_block_quantization_gb300 as mx
    g = W.moe_grouped(seed=24, tokens=512, top_k=4, num_experts=9, K=320, device="cuda")
    total, E, K = g.row_index.numel(), 9, 320
    ref = _outputs(mx, total, K, E)
    assert _call(mx._lib.mxfp4_quantize_grouped_gather_noalloc, g.x_tokens, g.row_index,
                 g.offsets, ref) == mx.MXFP4_OK
    got = _outputs(mx, total, K, E)
    mx.mxfp4_quantize_grouped_gather_noalloc(g.x_tokens, g.row_index, g.offsets, *got)
    torch.cuda.synchronize()
    assert int(got[3].item()) == mx.MXFP4_OK
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    with pytest.raises(mx.MXFP4Error):
        mx.mxfp4_quantize_grouped_gather_noalloc(g.x_tokens[:, :K - 16], g.row_index, g.offsets,
                                                 *got)
    with pytest.raises(ValueError):
        mx.mxfp4_quantize_grouped_gather_noalloc(g.x_tokens.float(), g.row_index, g.offsets,
                                                 *got)
