"""The whole API through the bounds-checking build of the library
(-DMXFP4_DEBUG_BOUNDS): every global access of every kernel is checked
against the byte range of its buffer.  Every call must give the same bytes as
the normal build and no access may fall outside its buffer, on ragged,
strided, misaligned-to-32-byte, grouped (empty, skewed, invalid) and gather
cases."""
import contextlib

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    assert torch.cuda.is_available()
    import mxfp4_block_quantization_gb300 as mx
    dbg = mx._load(mx.DEBUG_LIB_PATH)
    assert dbg.mxfp4_debug_bounds_violations() == 0
    return mx, mx._lib, dbg


@contextlib.contextmanager
def using(mx, lib):
    saved = mx._lib
    mx._lib = lib
    try:
        yield
    finally:
        mx._lib = saved


def both(libs, fn):
    """Run fn() with the normal and with the bounds-checking library; return
    both results (tuples of tensors) moved to the host."""
    mx, rel, dbg = libs
    out = []
    for lib in (rel, dbg):
        with using(mx, lib):
            r = fn()
            torch.cuda.synchronize()
            out.append([t.cpu() if isinstance(t, torch.Tensor) else t for t in r])
    return out


def same(a, b):
    for x, y in zip(a, b):
        if isinstance(x, torch.Tensor):
            assert torch.equal(x.view(torch.uint8) if x.dtype != torch.uint8 else x,
                               y.view(torch.uint8) if y.dtype != torch.uint8 else y)
        else:
            assert x == y


def written(r, K):
    """A grouped result without the scale bytes past the padded total (the
    scale buffer is allocated at its upper bound; the slack is never
    written)."""
    codes, scales, sro, status = r
    return codes, scales[: int(sro[-1]) * ((K // 32 + 3) // 4) * 4], sro, status


def offset16(x):
    flat = torch.empty(x.numel() + 8, dtype=x.dtype, device=x.device)
    y = flat[8:].view(x.shape)
    y.copy_(x)
    return y


def test_everything_in_bounds(libs):
    mx, rel, dbg = libs
    cases = []
    for M, K in [(1, 32), (129, 160), (300, 2880), (128, 256)]:
        x = W.dense_activation(M + K, M, K, device="cuda")
        cases.append(lambda x=x: mx.quantize(x))
        cases.append(lambda x=x: mx.quantize(offset16(x)))
        cases.append(lambda x=x: mx.quantize(x.to(torch.float16)))
        cases.append(lambda x=x, M=M, K=K: (lambda c, s: (mx.dequantize(c, s, M, K),))(*mx.quantize(x)))
        g = torch.tensor([3.0], device="cuda")
        if K % 16 == 0:
            cases.append(lambda x=x, g=g: mx.quantize_nvfp4(x, g))
            cases.append(lambda x=x, g=g, M=M, K=K:
                         (lambda c, s: (mx.dequantize_nvfp4(c, s, g, M, K),))(*mx.quantize_nvfp4(x, g)))
    wide = W.dense_activation(5, 200, 1032, device="cuda")
    cases.append(lambda: mx.quantize(wide[:, :1024]))                  # row stride 16-byte multiple
    for K in (16, 48, 80):
        xs = W.normal_bf16((127, K), seed=K, device="cuda")
        g = torch.tensor([1.0], device="cuda")
        cases.append(lambda xs=xs, g=g: mx.quantize_nvfp4(xs, g))
    # dequantize into a 16-byte (not 32-byte) aligned output: the narrow kernel
    def narrow():
        x = W.dense_activation(9, 130, 256, device="cuda")
        c, s = mx.quantize(x)
        y = offset16(torch.empty((130, 256), dtype=torch.bfloat16, device="cuda"))
        mx.mxfp4_dequantize(c, s, 130, 256, y)
        return (y,)
    cases.append(narrow)
    # grouped / gather: normal, empty segments, skewed many experts, invalid
    gsmall = W.moe_grouped(seed=2, tokens=200, top_k=4, num_experts=12, K=288, device="cuda")
    cases.append(lambda: written(mx.quantize_grouped(gsmall.x, gsmall.offsets), 288))
    cases.append(lambda: written(mx.quantize_grouped_gather(gsmall.x_tokens, gsmall.row_index,
                                                            gsmall.offsets), 288))
    xe = W.small_matrix(3, 512, 256).cuda()
    off_e = torch.tensor([0, 0, 130, 130, 130, 512, 512], dtype=torch.int32, device="cuda")
    cases.append(lambda: written(mx.quantize_grouped(xe, off_e), 256))
    off_bad = torch.tensor([0, 300, 200, 512], dtype=torch.int32, device="cuda")
    cases.append(lambda: mx.quantize_grouped(xe, off_bad)[2:])
    idx_bad = torch.tensor([0, 5, 99, 7, -1, 3], dtype=torch.int32, device="cuda")
    off6 = torch.tensor([0, 2, 6], dtype=torch.int32, device="cuda")
    xt = W.small_matrix(4, 16, 64).cuda()
    cases.append(lambda: written(mx.quantize_grouped_gather(xt, idx_bad, off6), 64))
    rng = np.random.default_rng(12)
    sizes = np.minimum((rng.zipf(1.6, 1500) - 1) * 3, 600)
    sizes[rng.random(1500) < 0.3] = 0
    off_z = torch.from_numpy(np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)).cuda()
    xt2 = W.normal_bf16((300, 160), seed=14, device="cuda")
    ri = torch.from_numpy(rng.integers(0, 300, int(sizes.sum())).astype(np.int32)).cuda()
    cases.append(lambda: written(mx.quantize_grouped_gather(xt2, ri, off_z), 160))
    cases.append(lambda: written(mx.quantize_grouped_gather(xt2, ri, off_z, via_scatter=False), 160))
    cases.append(lambda: written(mx.quantize_grouped_gather(xt, idx_bad, off6, via_scatter=False),
                                 64))
    cases.append(lambda: written(mx.quantize_grouped(xt2.index_select(0, ri.long()), off_z), 160))
    # the gather without a workspace, large enough to borrow the tail of its codes output
    g4 = W.moe_grouped(seed=62, tokens=2048, top_k=8, num_experts=64, K=1024, device="cuda")
    ri4 = g4.row_index.clone()
    ri4[[3, ri4.numel() - 2]] = -1
    cases.append(lambda: written(mx.quantize_grouped_gather(g4.x_tokens, ri4, g4.offsets,
                                                            via_scatter=False), 1024))
    # scatter: all routes, dropped routes, bad entries, no tokens, strided
    cases.append(lambda: written(mx.quantize_grouped_scatter(gsmall.x_tokens, gsmall.dest_rows,
                                                             gsmall.offsets), 288))
    dsc = gsmall.dest_rows.clone()
    dsc[::3, 1] = -1
    dsc[5, 0] = 1 << 20
    cases.append(lambda: written(mx.quantize_grouped_scatter(gsmall.x_tokens, dsc,
                                                             gsmall.offsets), 288))
    cases.append(lambda: written(mx.quantize_grouped_scatter(gsmall.x_tokens, dsc, gsmall.offsets,
                                                             staged=False), 288))
    cases.append(lambda: written(mx.quantize_grouped_scatter(gsmall.x_tokens[:0], dsc[:0],
                                                             gsmall.offsets, dsc.numel()), 288))
    g3 = W.moe_grouped(seed=9, tokens=130, top_k=3, num_experts=5, K=1056, device="cuda")
    wide3 = torch.zeros((130, 1064), dtype=torch.bfloat16, device="cuda")
    wide3[:, :1056] = g3.x_tokens
    cases.append(lambda: written(mx.quantize_grouped_scatter(wide3[:, :1056], g3.dest_rows,
                                                             g3.offsets), 1056))
    # FP16 input through the scatter and gather forms
    cases.append(lambda: written(mx.quantize_grouped_scatter(g3.x_tokens.to(torch.float16),
                                                             g3.dest_rows, g3.offsets), 1056))
    cases.append(lambda: written(mx.quantize_grouped_gather(g3.x_tokens.to(torch.float16),
                                                            g3.row_index, g3.offsets), 1056))
    # NVFP4 experts quant with the dispatch as a scatter: dropped routes, bad entries
    gsc = torch.linspace(0.5, 40.0, 5, device="cuda")
    g3d = g3.dest_rows.clone()
    g3d[::4, 1] = -1
    g3d[2, 0] = 1 << 20
    cases.append(lambda: written(mx.quantize_nvfp4_grouped_scatter(g3.x_tokens, g3d, g3.offsets,
                                                                   gsc), 2 * 1056))  # K/16 cols
    cases.append(lambda: written(mx.quantize_nvfp4_grouped_scatter(g3.x_tokens, g3d, g3.offsets,
                                                                   gsc, staged=False), 2 * 1056))
    # the same with one global scale for every expert (routes share their bytes and codes)
    gs1 = torch.full((5,), 6.5, device="cuda")
    cases.append(lambda: written(mx.quantize_nvfp4_grouped_scatter(g3.x_tokens, g3d, g3.offsets,
                                                                   gs1), 2 * 1056))
    cases.append(lambda: written(mx.quantize_nvfp4_grouped_scatter(g3.x_tokens, g3d, g3.offsets,
                                                                   gs1, staged=False), 2 * 1056))
    # NVFP4 experts quant (K a multiple of 16 but not 32 included)
    gn = W.moe_grouped(seed=10, tokens=150, top_k=3, num_experts=7, K=80, device="cuda")
    gsn = torch.linspace(0.5, 40.0, 7, device="cuda")
    cases.append(lambda: mx.quantize_nvfp4_grouped(gn.x, gn.offsets, gsn)[:1] +
                 (mx.quantize_nvfp4_grouped(gn.x, gn.offsets, gsn)[2],))
    # swap: tiled with N % 128 == 0 and != 0, flat aligned and not
    for E, two_n, K, tiled in [(2, 256, 2048, True), (3, 200, 160, True), (3, 200, 160, False),
                               (2, 256, 64, False)]:
        codes = torch.randint(0, 256, (E, two_n, K // 2), dtype=torch.uint8, device="cuda")
        nsb = mx.mxfp4_scale_bytes(two_n, K) * E if tiled else E * two_n * (K // 32)
        scales = torch.randint(0, 256, (nsb,), dtype=torch.uint8, device="cuda")
        b13 = torch.randn(E, two_n, device="cuda")
        b2 = torch.randn(E, 33, device="cuda")
        cases.append(lambda c=codes, s=scales, b13=b13, b2=b2, t=tiled:
                     mx.swap_w13(c, s, b13, b2, scales_tiled=t))
    # the dispatch permutation from router ids: chunk boundaries, dropped and
    # invalid ids, many experts
    def route_case(ids, E):
        off, dest, rows, st = mx.moe_route(ids, E)
        return off, dest, rows[:int(off[-1])], st       # rows past the total are not written

    rng = np.random.default_rng(12)
    for T, k, E in [(1025, 1, 7), (300, 8, 384), (40, 2, 5000)]:
        ids = torch.from_numpy(rng.integers(-1, E + 1, (T, k)).astype(np.int32)).cuda()
        cases.append(lambda ids=ids, E=E: route_case(ids, E))
    for fn in cases:
        r, d = both(libs, fn)
        same(r, d)
    assert dbg.mxfp4_debug_bounds_violations() == 0
