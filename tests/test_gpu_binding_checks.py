"""The Python binding refuses, before anything is launched, every buffer the
library would read or write past its end (the C ABI sees pointers only, so
the sizes are checked where the tensors are known) and every strided one.
Each case calls a wrapper with one buffer a byte short, or a strided view of
the right size, and checks that it raises ValueError and that no output
changed (nothing ran); the same call with full buffers succeeds."""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

FILL = 0xA5


@pytest.fixture(scope="module")
def mx():
    assert torch.cuda.is_available()
    import mxfp4_block_quantization_gb300 as m
    return m


def _u8(n):
    return torch.full((n,), FILL, dtype=torch.uint8, device="cuda")


def _short(t):
    """A contiguous view one element short of ``t`` (one byte for uint8)."""
    return t.view(-1)[: t.numel() - 1]


def _strided(t):
    """A strided view with the element count of ``t`` (every second element of
    a buffer twice its size)."""
    big = torch.full((2 * t.numel(),), FILL, dtype=t.dtype, device="cuda")
    return big[::2]


def _expect_refused(call, outputs):
    before = [o.clone() for o in outputs]
    with pytest.raises(ValueError):
        call()
    torch.cuda.synchronize()
    for b, o in zip(before, outputs):
        assert torch.equal(b, o), "a refused call changed an output"


def test_dense_quantize_and_dequantize(mx):
    M, K = 256, 512
    x = W.dense_activation(1, M, K, device="cuda")
    codes = _u8(M * K // 2).view(M, K // 2)
    scales = _u8(mx.mxfp4_scale_bytes(M, K))
    _expect_refused(lambda: mx.mxfp4_quantize(x, _short(codes), scales), [scales])
    _expect_refused(lambda: mx.mxfp4_quantize(x, codes, _short(scales)), [codes])
    _expect_refused(lambda: mx.mxfp4_quantize(x, _strided(codes.view(-1)), scales), [scales])
    mx.mxfp4_quantize(x, codes, scales)
    y = torch.full((M, K), 7.0, dtype=torch.bfloat16, device="cuda")
    _expect_refused(lambda: mx.mxfp4_dequantize(codes, scales, M, K, _short(y)), [y])
    _expect_refused(lambda: mx.mxfp4_dequantize(_short(codes), scales, M, K, y), [y])
    _expect_refused(lambda: mx.mxfp4_dequantize(codes, _short(scales), M, K, y), [y])
    mx.mxfp4_dequantize(codes, scales, M, K, y)
    torch.cuda.synchronize()


def test_nvfp4_dense_quantize_and_dequantize(mx):
    M, K = 256, 512
    x = W.dense_activation(1, M, K, device="cuda")
    g = torch.tensor([448.0 * 6.0 / 4.0], device="cuda")
    codes = _u8(M * K // 2)
    scales = _u8(mx.mxfp4_nvfp4_scale_bytes(M, K))
    _expect_refused(lambda: mx.mxfp4_quantize_nvfp4(x, g, _short(codes), scales), [scales])
    _expect_refused(lambda: mx.mxfp4_quantize_nvfp4(x, g, codes, _short(scales)), [codes])
    _expect_refused(lambda: mx.mxfp4_quantize_nvfp4(x, g[:0], codes, scales), [codes, scales])
    mx.mxfp4_quantize_nvfp4(x, g, codes, scales)
    y = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    _expect_refused(lambda: mx.mxfp4_dequantize_nvfp4(codes, scales, g, M, K, _short(y)), [y])
    mx.mxfp4_dequantize_nvfp4(codes, scales, g, M, K, y)
    torch.cuda.synchronize()


def _grouped_case(mx, nvfp4=False):
    total, K, E = 300, 256, 3
    x = W.dense_activation(2, total, K, device="cuda")
    off = torch.tensor([0, 100, 100, total], dtype=torch.int32, device="cuda")
    bound = (mx.mxfp4_nvfp4_grouped_scale_bytes_bound if nvfp4
             else mx.mxfp4_grouped_scale_bytes_bound)(total, E, K)
    out = dict(codes=_u8(total * K // 2), scales=_u8(bound),
               sro=torch.zeros(E + 1, dtype=torch.int32, device="cuda"),
               status=torch.zeros(1, dtype=torch.int32, device="cuda"))
    return x, off, out


@pytest.mark.parametrize("short", ["codes", "scales", "sro", "status"])
def test_grouped_quantize(mx, short):
    x, off, out = _grouped_case(mx)
    args = dict(out)
    args[short] = _short(out[short])
    kept = [v for k, v in out.items() if k != short]
    _expect_refused(lambda: mx.mxfp4_quantize_grouped(x, off, args["codes"], args["scales"],
                                                       args["sro"], args["status"]), kept)
    mx.mxfp4_quantize_grouped(x, off, out["codes"], out["scales"], out["sro"], out["status"])
    torch.cuda.synchronize()


@pytest.mark.parametrize("short", ["codes", "scales", "sro"])
def test_nvfp4_grouped_quantize(mx, short):
    x, off, out = _grouped_case(mx, nvfp4=True)
    g = torch.full((3,), 448.0 * 6.0 / 4.0, device="cuda")
    args = dict(out)
    args[short] = _short(out[short])
    kept = [v for k, v in out.items() if k != short]
    _expect_refused(lambda: mx.mxfp4_quantize_nvfp4_grouped(
        x, off, g, args["codes"], args["scales"], args["sro"], args["status"]), kept)
    mx.mxfp4_quantize_nvfp4_grouped(x, off, g, out["codes"], out["scales"], out["sro"],
                                    out["status"])
    torch.cuda.synchronize()


def _moe(mx, nvfp4=False):
    g = W.moe_grouped(seed=5, tokens=64, top_k=4, num_experts=8, K=256, device="cuda")
    total = g.row_index.numel()
    E = g.num_experts
    K = g.x_tokens.shape[1]
    bound = (mx.mxfp4_nvfp4_grouped_scale_bytes_bound if nvfp4
             else mx.mxfp4_grouped_scale_bytes_bound)(total, E, K)
    out = dict(codes=_u8(total * K // 2), scales=_u8(bound),
               sro=torch.zeros(E + 1, dtype=torch.int32, device="cuda"),
               status=torch.zeros(1, dtype=torch.int32, device="cuda"))
    return g, total, out


@pytest.mark.parametrize("short", ["codes", "scales"])
def test_gather_forms(mx, short):
    g, total, out = _moe(mx)
    args = dict(out)
    args[short] = _short(out[short])
    kept = [v for k, v in out.items() if k != short]
    ws = _u8(max(mx.mxfp4_gather_workspace_bytes(g.x_tokens.shape[0], total, g.num_experts,
                                                 g.x_tokens.shape[1]), 16))
    calls = [
        lambda: mx.mxfp4_quantize_grouped_gather(g.x_tokens, g.row_index, g.offsets,
                                                 args["codes"], args["scales"], args["sro"],
                                                 args["status"]),
        lambda: mx.mxfp4_quantize_grouped_gather_ws(g.x_tokens, g.row_index, g.offsets, ws,
                                                    args["codes"], args["scales"], args["sro"],
                                                    args["status"]),
        lambda: mx.mxfp4_quantize_grouped_gather_noalloc(g.x_tokens, g.row_index, g.offsets,
                                                         args["codes"], args["scales"],
                                                         args["sro"], args["status"]),
    ]
    for call in calls:
        _expect_refused(call, kept)
    mx.mxfp4_quantize_grouped_gather(g.x_tokens, g.row_index, g.offsets, out["codes"],
                                     out["scales"], out["sro"], out["status"])
    torch.cuda.synchronize()


@pytest.mark.parametrize("short", ["codes", "scales", "sro"])
def test_scatter_forms(mx, short):
    g, total, out = _moe(mx)
    args = dict(out)
    args[short] = _short(out[short])
    kept = [v for k, v in out.items() if k != short]
    T, K = g.x_tokens.shape
    ws = _u8(max(mx.mxfp4_scatter_workspace_bytes(T, total, g.num_experts, K), 16))
    _expect_refused(lambda: mx.mxfp4_quantize_grouped_scatter(
        g.x_tokens, g.dest_rows, g.offsets, total, args["codes"], args["scales"], args["sro"],
        args["status"]), kept)
    _expect_refused(lambda: mx.mxfp4_quantize_grouped_scatter_ws(
        g.x_tokens, g.dest_rows, g.offsets, total, ws, args["codes"], args["scales"],
        args["sro"], args["status"]), kept)
    mx.mxfp4_quantize_grouped_scatter_ws(g.x_tokens, g.dest_rows, g.offsets, total, ws,
                                         out["codes"], out["scales"], out["sro"], out["status"])
    torch.cuda.synchronize()


@pytest.mark.parametrize("short", ["codes", "scales", "global_scales"])
def test_nvfp4_scatter_forms(mx, short):
    g, total, out = _moe(mx, nvfp4=True)
    gs = torch.full((g.num_experts,), 448.0 * 6.0 / 4.0, device="cuda")
    args = dict(out, global_scales=gs)
    if short == "global_scales":
        args[short] = _strided(gs)
    else:
        args[short] = _short(out[short])
    kept = [v for k, v in out.items() if k != short]
    T, K = g.x_tokens.shape
    ws = _u8(max(mx.mxfp4_nvfp4_scatter_workspace_bytes(total, g.num_experts, K), 16))
    _expect_refused(lambda: mx.mxfp4_quantize_nvfp4_grouped_scatter(
        g.x_tokens, g.dest_rows, g.offsets, total, args["global_scales"], args["codes"],
        args["scales"], args["sro"], args["status"]), kept)
    _expect_refused(lambda: mx.mxfp4_quantize_nvfp4_grouped_scatter_ws(
        g.x_tokens, g.dest_rows, g.offsets, total, args["global_scales"], ws, args["codes"],
        args["scales"], args["sro"], args["status"]), kept)
    mx.mxfp4_quantize_nvfp4_grouped_scatter_ws(g.x_tokens, g.dest_rows, g.offsets, total, gs, ws,
                                               out["codes"], out["scales"], out["sro"],
                                               out["status"])
    torch.cuda.synchronize()


def test_route(mx):
    T, top_k, E = 64, 4, 8
    ids = torch.randint(0, E, (T, top_k), generator=torch.Generator().manual_seed(5),
                        dtype=torch.int32).cuda()
    ws = _u8(max(mx.mxfp4_route_workspace_bytes(T, top_k, E), 16))
    off = torch.full((E + 1,), -5, dtype=torch.int32, device="cuda")
    dest = torch.full((T, top_k), -5, dtype=torch.int32, device="cuda")
    rows = torch.full((T * top_k,), -5, dtype=torch.int32, device="cuda")
    _expect_refused(lambda: mx.mxfp4_moe_route(ids, E, ws, _short(off), dest, rows),
                    [dest, rows])
    _expect_refused(lambda: mx.mxfp4_moe_route(ids, E, ws, off, dest, _short(rows)),
                    [off, dest])
    mx.mxfp4_moe_route(ids, E, ws, off, dest, rows)
    torch.cuda.synchronize()
    assert int(off[-1]) == T * top_k


@pytest.mark.parametrize("tiled", [0, 1])
def test_swap_w13(mx, tiled):
    E, two_n, K = 2, 64, 128
    cb = E * two_n * K // 2
    sb = E * mx.mxfp4_scale_bytes(two_n, K) if tiled else E * two_n * (K // 32)
    codes_in, codes_out = _u8(cb), _u8(cb)
    scales_in, scales_out = _u8(sb), _u8(sb)
    b_in = torch.zeros(E * two_n, dtype=torch.float32, device="cuda")
    b_out = torch.zeros(E * two_n, dtype=torch.bfloat16, device="cuda")
    _expect_refused(lambda: mx.mxfp4_swap_w13(codes_in, scales_in, b_in, E, two_n, K, tiled,
                                              _short(codes_out), scales_out, b_out),
                    [scales_out, b_out])
    _expect_refused(lambda: mx.mxfp4_swap_w13(codes_in, scales_in, b_in, E, two_n, K, tiled,
                                              codes_out, _short(scales_out), b_out),
                    [codes_out, b_out])
    _expect_refused(lambda: mx.mxfp4_swap_w13(codes_in, scales_in, b_in, E, two_n, K, tiled,
                                              codes_out, scales_out, _short(b_out)),
                    [codes_out, scales_out])
    mx.mxfp4_swap_w13(codes_in, scales_in, b_in, E, two_n, K, tiled, codes_out, scales_out,
                      b_out)
    torch.cuda.synchronize()
