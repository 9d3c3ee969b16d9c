"""Pins of the oracle's whole-matrix quantize (steps 1-5), grouped quantize
(step 6) and dequantize (step 7): properties that hold for the method at any
size, checked on seeded inputs of the workloads' distributions."""
import numpy as np
import pytest
import torch

from mxfp4_block_quantization_gb300 import workloads as W


def _nibbles(codes):
    M, half = codes.shape
    n = np.zeros((M, half * 2), np.uint8)
    n[:, 0::2] = codes & 0xF
    n[:, 1::2] = codes >> 4
    return n


def test_quantize_equals_blockwise_steps(orc):
    """quantize == per-block absmax -> scale -> element codes -> tile."""
    x = W.bf16_bits(W.small_matrix(0, 128, 256))
    codes, tiled = orc.quantize(x)
    flat = orc.untile(tiled, 128, 8)
    nib = _nibbles(codes)
    xv = (x.astype(np.uint32) << 16).view(np.float32)
    for r in range(0, 128, 7):
        for b in range(8):
            blk = x[r, b * 32:(b + 1) * 32]
            vmax = np.abs(xv[r, b * 32:(b + 1) * 32]).max()
            s = orc.e8m0_scale(vmax)
            assert flat[r, b] == s
            assert np.array_equal(nib[r, b * 32:(b + 1) * 32], orc.e2m1_encode_many(blk, s))


def test_requantize_of_dequantized_is_identity(orc):
    """Every block the quantizer emits has s >= 1 with max code magnitude 4 or
    6 (the block max lands in [3.5, 7) and rounds to 4 or 6), or s == 0 with
    zero codes; decoding and quantizing again reproduces the same scale and
    codes exactly."""
    for x in (W.bf16_bits(W.edge_cases(4, 256, 2880)),
              W.bf16_bits(W.dense_activation(1, 256, 1024))):
        M, K = x.shape
        codes, tiled = orc.quantize(x)
        y = orc.dequantize(codes, tiled, M, K)
        codes2, tiled2 = orc.quantize(y)
        assert np.array_equal(codes, codes2)
        assert np.array_equal(tiled, tiled2)


def test_dequant_error_bound(orc):
    """|dequant(quant(x)) - x| <= half a code step of the block, except the
    saturated block max (|y| in (6, 7)) whose error is below 1 step of 2."""
    x = W.bf16_bits(W.dense_activation(1, 128, 2048))
    M, K = x.shape
    codes, tiled = orc.quantize(x)
    y = orc.dequantize(codes, tiled, M, K)
    xv = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    yv = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    flat = orc.untile(tiled, M, K // 32).astype(np.int64)
    scale = np.ldexp(1.0, np.repeat(flat, 32, axis=1) - 127)
    err = np.abs(yv - xv) / scale
    assert err.max() <= 1.0
    t = np.abs(xv) / scale
    inner = t <= 6.0
    # spacing of E2M1 is 0.5 below 2, 1 in [2, 4], 2 in [4, 6]
    half_step = np.where(t < 2, 0.25, np.where(t < 4, 0.5, 1.0))
    assert np.all(err[inner] <= half_step[inner])


def test_edge_case_inputs_hit_special_blocks(orc):
    x = W.bf16_bits(W.edge_cases(4))
    codes, tiled = orc.quantize(x)
    flat = orc.untile(tiled, 1000, 90)
    n_zero_scale = int((flat == 0).sum())
    assert n_zero_scale >= 1800            # 1% zero + 1% subnormal blocks
    nib = _nibbles(codes).reshape(1000, 90, 32)
    assert not nib[flat == 0].any()


def test_grouped_equals_per_segment(orc):
    g = W.moe_grouped(seed=2, tokens=96, top_k=4, num_experts=12, K=288)
    x = W.bf16_bits(g.x)
    off = g.offsets.numpy()
    rc, codes, scales, sro = orc.quantize_grouped(x, off)
    assert rc == 0
    K = x.shape[1]
    pk = (K // 32 + 3) // 4 * 4
    P = 0
    for e in range(len(off) - 1):
        a, b = int(off[e]), int(off[e + 1])
        assert sro[e] == P
        c_e, s_e = orc.quantize(x[a:b])
        assert np.array_equal(codes[a:b], c_e)
        assert np.array_equal(scales[P * pk:P * pk + s_e.size], s_e)
        P += (b - a + 127) // 128 * 128
    assert sro[-1] == P
    assert not scales[P * pk:].any()


def test_grouped_uniform_equals_dense(orc):
    x = W.bf16_bits(W.small_matrix(9, 512, 256))
    off = np.array([0, 128, 256, 384, 512], np.int32)
    rc, codes, scales, sro = orc.quantize_grouped(x, off)
    c_d, s_d = orc.quantize(x)
    assert rc == 0 and np.array_equal(codes, c_d)
    assert np.array_equal(scales[: s_d.size], s_d)
    assert list(sro) == [0, 128, 256, 384, 512]


def test_grouped_empty_segments(orc):
    x = W.bf16_bits(W.small_matrix(3, 200, 64))
    off = np.array([0, 0, 130, 130, 130, 200, 200], np.int32)
    rc, codes, scales, sro = orc.quantize_grouped(x, off)
    assert rc == 0
    assert list(sro) == [0, 0, 256, 256, 256, 384, 384]


@pytest.mark.parametrize("off", [[1, 10, 20], [0, 12, 8, 20], [0, 10, 19], [0, 10, 21]])
def test_grouped_bad_offsets(orc, off):
    x = W.bf16_bits(W.small_matrix(3, 20, 64))
    rc, codes, scales, sro = orc.quantize_grouped(x, np.array(off, np.int32))
    assert rc == -6
    assert list(sro) == [-1] * len(off)
    assert not codes.any() and not scales.any()


def test_grouped_gather_equals_grouped_of_gathered(orc):
    """The fused dispatch gather: quantizing rows x[row_index] directly equals
    the grouped quantize of the explicitly gathered matrix (numpy indexing)."""
    g = W.moe_grouped(seed=2, tokens=80, top_k=3, num_experts=7, K=192)
    xt = W.bf16_bits(g.x_tokens)
    idx = g.token_of_row.numpy().astype(np.int32)
    off = g.offsets.numpy()
    rc, c, s, sro = orc.quantize_grouped_gather(xt, idx, off)
    rc2, c2, s2, sro2 = orc.quantize_grouped(xt[idx], off)
    assert rc == 0 and rc2 == 0
    assert np.array_equal(c, c2) and np.array_equal(s, s2) and np.array_equal(sro, sro2)
    assert np.array_equal(xt[idx], W.bf16_bits(g.x))


def test_grouped_gather_bad_index_zero_row(orc):
    xt = W.bf16_bits(W.small_matrix(3, 16, 64))
    idx = np.array([0, 5, 99, 7, -1, 3], np.int32)
    off = np.array([0, 2, 6], np.int32)
    rc, c, s, sro = orc.quantize_grouped_gather(xt, idx, off)
    assert rc == -7
    g = xt[np.clip(idx, 0, 15)].copy()
    g[2] = 0
    g[4] = 0
    rc2, c2, s2, _ = orc.quantize_grouped(g, off)
    assert np.array_equal(c, c2) and np.array_equal(s, s2)
    assert not c[2].any() and not c[4].any()
