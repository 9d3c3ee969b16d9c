"""Pins of the oracle's whole-matrix quantize (steps 1-5), grouped quantize
(step 6) and dequantize (step 7): properties that hold for the method at any
size, checked on seeded inputs of the workloads' distributions."""
import numpy as np
import pytest
import torch

from conftest import load_golden
import workloads as W


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


def test_grouped_scatter_equals_gather_of_inverse(orc):
    """The dispatch as a scatter (token, route -> row) with every row
    targeted equals the gather form with the inverse map (row -> token) and
    the grouped quantize of the explicitly permuted matrix."""
    g = W.moe_grouped(seed=2, tokens=80, top_k=3, num_experts=7, K=192)
    xt = W.bf16_bits(g.x_tokens)
    idx = g.row_index.numpy()
    dst = g.dest_rows.numpy()
    off = g.offsets.numpy()
    assert np.array_equal(idx[dst], np.repeat(np.arange(80), 3).reshape(80, 3))
    rc, c, s, sro = orc.quantize_grouped_scatter(xt, dst, off, idx.size)
    rc2, c2, s2, sro2 = orc.quantize_grouped_gather(xt, idx, off)
    rc3, c3, s3, sro3 = orc.quantize_grouped(xt[idx], off)
    assert rc == rc2 == rc3 == 0
    for a, b in ((c, c2), (s, s2), (sro, sro2), (c, c3), (s, s3)):
        assert np.array_equal(a, b)


def _packed(nibbles):
    n = np.asarray(nibbles, np.uint8)
    return (n[0::2] | (n[1::2] << 4)).astype(np.uint8)


def _golden_block(blk):
    x = np.zeros(32, np.uint16)
    x[: len(blk["x"])] = [int(h, 16) for h in blk["x"]]
    nib = np.zeros(32, np.uint8)
    nib[: len(blk["codes"])] = [int(c, 16) for c in blk["codes"]]
    return x, _packed(nib), blk["s"]


def test_grouped_scatter_worked_example(orc):
    """Two tokens (worked blocks A and B), two routes each, two experts of two
    rows, K = 32.  Token A goes to rows 1 and 2, token B to rows 0 and 3
    (route 1 of B dropped in the second call).  Expected bytes written out by
    hand: expert 1's scales start at padded row 128 (byte 512); padded row r
    of a segment with one k-tile holds its 4 scale bytes at (r % 32) * 16 +
    ((r % 128) // 32) * 4; codes rows are the blocks' packed codes."""
    g = load_golden("e8m0_e2m1_worked_blocks.json")["blocks"]
    xa, pa, sa = _golden_block(g[0])
    xb, pb, sb = _golden_block(g[1])
    x = np.stack([xa, xb])
    off = np.array([0, 2, 4], np.int32)
    for dropped in (False, True):
        dst = np.array([[1, 2], [0, -1 if dropped else 3]], np.int32)
        codes0 = np.full((4, 16), 0xA5, np.uint8)
        scales0 = np.full(1024, 0xA5, np.uint8)
        rc, c, s, sro = orc.quantize_grouped_scatter(x, dst, off, 4, codes0, scales0)
        assert rc == 0 and list(sro) == [0, 128, 256]
        want_c = np.stack([pb, pa, pa, pb])
        want_s = np.zeros(1024, np.uint8)
        want_s[0], want_s[16], want_s[512], want_s[528] = sb, sa, sa, sb
        if dropped:
            want_c[3] = 0xA5
            want_s[528:532] = 0xA5
        assert np.array_equal(c, want_c)
        assert np.array_equal(s, want_s), np.nonzero(s != want_s)


def test_grouped_scatter_untargeted_rows_untouched(orc):
    """Dropped routes (-1) leave their rows as they were, codes and scale
    bytes; every targeted row and every pad row is as in the full result."""
    g = W.moe_grouped(seed=6, tokens=150, top_k=4, num_experts=9, K=160)
    xt = W.bf16_bits(g.x_tokens)
    idx = g.row_index.numpy()
    dst = g.dest_rows.numpy().copy()
    off = g.offsets.numpy()
    total = idx.size
    rng = np.random.default_rng(0)
    drop = rng.random(dst.shape) < 0.2
    dropped_rows = dst[drop]
    dst[drop] = -1
    nsb = orc.grouped_scale_bytes_bound(total, 9, 160)
    codes0 = rng.integers(0, 256, (total, 80), dtype=np.uint8)
    scales0 = rng.integers(0, 256, nsb, dtype=np.uint8)
    rc, c, s, sro = orc.quantize_grouped_scatter(xt, dst, off, total, codes0, scales0)
    rc_f, c_f, s_f, _ = orc.quantize_grouped(xt[idx], off)
    assert rc == 0 and rc_f == 0
    kept = np.setdiff1d(np.arange(total), dropped_rows)
    assert np.array_equal(c[kept], c_f[kept])
    assert np.array_equal(c[dropped_rows], codes0[dropped_rows])
    # scale bytes: untile each segment from both buffers and compare per row
    sK = 5
    for e in range(9):
        n = int(off[e + 1] - off[e])
        pad_n = (n + 127) // 128 * 128
        seg = slice(int(sro[e]) * 8, (int(sro[e]) + pad_n) * 8)
        got = orc.untile(s[seg], pad_n, 8)
        full = orc.untile(s_f[seg], pad_n, 8)
        before = orc.untile(scales0[seg], pad_n, 8)
        rows = np.arange(pad_n)
        untargeted = np.isin(off[e] + rows, dropped_rows) & (rows < n)
        assert np.array_equal(got[~untargeted], full[~untargeted])
        assert not full[rows >= n].any() and not full[:, sK:].any()
        assert np.array_equal(got[untargeted], before[untargeted])


def test_grouped_scatter_bad_entries(orc):
    """An entry outside [-1, total_rows) is skipped (as if -1) and reported."""
    g = W.moe_grouped(seed=7, tokens=40, top_k=2, num_experts=3, K=64)
    xt = W.bf16_bits(g.x_tokens)
    dst = g.dest_rows.numpy().copy()
    off = g.offsets.numpy()
    total = g.row_index.numel()
    bad = dst.copy()
    bad[3, 1] = total
    bad[7, 0] = -2
    ok = dst.copy()
    ok[3, 1] = -1
    ok[7, 0] = -1
    rc, c, s, _ = orc.quantize_grouped_scatter(xt, bad, off, total)
    rc2, c2, s2, _ = orc.quantize_grouped_scatter(xt, ok, off, total)
    assert rc == -7 and rc2 == 0
    assert np.array_equal(c, c2) and np.array_equal(s, s2)
    rc3, _, _, sro = orc.quantize_grouped_scatter(xt, dst, np.array([0, 50, 40, total], np.int32),
                                                  total)
    assert rc3 == -6 and (sro == -1).all()
