"""Pins of the oracle's NVFP4 path: FP8 E4M3 conversion, the block steps, the
tiled layout with 16-element scale columns, and dequantize."""
import numpy as np
import pytest
import torch

from conftest import load_golden
import workloads as W

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def torch_e4m3(vals):
    t = torch.tensor(np.asarray(vals, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch(orc):
    b = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(b.copy()).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = np.array([orc.e4m3_to_double(int(v)) for v in b])
    fin = np.isfinite(want)
    assert np.array_equal(got[fin], want[fin]) and np.isnan(got[~fin]).all()
    assert orc.e4m3_to_double(0x7E) == 448.0


def test_e4m3_encode_matches_torch_in_range(orc):
    """Round to nearest even against torch's float32 -> float8_e4m3fn cast:
    random values, every exact midpoint between neighbours, subnormals."""
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.uniform(-448, 448, 20000),
        np.exp2(rng.uniform(-12, 8.8, 20000)) * rng.choice([-1, 1], 20000),
    ])
    grid = np.unique(np.abs([orc.e4m3_to_double(i) for i in range(0x7F)]))
    mids = (grid[:-1] + grid[1:]) / 2
    vals = np.concatenate([vals, mids, -mids, grid]).astype(np.float32)
    vals = vals[np.abs(vals) <= 448]
    assert np.array_equal(orc.e4m3_from_double_many(vals.astype(np.float64)), torch_e4m3(vals))


def test_e4m3_saturates(orc):
    big = np.array([448.0, 449.0, 463.99, 464.0, 1e6, -500.0])
    assert [hex(v) for v in orc.e4m3_from_double_many(big)] == ["0x7e"] * 5 + ["0xfe"]


def _nibbles(codes):
    n = np.zeros((codes.shape[0], codes.shape[1] * 2), np.uint8)
    n[:, 0::2] = codes & 0xF
    n[:, 1::2] = codes >> 4
    return n


def test_nvfp4_worked_blocks(orc):
    g = load_golden("nvfp4_worked_blocks.json")
    for blk in g["blocks"]:
        x = np.zeros((1, 16), np.uint16)
        vals = [int(h, 16) for h in blk["x"]]
        x[0, :len(vals)] = vals
        codes, flat = orc.nvfp4_quantize_flat(x, blk["g"])
        assert int(flat[0, 0]) == int(blk["sf"], 16), blk["name"]
        want = np.zeros(16, np.uint8)
        want[:len(blk["codes"])] = [int(c, 16) for c in blk["codes"]]
        assert list(_nibbles(codes)[0]) == list(want), blk["name"]
    for c in g["dequant"]:
        codes = np.zeros((1, 32), np.uint8)
        codes[0, 0] = int(c["code"], 16)
        flat = np.zeros((1, 4), np.uint8)
        flat[0, 0] = int(c["sf"], 16)
        y = orc.nvfp4_dequantize(codes, orc.tile(flat), 1, 64, c["g"])
        assert int(y[0, 0]) == int(c["y"], 16), c


@pytest.mark.parametrize("g", [1.0, 0.37, 2688.0 / 17.0])
def test_nvfp4_block_properties(orc, g):
    """Every block: the scale byte is the nearest E4M3 to g*vecMax/6 (within
    its half-ulp, or saturated), and every code is the E2M1 value nearest to
    x*g/SFValue (up to the float32 rounding of g/SFValue)."""
    x = W.dense_activation(21, 64, 256)
    xb = W.bf16_bits(x)
    codes, flat = orc.nvfp4_quantize_flat(xb, g)
    xv = x.float().numpy().astype(np.float64).reshape(64, 16, 16)
    vmax = np.abs(xv).max(axis=2)
    target = g * vmax / 6
    sfv = np.vectorize(orc.e4m3_to_double)(flat)
    grid = np.unique(np.abs([orc.e4m3_to_double(i) for i in range(0x7F)]))
    for t, v in zip(target.ravel(), sfv.ravel()):
        if t >= 448:
            assert v == 448
        else:
            nearest = grid[np.argmin(np.abs(grid - t))]
            assert abs(v - t) <= abs(nearest - t) * (1 + 1e-6) + 1e-12
    nib = _nibbles(codes).reshape(64, 16, 16)
    mag = E2M1[nib & 7]
    y = np.abs(xv) * g / np.where(sfv > 0, sfv, 1)[:, :, None]
    y = np.minimum(y, 6.5)
    err = np.abs(mag - y)
    step = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0))
    live = (sfv > 0)[:, :, None] & np.ones_like(y, bool)
    assert np.all(err[live] <= step[live] * (1 + 1e-5) + 1e-6)
    assert not nib[~live].any()


def test_nvfp4_tiled_layout_is_the_mx_layout_on_16_element_columns(orc):
    x = W.bf16_bits(W.dense_activation(22, 200, 480))
    codes, tiled = orc.nvfp4_quantize(x, 1.0)
    c2, flat = orc.nvfp4_quantize_flat(x, 1.0)
    assert np.array_equal(codes, c2)
    assert tiled.size == orc.nvfp4_scale_bytes(200, 480) == 256 * 32
    assert np.array_equal(orc.untile(tiled, 200, 30), flat)


def test_nvfp4_grouped_equals_per_segment_dense(orc):
    """NVFP4 experts quant: each segment equals the dense NVFP4 quantize of
    its rows with its own global scale, at its padded scale offset; empty
    segments contribute nothing."""
    g = W.moe_grouped(seed=3, tokens=90, top_k=2, num_experts=6, K=96)
    xb = W.bf16_bits(g.x)
    off = g.offsets.numpy().copy()
    off[3] = off[2]                                   # make segment 2 empty
    gs = np.array([1.0, 0.37, 5.0, 448 * 6 / 3.7, 2.0 ** -10, 17.0], np.float32)
    rc, codes, scales, sro = orc.nvfp4_quantize_grouped(xb, off, gs)
    assert rc == 0
    pk = (96 // 16 + 3) // 4 * 4
    P = 0
    for e in range(6):
        a, b = int(off[e]), int(off[e + 1])
        assert sro[e] == P
        if b > a:
            c_e, s_e = orc.nvfp4_quantize(xb[a:b], float(gs[e]))
            assert np.array_equal(codes[a:b], c_e), e
            assert np.array_equal(scales[P * pk:P * pk + s_e.size], s_e), e
        P += (b - a + 127) // 128 * 128
    assert sro[6] == P


def test_nvfp4_grouped_uniform_tiles_equal_dense_and_bad_offsets(orc):
    xb = W.bf16_bits(W.small_matrix(5, 384, 64))
    off = np.array([0, 128, 256, 384], np.int32)
    rc, codes, scales, _ = orc.nvfp4_quantize_grouped(xb, off, np.full(3, 2.5, np.float32))
    c_d, s_d = orc.nvfp4_quantize(xb, 2.5)
    assert rc == 0 and np.array_equal(codes, c_d) and np.array_equal(scales[:s_d.size], s_d)
    rc, _, _, sro = orc.nvfp4_quantize_grouped(xb, np.array([0, 200, 100, 384], np.int32),
                                               np.ones(3, np.float32))
    assert rc == -6 and (sro == -1).all()


def test_nvfp4_f16_equals_bf16_on_shared_values(orc):
    """NVFP4 on FP16 input decodes the element and nothing else: on values
    both formats hold exactly (BF16 values inside FP16's normal range) the
    FP16 and BF16 paths give the same bytes, dense and grouped; FP16 values
    BF16 cannot hold change the result."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((200, 96)) * np.exp2(rng.uniform(-8, 8, (200, 1))))
    x[np.abs(x) < 2.0 ** -13] = 0.0                              # stay in FP16's normal range
    xb = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    xh = xb.to(torch.float16)
    assert torch.equal(xh.float(), xb.float())                 # exact in both
    bb = xb.view(torch.int16).numpy().view(np.uint16)
    hb = xh.view(torch.int16).numpy().view(np.uint16)
    for g in (1.0, 37.5, 448 * 6 / 300.0):
        c1, s1 = orc.nvfp4_quantize(bb, g)
        c2, s2 = orc.nvfp4_quantize(hb, g, f16=True)
        assert np.array_equal(c1, c2) and np.array_equal(s1, s2)
    off = np.array([0, 70, 70, 200], np.int32)
    gs = np.array([2.0, 5.0, 0.75], np.float32)
    r1 = orc.nvfp4_quantize_grouped(bb, off, gs)
    r2 = orc.nvfp4_quantize_grouped(hb, off, gs, f16=True)
    assert r1[0] == r2[0] == 0 and all(np.array_equal(a, b) for a, b in zip(r1[1:], r2[1:]))
    # an FP16 value with more than 8 significant bits changes some code or scale
    hf = torch.from_numpy(x.astype(np.float32)).to(torch.float16)
    hf_b = hf.view(torch.int16).numpy().view(np.uint16)
    c3, _ = orc.nvfp4_quantize(hf_b, 1.0, f16=True)
    c4, _ = orc.nvfp4_quantize(bb, 1.0)
    assert not np.array_equal(c3, c4)


# ------------------------------------------------ NVFP4 experts quant, scatter
def test_nvfp4_scatter_hand_example(orc):
    """Two tokens of one 16-element block, two experts with global scales 1
    and 2; token 0 -> rows 0 (expert 0) and 2 (expert 1), token 1 -> row 1
    (expert 0), its second route dropped, so row 3 keeps its bytes.
      row 0: block N1 at g = 1: vecMax 6, sf 1.0 = 0x38, codes 7 D 3 2;
      row 1: block N7's x at g = 1: vecMax 3, q = 0.5, sf 0.5 = 0x30,
             inv = 1 / 0.5 = 2 (as N7's inv at g = 2), codes 7 4 B;
      row 2: block N1 at g = 2: sf 2.0 = 0x40, inv = 2 / 2 = 1, codes 7 D 3 2.
    One scale column (K = 16), so padded row p of a segment puts its byte at
    (p % 32) * 16 + (p / 32) * 4 of the segment's 512-byte chunk; expert 1's
    chunk starts at byte 128 * 4 = 512."""
    x = np.zeros((2, 16), np.uint16)
    x[0, :4] = [0x40C0, 0xC040, 0x3FC0, 0x3F40]
    x[1, :3] = [0x4040, 0x3F80, 0xBF40]
    dest = np.array([[0, 2], [1, -1]], np.int32)
    off = np.array([0, 2, 4], np.int32)
    g = np.array([1.0, 2.0], np.float32)
    c0 = np.full((4, 8), 0xEE, np.uint8)
    s0 = np.full(orc.nvfp4_grouped_scale_bytes_bound(4, 2, 16), 0xEE, np.uint8)
    rc, c, s, sro = orc.nvfp4_quantize_grouped_scatter(x, dest, off, 4, g, c0, s0)
    assert rc == 0 and list(sro) == [0, 128, 256]
    want_c = np.zeros((4, 8), np.uint8)
    want_c[0, :2] = [0xD7, 0x23]
    want_c[1, :2] = [0x47, 0x0B]
    want_c[2, :2] = [0xD7, 0x23]
    want_c[3] = 0xEE                                   # untargeted row: kept
    assert np.array_equal(c, want_c)
    want_s = np.zeros(1024, np.uint8)
    want_s[0], want_s[16], want_s[512] = 0x38, 0x30, 0x40
    want_s[528:532] = 0xEE                             # row 3 = expert 1's padded row 1: kept
    assert np.array_equal(s, want_s)


def _permuted(xb, dest, total):
    rows = np.zeros((total, xb.shape[1]), np.uint16)
    hit = np.zeros(total, bool)
    for t in range(dest.shape[0]):
        for d in dest[t]:
            if d >= 0:
                rows[d] = xb[t]
                hit[d] = True
    return rows, hit


@pytest.mark.parametrize("f16", [False, True])
def test_nvfp4_scatter_equals_experts_quant_of_the_permuted_batch(orc, f16):
    g = W.moe_grouped(seed=41, tokens=150, top_k=3, num_experts=7, K=80)
    xt = g.x_tokens
    if f16:
        xt = xt.float().clamp(-60000, 60000).to(torch.float16)
        xb = xt.view(torch.int16).numpy().view(np.uint16)
    else:
        xb = W.bf16_bits(xt)
    dest = g.dest_rows.numpy()
    off = g.offsets.numpy()
    total = dest.size
    gs = (448.0 * 6.0 / np.exp(np.random.default_rng(41).uniform(0, 3, 7))).astype(np.float32)
    perm, _ = _permuted(xb, dest, total)
    rc0, c0, s0, sro0 = orc.nvfp4_quantize_grouped(perm, off, gs, f16=f16)
    rc, c, s, sro = orc.nvfp4_quantize_grouped_scatter(xb, dest, off, total, gs, f16=f16)
    assert rc == rc0 == 0 and np.array_equal(sro, sro0)
    assert np.array_equal(c, c0) and np.array_equal(s, s0)
    # dropped routes: targeted rows and pad rows as above, untargeted rows keep
    # a random prefill (codes and all their scale bytes)
    rng = np.random.default_rng(42)
    dd = dest.copy()
    dd[rng.random(dd.shape) < 0.25] = -1
    cp = rng.integers(0, 256, c0.shape, dtype=np.uint8)
    sp = rng.integers(0, 256, s0.shape, dtype=np.uint8)
    rc, c, s, _ = orc.nvfp4_quantize_grouped_scatter(xb, dd, off, total, gs, cp, sp, f16=f16)
    _, hit = _permuted(xb, dd, total)
    assert rc == 0
    assert np.array_equal(c[hit], c0[hit]) and np.array_equal(c[~hit], cp[~hit])
    nkt = (80 // 16 + 3) // 4
    for e in range(7):
        for p in range((off[e + 1] - off[e] + 127) // 128 * 128):
            r = off[e] + p
            base = int(sro0[e]) * nkt * 4
            idx = [base + (p // 128 * nkt + c // 4) * 512 + (p % 32) * 16 + (p % 128) // 32 * 4
                   + c % 4 for c in range(nkt * 4)]
            src = sp if (p < off[e + 1] - off[e] and not hit[r]) else s0
            assert np.array_equal(s[idx], src[idx]), (e, p)


def test_nvfp4_scatter_one_scale_every_route_is_the_dense_row(orc):
    """With one global scale for every expert, each route of a token carries
    the dense NVFP4 quantization of its token row: the same codes, and in
    every scale column the same E4M3 byte (read through the tiled layout:
    padded row p, column c at ((p/128)*nKT + c/4)*512 + (p%32)*16 +
    ((p%128)/32)*4 + c%4, segment e's rows starting at its padded start)."""
    g = W.moe_grouped(seed=43, tokens=40, top_k=4, num_experts=6, K=96)
    xb = W.bf16_bits(g.x_tokens)
    dest = g.dest_rows.numpy()
    off = g.offsets.numpy()
    gs = np.full(6, 448.0 * 6.0 / 5.0, np.float32)
    rc, c, s, sro = orc.nvfp4_quantize_grouped_scatter(xb, dest, off, dest.size, gs)
    assert rc == 0
    sK = 96 // 16
    nKT = (sK + 3) // 4

    def col_bytes(buf, p):
        return [int(buf[((p // 128) * nKT + k // 4) * 512 + (p % 32) * 16 +
                        ((p % 128) // 32) * 4 + k % 4]) for k in range(sK)]

    for t in range(40):
        cd, sd = orc.nvfp4_quantize(xb[t:t + 1], float(gs[0]))
        for v in dest[t]:
            e = int(np.searchsorted(off, v, side="right")) - 1
            p = int(sro[e]) + int(v) - int(off[e])
            assert np.array_equal(c[v], cd[0]), (t, v)
            assert col_bytes(s, p) == col_bytes(sd, 0), (t, v)


def test_nvfp4_scatter_bad_entries_and_offsets(orc):
    g = W.moe_grouped(seed=43, tokens=40, top_k=2, num_experts=3, K=32)
    xb = W.bf16_bits(g.x_tokens)
    dest = g.dest_rows.numpy().copy()
    off = g.offsets.numpy()
    gs = np.array([1.0, 5.0, 0.25], np.float32)
    clean = dest.copy()
    clean[3, 1] = -1
    clean[7, 0] = -1
    dest[3, 1] = 80            # == total_rows: outside
    dest[7, 0] = -5
    r1 = orc.nvfp4_quantize_grouped_scatter(xb, dest, off, 80, gs)
    r2 = orc.nvfp4_quantize_grouped_scatter(xb, clean, off, 80, gs)
    assert r1[0] == -7 and r2[0] == 0
    assert all(np.array_equal(a, b) for a, b in zip(r1[1:], r2[1:]))
    bad = np.array([0, 50, 40, 80], np.int32)
    cp = np.full((80, 16), 0x5A, np.uint8)
    rc, c, s, sro = orc.nvfp4_quantize_grouped_scatter(xb, clean, bad, 80, gs, cp)
    assert rc == -6 and (sro == -1).all() and (c == 0x5A).all() and not s.any()


@pytest.mark.parametrize("g", [1.0, 0.37, 2688.0 / 25.0, 1.0e30, 1.0e-30])
def test_nvfp4_dequantize_every_code_and_scale_byte(orc, g):
    """All 16 codes x all 256 E4M3 scale bytes (negative, subnormal and the
    NaN bytes 0x7F / 0xFF included) against torch: the E4M3 value from
    torch's float8_e4m3fn, the float32 products (e2m1 * float(byte)) *
    float32(1/g), torch's BF16 cast; the NaN bytes give 0x7FC0 for the block
    (the library's NaN, as for the E8M0 NaN 255)."""
    torch = pytest.importorskip("torch")
    e2m1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6], np.float32)
    M, K = 256, 256                         # one scale byte per 16-element block
    sb = np.arange(M * (K // 16)) % 256     # every byte, 16 times over
    flat = sb.astype(np.uint8).reshape(M, K // 16)
    nib = np.tile(np.arange(16), M * K // 16).reshape(M, K)
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    y = orc.nvfp4_dequantize(codes, orc.tile(flat), M, K, g)
    sfv = torch.from_numpy(flat).view(torch.float8_e4m3fn).float().numpy()
    inv = np.float32(1.0) / np.float32(g)
    prod = (e2m1[nib] * np.repeat(sfv, 16, axis=1)).astype(np.float32) * inv
    want = torch.from_numpy(prod.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
    want = want.numpy().view(np.uint16).copy()
    nan_blk = np.repeat((flat & 0x7F) == 0x7F, 16, axis=1)
    want[nan_blk] = 0x7FC0
    assert not np.isnan(prod[~nan_blk]).any()
    assert np.array_equal(y, want), (np.argwhere(y != want)[:3], y[y != want][:3],
                                     want[y != want][:3])
