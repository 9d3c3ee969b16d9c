"""Pins of the oracle's [w1; w3] -> [w3; w1] swap (step 8), from the worked
tensors of the PR #51038 page ('[Bugfix][Quantization] Fix MXFP4 conversion
for FlashInfer CUTLASS', test_convert_standard_mxfp4_weights_for_flashinfer_cutlass)."""
import numpy as np

from conftest import load_golden


def test_page_arange_case(orc):
    g = load_golden("swap_w13_arange.json")
    w13 = np.array(g["w13"], np.uint8)
    assert np.array_equal(orc.swap_halves(w13), np.array(g["w13_expected"], np.uint8))
    s13 = np.array(g["w13_scale"], np.uint8)
    assert np.array_equal(orc.swap_halves(s13), np.array(g["w13_scale_expected"], np.uint8))
    b13 = np.array(g["w13_bias"], np.float32)
    want = np.array([[int(h, 16) for h in row] for row in g["w13_bias_expected_bf16_hex"]], np.uint16)
    assert np.array_equal(orc.swap_bias_bf16(b13), want)
    b2 = np.array(g["w2_bias"], np.float32)
    want2 = np.array([[int(h, 16) for h in row] for row in g["w2_bias_expected_bf16_hex"]], np.uint16)
    assert np.array_equal(orc.cast_bf16(b2), want2)


def test_full_swap_page_shapes(orc):
    """The page's w13_scale [1, 4, 2] is the flat scale layout of K = 64."""
    g = load_golden("swap_w13_arange.json")
    K = 64
    codes = np.arange(4 * 32, dtype=np.uint16).astype(np.uint8).reshape(1, 4, 32)
    s13 = np.array(g["w13_scale"], np.uint8)
    b13 = np.array(g["w13_bias"], np.float32)
    b2 = np.array(g["w2_bias"], np.float32)
    c_out, s_out, b13_out, b2_out = orc.swap_w13(codes, s13, b13, 1, 4, K, 0, b2)
    assert np.array_equal(c_out[0], codes[0][[2, 3, 0, 1]])
    assert np.array_equal(s_out, np.array(g["w13_scale_expected"], np.uint8))
    assert [hex(v) for v in b13_out[0]] == ["0x4000", "0x4040", "0x0", "0x3f80"]
    assert [hex(v) for v in b2_out[0]] == ["0x0", "0x3f80", "0x4000", "0x4040"]


def test_swap_twice_identity_and_tiled_commutes(orc):
    rng = np.random.default_rng(11)
    E, two_n, K = 3, 200, 160
    sK = K // 32
    codes = rng.integers(0, 256, (E, two_n, K // 2), dtype=np.uint16).astype(np.uint8)
    flat = rng.integers(0, 256, (E, two_n, sK), dtype=np.uint16).astype(np.uint8)
    tiled = np.concatenate([orc.tile(flat[e]) for e in range(E)])
    bias = rng.standard_normal((E, two_n)).astype(np.float32)
    c1, s1, b1, _ = orc.swap_w13(codes, flat, bias, E, two_n, K, 0)
    c2, s2, _, _ = orc.swap_w13(c1, s1, None, E, two_n, K, 0)
    assert np.array_equal(c2, codes) and np.array_equal(s2, flat)
    _, st, bt, _ = orc.swap_w13(codes, tiled, bias, E, two_n, K, 1)
    want = np.concatenate([orc.tile(s1[e]) for e in range(E)])
    assert np.array_equal(st, want)
    assert np.array_equal(bt, b1)
    n = two_n // 2
    assert np.array_equal(b1, orc.cast_bf16(np.concatenate([bias[:, n:], bias[:, :n]], 1)))
