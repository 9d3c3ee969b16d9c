"""The oracle's host-thread drivers equal its single calls byte for byte:
the unchanged routines run on 128-row bands (dense quantize, dequantize) or
on contiguous ranges of experts (grouped MXFP4 and NVFP4), so the full-size
GPU comparisons can use all host cores.  Ragged bands, empty experts at
either end, more threads than parts and malformed offsets included."""
import numpy as np
import pytest


def _bf16(rng, shape, scale=1.0):
    f = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("M,K,threads", [(1000, 288, 3), (128, 64, 8), (1, 32, 4), (257, 7168, 2)])
def test_dense_bands(orc, M, K, threads):
    rng = np.random.default_rng(M + K)
    x = _bf16(rng, (M, K), 3.0)
    c, s = orc.quantize(x)
    c2, s2 = orc.quantize_threads(x, threads)
    assert np.array_equal(c, c2) and np.array_equal(s, s2)
    y = orc.dequantize(c, s, M, K)
    assert np.array_equal(y, orc.dequantize_threads(c, s, M, K, threads))


OFFSETS = [
    [0, 0, 130, 131, 500, 500, 999, 1000],
    [0, 1000],
    [0, 0, 0, 1000, 1000],
    [0, 128, 256, 384, 512, 640, 768, 896, 1000],
]


@pytest.mark.parametrize("off", OFFSETS)
@pytest.mark.parametrize("threads", [1, 3, 16])
def test_grouped_ranges(orc, off, threads):
    rng = np.random.default_rng(len(off) * 7 + threads)
    x = _bf16(rng, (1000, 160))
    o = np.array(off, np.int32)
    rc, c, s, sro = orc.quantize_grouped(x, o)
    rc2, c2, s2, sro2 = orc.quantize_grouped_threads(x, o, threads)
    assert rc == rc2 == 0
    assert np.array_equal(c, c2) and np.array_equal(sro, sro2)
    assert s2.size == int(sro[-1]) * 8 and np.array_equal(s[:s2.size], s2)
    assert not s[s2.size:].any()                 # the bound's slack holds nothing
    g = rng.uniform(0.1, 3000.0, o.size - 1).astype(np.float32)
    rc, c, s, sro = orc.nvfp4_quantize_grouped(x, o, g)
    rc2, c2, s2, sro2 = orc.nvfp4_quantize_grouped_threads(x, o, g, threads)
    assert rc == rc2 == 0
    assert np.array_equal(c, c2) and np.array_equal(sro, sro2)
    assert s2.size == int(sro[-1]) * 12 and np.array_equal(s[:s2.size], s2)


def test_grouped_ranges_bad_offsets_fall_back_to_the_single_call(orc):
    x = _bf16(np.random.default_rng(1), (20, 64))
    for off in ([1, 10, 20], [0, 12, 8, 20], [0, 10, 19]):
        o = np.array(off, np.int32)
        rc, _, _, sro = orc.quantize_grouped_threads(x, o, 4)
        assert rc == -6 and (sro == -1).all()
