"""Pins of the oracle's tiled scale layout (step 5).

The tiled layout is defined on the PR #43557 page ('Key source snippets',
untile_cutlass_scale) by a reshape to [numMTiles, numKTiles, 32, 4, 4], a
permute (0,3,2,1,4), a reshape to [padded_M, padded_sK] and a crop.  That
definition is restated here with numpy and the oracle's tile/untile are
checked against it, together with hand-derived byte offsets.
"""
import numpy as np
import pytest

from conftest import load_golden

SHAPES = [(128, 256), (1000, 2880), (1, 32), (129, 160), (256, 7168), (300, 96)]


def untile_by_permute(raw, rows, K):
    sK = K // 32
    nm, nk = (rows + 127) // 128, (sK + 3) // 4
    pm, pk = nm * 128, nk * 4
    t = raw[: pm * pk].reshape(nm, nk, 32, 4, 4).transpose(0, 3, 2, 1, 4)
    return np.ascontiguousarray(t).reshape(pm, pk)


@pytest.mark.parametrize("M,K", SHAPES)
def test_tile_matches_permute_definition(orc, M, K):
    sK = K // 32
    rng = np.random.default_rng(M * 7 + K)
    flat = rng.integers(1, 256, (M, sK), dtype=np.uint16).astype(np.uint8)
    tiled = orc.tile(flat)
    assert tiled.size == orc.scale_bytes(M, K)
    full = untile_by_permute(tiled, M, K)
    assert np.array_equal(full[:M, :sK], flat)
    pad = full.copy()
    pad[:M, :sK] = 0
    assert not pad.any(), "pad bytes must be zero"
    assert np.array_equal(orc.untile(tiled, M, sK), flat)


@pytest.mark.parametrize("M,K", SHAPES)
def test_untile_tile_roundtrip(orc, M, K):
    sK = K // 32
    rng = np.random.default_rng(M + K)
    raw = rng.integers(0, 256, orc.scale_bytes(M, K), dtype=np.uint16).astype(np.uint8)
    full = untile_by_permute(raw, M, K)
    full[M:, :] = 0
    full[:, sK:] = 0
    # build a tiled buffer with zero pads by inverting the permute definition
    nm, nk = (M + 127) // 128, (sK + 3) // 4
    t = full.reshape(nm, 4, 32, nk, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
    assert np.array_equal(orc.tile(orc.untile(t, M, sK)), t)


def test_tile_hand_offsets(orc):
    g = load_golden("tile_offsets.json")
    M, K = g["M"], g["K"]
    sK = K // 32
    assert orc.scale_bytes(M, K) == g["total_bytes"]
    for c in g["cases"]:
        flat = np.zeros((M, sK), np.uint8)
        flat[c["r"], c["c"]] = 0xAB
        t = orc.tile(flat)
        assert np.nonzero(t)[0].tolist() == [c["offset"]], c


def test_scale_bytes_closed_form(orc):
    assert orc.scale_bytes(128, 256) == 1024
    assert orc.scale_bytes(4096, 7168) == 4096 * 224
    assert orc.scale_bytes(1000, 2880) == 1024 * 92
    assert orc.scale_bytes(1, 32) == 128 * 4
    assert orc.scale_bytes(0, 32) == 0
    assert orc.scale_bytes(5, 33) == 0
