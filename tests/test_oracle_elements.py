"""Pins of the oracle's E2M1 element step (step 3) and dequantize value
(step 7).

Element: exhaustive over all finite BF16 inputs x 254 scale exponents
(s = 1..254) against an independent nearest-value search: y = x * 2^(127-s)
in float64, distance to each of the 8 E2M1 magnitudes, the smallest wins,
an exact tie goes to the even code (even mantissa bit), the sign bit is kept.
Blocks with s == 0 emit 0x0 (library convention).

Dequantize: all 16 codes x 256 scale bytes against the E2M1 value table of
the OCP MX definition times 2^(s-127) taken through float32 (exact for these
values, or +-Inf on overflow), upper 16 bits = BF16.
"""
import numpy as np

from conftest import load_golden

E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16)
FINITE = ALL[(ALL & 0x7F80) != 0x7F80]
XV = (FINITE.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
SIGN = ((FINITE >> 15) & 1).astype(np.uint8)


def nearest_code(y, sign):
    # every magnitude above 6 is nearest to 6 (saturation); capping at 7 keeps
    # that while avoiding float64 distance ties for huge |y|
    m = np.minimum(np.abs(y), 7.0)
    d = np.abs(m[:, None] - E2M1_MAG[None, :])
    dmin = d.min(axis=1, keepdims=True)
    weight = np.where(np.arange(8) % 2 == 0, 2, 1)[None, :]
    idx = np.argmax((d == dmin) * weight, axis=1).astype(np.uint8)
    return (sign << 3) | idx


def test_element_map_exhaustive(orc):
    for s in range(1, 255):
        got = orc.e2m1_encode_many(FINITE, s)
        want = nearest_code(np.ldexp(XV, 127 - s), SIGN)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (s, [(hex(int(FINITE[i])), int(got[i]), int(want[i])) for i in bad[:8]])


def test_element_s0_blocks_zero(orc):
    assert not orc.e2m1_encode_many(FINITE, 0).any()


def test_element_worked_blocks(orc):
    g = load_golden("e8m0_e2m1_worked_blocks.json")
    for blk in g["blocks"]:
        x = np.zeros((1, 32), np.uint16)
        vals = [int(h, 16) for h in blk["x"]]
        x[0, : len(vals)] = vals
        codes, flat = orc.quantize_flat(x)
        assert int(flat[0, 0]) == blk["s"], blk["name"]
        nib = np.zeros(32, np.uint8)
        nib[0::2] = codes[0] & 0xF       # element 2j in the low nibble
        nib[1::2] = codes[0] >> 4
        want = np.zeros(32, np.uint8)
        want[: len(blk["codes"])] = [int(c, 16) for c in blk["codes"]]
        assert list(nib) == list(want), blk["name"]
        if "packed_first_16_bytes" in blk:
            assert [int(b, 16) for b in blk["packed_first_16_bytes"]] == list(codes[0])


def test_dequant_values_exhaustive(orc):
    codes = np.repeat(np.arange(16, dtype=np.uint8), 256)
    scales = np.tile(np.arange(256, dtype=np.uint16), 16).astype(np.uint8)
    got = orc.dequant_value_many(codes, scales)
    mag = E2M1_MAG[codes & 7]
    val = np.where(codes >= 8, -mag, mag)
    val = np.where((codes & 7) == 0, np.where(codes >= 8, -0.0, 0.0), val)
    with np.errstate(over="ignore"):
        f32 = np.ldexp(val, scales.astype(np.int64) - 127).astype(np.float32)
    bits32 = f32.view(np.uint32)
    assert np.all(bits32[scales != 255] & 0xFFFF == 0)
    want = (bits32 >> 16).astype(np.uint16)
    want[scales == 255] = 0x7FC0
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(int(codes[i]), int(scales[i]), hex(int(got[i])), hex(int(want[i]))) for i in bad[:8]]


def test_dequant_worked(orc):
    g = load_golden("e8m0_e2m1_worked_blocks.json")["dequant"]["cases"]
    for c in g:
        y = orc.dequant_value_many(np.array([int(c["code"], 16)]), np.array([c["s"]]))
        assert int(y[0]) == int(c["y"], 16), c


def test_bf16_cast_matches_torch(orc):
    """double -> BF16 round-to-nearest-even against torch's float32 -> bfloat16
    cast (a library routine), on random float32 patterns, exact ties and
    subnormals."""
    import torch
    rng = np.random.default_rng(7)
    b = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    ties = (b & 0xFFFF0000) | 0x8000
    sub = b & 0x807FFFFF
    pats = np.concatenate([b, ties, sub])
    f = pats.view(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.cast_bf16(f)
    assert np.array_equal(got, want)


def test_decode_table(orc):
    for nib in range(16):
        v = orc.e2m1_decode(nib)
        mag = E2M1_MAG[nib & 7]
        assert abs(v) == mag and (np.signbit(v) == bool(nib & 8))
