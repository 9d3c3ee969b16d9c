"""Pins of the oracle's E8M0 scale (step 2) and block absmax (step 1).

The scale rule of the PR #43557 page ('Implementation breakdown' item 1, the
UE8M0 branch of the cvt_warp_fp16_to_fp4 excerpt) is checked over all 65,536
BF16 bit patterns against an independent formulation derived from it:
adding 2^21 to the float bits rounds the exponent up exactly when the
normalised mantissa is >= 1.75, so for v > 0
    s = clamp(floor(log2 v) + 127 + [mantissa >= 1.75] - 2, 0, 254),
computed here with frexp in float64.
"""
import numpy as np
import pytest

from conftest import load_golden

ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _bf16_values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _finite(bits):
    return (bits & 0x7F80) != 0x7F80


def independent_scale(v):
    m, e = np.frexp(v)              # v = m * 2^e, m in [0.5, 1)
    floor_log2 = e - 1
    mant = 2.0 * m                  # in [1, 2)
    s = floor_log2 + 127 + (mant >= 1.75) - 2
    s = np.clip(s, 0, 254)
    return np.where(v > 0, s, 0).astype(np.int64)


def test_scale_exhaustive_vs_log2_form(orc):
    fin = ALL[_finite(ALL)]
    assert fin.size == 65536 - 256   # 2 signs x 128 Inf/NaN patterns
    got = orc.e8m0_scale_many(fin).astype(np.int64)
    want = independent_scale(_bf16_values(fin))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(hex(int(fin[i])), int(got[i]), int(want[i])) for i in bad[:10]]


def test_scale_nonfinite_literal(orc):
    # +Inf: 0x7F800000 + 0x200000 keeps exponent 255 -> 253 (the cap never binds)
    assert orc.e8m0_scale(float("inf")) == 253


def test_scale_invariant_normal_blocks(orc):
    pos = ALL[(ALL < 0x7F80) & (ALL > 0)]          # positive finite
    v = _bf16_values(pos)
    s = orc.e8m0_scale_many(pos).astype(np.int64)
    nz = s >= 1
    ratio = v[nz] / np.ldexp(1.0, s[nz] - 127)
    assert ratio.min() >= 3.5 and ratio.max() < 7.0
    # s == 0 exactly below the smallest block max that reaches s = 1
    assert np.all(v[~nz] < 1.75 * 2.0 ** -125)
    assert np.all(v[nz] >= 1.75 * 2.0 ** -125)
    assert s.max() == 253


def test_scale_monotone(orc):
    pos = np.arange(0x0000, 0x7F80, dtype=np.uint16)
    s = orc.e8m0_scale_many(pos).astype(np.int64)
    assert np.all(np.diff(s) >= 0)
    # each step of s happens at a mantissa of 1.75 * 2^e
    steps = pos[1:][np.diff(s) == 1]
    assert np.all((steps & 0x7F) == 0x60)


def test_scale_worked_blocks(orc):
    g = load_golden("e8m0_e2m1_worked_blocks.json")
    for blk in g["blocks"]:
        x = np.zeros(32, np.uint16)
        vals = [int(h, 16) for h in blk["x"]]
        x[: len(vals)] = vals
        vmax = orc.lib().orc_block_absmax(x.ctypes.data_as(orc._u16p), 32)
        assert orc.e8m0_scale(vmax) == blk["s"], blk["name"]


def test_absmax_exact(orc):
    rng = np.random.default_rng(5)
    for _ in range(200):
        bits = rng.integers(0, 65536, 32, dtype=np.uint32).astype(np.uint16)
        bits = bits[_finite(bits)]
        if bits.size == 0:
            continue
        x = np.ascontiguousarray(bits)
        got = orc.lib().orc_block_absmax(x.ctypes.data_as(orc._u16p), x.size)
        assert got == np.abs(_bf16_values(x)).max()


def test_legacy_scale_is_one_too_small(orc):
    """The pages' root-cause statement (PR #43557 page, 'Motivation'): the
    old biased_exp(max/6) scale is one smaller than the fixed one for most
    inputs, because floor(log2(a/b)) != floor(log2 a) - floor(log2 b).
    Checked for the oracle's scale over every BF16 vecMax in [1, 8)."""
    bits = np.arange(0x3F80, 0x4100, dtype=np.uint16)
    v = _bf16_values(bits)
    new = orc.e8m0_scale_many(bits).astype(np.int64)
    old = np.floor(np.log2(v / 6.0)).astype(np.int64) + 127
    frac_smaller = np.mean(old < new)
    assert frac_smaller > 0.5
    # with the old scale the block max lands far above 6 (saturation)
    assert np.max(v / np.ldexp(1.0, old - 127)) > 10.0
