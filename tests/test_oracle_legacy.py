"""The scale rule the pages' fix replaced, as a reported comparison.

PR #43557 page, "Motivation": the old kernel took the biased exponent of
max/6 as the block scale; because floor(log2(a/b)) is not floor(log2 a) -
floor(log2 b), that scale is one too small for most inputs and the block
max, divided by the scale, lands far above 6 (E2M1's largest magnitude), so
the block saturates.  The oracle reproduces that rule (comparison only; the
library never uses it) and these tests pin it and report what it costs on
the workloads."""
import numpy as np

import workloads as W


def _bf16_values(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_legacy_scale_closed_form(orc):
    """biased_exp(v/6) == floor(log2(v/6)) + 127 for every positive normal
    BF16 v whose quotient stays a normal float32 (the quotient of an 8-bit
    significand by 3 never rounds onto a power of two)."""
    bits = np.arange(0x0180, 0x7F80, 97, dtype=np.uint16)
    for b in bits:
        v = float(_bf16_values(np.array([b]))[0])
        want = int(np.floor(np.log2(v / 6.0))) + 127
        assert orc.e8m0_scale_legacy(v) == want, hex(int(b))
    assert orc.e8m0_scale_legacy(0.0) == 0


def test_legacy_vs_fixed_ratio_table(orc):
    """For block maxima across the page's 1.2 .. 5.5 range: the fixed rule
    puts vecMax / 2^(s-127) in [3.5, 7), the legacy rule in [6, 12), one
    scale step lower (or equal when vecMax/6 sits just above a power of two)."""
    rows = []
    for v in (1.2, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 4.5, 5.0, 5.5):
        vb = float(np.float32(v))
        s_new = orc.e8m0_scale(vb)
        s_old = orc.e8m0_scale_legacy(vb)
        r_new = vb / 2.0 ** (s_new - 127)
        r_old = vb / 2.0 ** (s_old - 127)
        rows.append((v, s_old, s_new, r_old, r_new))
        assert 3.5 <= r_new < 7.0 and 6.0 <= r_old < 12.0
        assert s_old in (s_new - 1, s_new)
    print("\nvecMax  s_legacy  s_fixed  max/scale legacy  max/scale fixed")
    for v, so, sn, ro, rn in rows:
        print(f"{v:6.2f}  {so:8d}  {sn:7d}  {ro:16.3f}  {rn:15.3f}")
    assert sum(so < sn for _, so, sn, _, _ in rows) > len(rows) // 2


def _report(orc, xb):
    M, K = xb.shape
    x = _bf16_values(xb)
    out = {}
    for name, fn in (("fixed", orc.quantize_flat), ("legacy", orc.quantize_flat_legacy)):
        codes, flat = fn(xb)
        y = _bf16_values(orc.dequantize(codes, orc.tile(flat), M, K))
        scale = np.ldexp(1.0, np.repeat(flat.astype(np.int64), 32, axis=1) - 127)
        live = flat.repeat(32, axis=1) > 0
        ratio = np.where(live, np.abs(x) / scale, 0.0)
        sat = float(np.mean(ratio > 6.0))
        rel = float(np.linalg.norm(y - x) / np.linalg.norm(x))
        out[name] = (sat, rel, float(ratio.max()))
    return out


def test_legacy_scale_saturates_workloads(orc):
    """Reported comparison on the dense activation (256 rows of 4096 x 7168)
    and the edge-case matrix: saturated-element fraction and reconstruction
    relative L2 error under each rule, and the largest |x|/scale.  Under the
    fixed rule only block maxima with a mantissa in (1.5, 1.75) exceed 6 (by
    less than 7/6); under the legacy rule the block maxima reach up to 12 and
    many more elements saturate."""
    print("\nworkload                 rule    saturated  rel-L2   max |x|/scale")
    for label, xb in (("dense 256x7168", W.bf16_bits(W.dense_activation(1, 256, 7168))),
                      ("edge 1000x2880", W.bf16_bits(W.edge_cases(4)))):
        r = _report(orc, xb)
        for rule in ("fixed", "legacy"):
            print(f"{label:24s} {rule:7s} {r[rule][0]:9.5f}  {r[rule][1]:.5f}  {r[rule][2]:.3f}")
        assert r["fixed"][2] < 7.0 and r["legacy"][2] > 10.0
        assert r["legacy"][0] > 5.0 * r["fixed"][0]
        assert r["legacy"][1] > 1.5 * r["fixed"][1]
