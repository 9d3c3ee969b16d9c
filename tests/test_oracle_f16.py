"""Pins of the oracle's FP16-input path (same MX method, binary16 input)."""
import numpy as np

import workloads as W

E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16)
FIN16 = ALL[(ALL & 0x7C00) != 0x7C00]


def test_f16_decode_matches_numpy(orc):
    got = orc.f16_to_double_many(ALL)
    want = ALL.view(np.float16).astype(np.float64)
    fin = np.isfinite(want)
    assert np.array_equal(got[fin], want[fin])
    assert np.array_equal(np.isinf(got), np.isinf(want)) and np.array_equal(np.isnan(got), np.isnan(want))


def test_f16_element_map_exhaustive(orc):
    xv = FIN16.view(np.float16).astype(np.float64)
    sign = ((FIN16 >> 15) & 1).astype(np.uint8)
    for s in range(1, 255):
        m = np.minimum(np.abs(np.ldexp(xv, 127 - s)), 7.0)
        d = np.abs(m[:, None] - E2M1_MAG[None, :])
        dmin = d.min(axis=1, keepdims=True)
        w = np.where(np.arange(8) % 2 == 0, 2, 1)[None, :]
        want = (sign << 3) | np.argmax((d == dmin) * w, axis=1).astype(np.uint8)
        got = orc.e2m1_encode_f16_many(FIN16, s)
        assert np.array_equal(got, want), s
    assert not orc.e2m1_encode_f16_many(FIN16, 0).any()


def test_f16_quantize_is_blockwise_steps(orc):
    x = W.dense_activation(11, 64, 256).to(__import__("torch").float16)
    h = x.view(__import__("torch").int16).numpy().view(np.uint16)
    codes, flat = orc.quantize_flat_f16(h)
    xv = h.view(np.float16).astype(np.float64)
    nib = np.zeros((64, 256), np.uint8)
    nib[:, 0::2] = codes & 0xF
    nib[:, 1::2] = codes >> 4
    for r in range(0, 64, 5):
        for b in range(8):
            vmax = np.abs(xv[r, b * 32:(b + 1) * 32]).max()
            s = orc.e8m0_scale(vmax)
            assert flat[r, b] == s
            assert np.array_equal(nib[r, b * 32:(b + 1) * 32],
                                  orc.e2m1_encode_f16_many(h[r, b * 32:(b + 1) * 32], s))


def test_f16_and_bf16_agree_on_shared_values(orc):
    """Values exactly representable in both formats quantize identically."""
    import torch
    x = W.dense_activation(12, 128, 512).float()
    x = torch.where(x.abs() < 2.0 ** -14, torch.zeros_like(x), x).to(torch.bfloat16)
    x16 = x.to(torch.float16)                            # FP16 normals hold any BF16 value exactly
    assert torch.equal(x16.to(torch.bfloat16), x)        # every value survives the round trip
    cb, sb = orc.quantize(W.bf16_bits(x))
    ch, sh = orc.quantize_f16(x16.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(cb, ch) and np.array_equal(sb, sh)


def test_f16_grouped_forms_compose(orc):
    """FP16 grouped quantize equals the FP16 dense quantize of every segment;
    the FP16 gather and scatter forms equal the FP16 grouped quantize of the
    permuted matrix (the composition the BF16 forms are pinned by)."""
    import torch
    g = W.moe_grouped(seed=4, tokens=70, top_k=3, num_experts=6, K=96)
    xt = g.x_tokens.float().to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    idx = g.row_index.numpy()
    dst = g.dest_rows.numpy()
    off = g.offsets.numpy()
    xs = xt[idx]
    rc, c, s, sro = orc.quantize_grouped(xs, off, f16=True)
    assert rc == 0
    pk = 4
    for e in range(6):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            c_e, s_e = orc.quantize_f16(xs[a:b])
            assert np.array_equal(c[a:b], c_e)
            assert np.array_equal(s[sro[e] * pk:sro[e] * pk + s_e.size], s_e)
    rc2, c2, s2, sro2 = orc.quantize_grouped_gather(xt, idx, off, f16=True)
    rc3, c3, s3, sro3 = orc.quantize_grouped_scatter(xt, dst, off, idx.size, f16=True)
    assert rc2 == rc3 == 0
    for a_, b_ in ((c, c2), (s, s2), (c, c3), (s, s3), (sro, sro2), (sro, sro3)):
        assert np.array_equal(a_, b_)
    # and FP16 differs from reading the same bits as BF16 (the flag is live)
    rc4, c4, _, _ = orc.quantize_grouped(xs, off)
    assert not np.array_equal(c, c4)
