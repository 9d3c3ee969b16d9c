"""Seeded random cases across every quantize form, each compared with the
oracle byte for byte: random row counts, K, row strides, 16- versus 32-byte
alignment, BF16 / FP16, expert segment sizes (empty ones included), routings
with dropped routes, top_k, and NVFP4 global scales.  MXFP4_FUZZ_SCALE=n
(default 1) runs n times as many seeds of each kind."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

SCALE = max(1, int(os.environ.get("MXFP4_FUZZ_SCALE", "1")))


@pytest.fixture(scope="module")
def mx():
    assert torch.cuda.is_available()
    import mxfp4_block_quantization_gb300 as m
    return m


def _bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _place(x, rng):
    """x in a buffer with a random extra row stride and a 16- or 32-byte
    aligned base."""
    M, K = x.shape
    pad = int(rng.integers(0, 3)) * 8
    off = int(rng.integers(0, 2)) * 8
    buf = torch.zeros(M * (K + pad) + off + 8, dtype=x.dtype, device="cuda")
    y = buf[off:off + M * (K + pad)].view(M, K + pad)[:, :K]
    y.copy_(x)
    return y


def _random_x(rng, M, K, f16):
    x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32))
    x = x * torch.exp2(torch.from_numpy(rng.uniform(-10, 10, (M, 1)).astype(np.float32)))
    return x.to(torch.float16 if f16 else torch.bfloat16).cuda()


@pytest.mark.parametrize("seed", range(12 * SCALE))
def test_fuzz_dense(mx, seed):
    rng = np.random.default_rng(100 + seed)
    M, K = int(rng.integers(1, 700)), 32 * int(rng.integers(1, 100))
    f16 = bool(seed % 3 == 0)
    x = _place(_random_x(rng, M, K, f16), rng)
    c, s = mx.quantize(x)
    c_o, s_o = (oracle.quantize_f16 if f16 else oracle.quantize)(_bits(x))
    assert np.array_equal(c.cpu().numpy(), c_o) and np.array_equal(s.cpu().numpy(), s_o), (M, K)
    if not f16:
        # into a 32-byte (wide kernel) or a 16-byte aligned output (narrow kernel)
        flat = torch.full((M * K + 16,), 7.0, dtype=torch.bfloat16, device="cuda")
        y = flat[8 * (seed % 2):][:M * K].view(M, K)
        mx.mxfp4_dequantize(c, s, M, K, y)
        assert np.array_equal(_bits(y), oracle.dequantize(c_o, s_o, M, K))


def _random_offsets(rng, E, total):
    cuts = np.sort(rng.integers(0, total + 1, E - 1))
    cuts[rng.random(E - 1) < 0.2] = cuts[0] if E > 1 else 0  # some empty segments
    cuts = np.sort(cuts)
    return np.concatenate([[0], cuts, [total]]).astype(np.int32)


@pytest.mark.parametrize("seed", range(8 * SCALE))
def test_fuzz_grouped_gather_scatter(mx, seed):
    rng = np.random.default_rng(200 + seed)
    T, top_k = int(rng.integers(1, 400)), int(rng.integers(1, 13))
    K = 32 * int(rng.integers(1, 60))
    E = int(rng.integers(1, 40))
    f16 = bool(seed % 2)
    xt = _random_x(rng, T, K, f16)
    # routing: every route a distinct row; 15 % of routes dropped
    total = T * top_k
    perm = rng.permutation(total).astype(np.int32)
    dest = perm.reshape(T, top_k).copy()
    drop = rng.random((T, top_k)) < 0.15
    dest[drop] = -1
    row_tok = np.full(total, -1, np.int32)
    for t in range(T):
        for j in range(top_k):
            if dest[t, j] >= 0:
                row_tok[dest[t, j]] = t
    off = _random_offsets(rng, E, total)
    xb = _bits(xt)
    xp = _place(xt, rng)
    off_d = torch.from_numpy(off).cuda()
    # scatter: untargeted rows keep the prefill
    nsb = mx.mxfp4_grouped_scale_bytes_bound(total, E, K)
    c0 = rng.integers(0, 256, (total, K // 2), dtype=np.uint8)
    s0 = rng.integers(0, 256, nsb, dtype=np.uint8)
    rc, c_o, s_o, sro_o = oracle.quantize_grouped_scatter(xb, dest, off, total, c0, s0, f16=f16)
    for staged in (False, True):                       # per-route scale words / workspace
        codes = torch.from_numpy(c0).cuda()
        scales = torch.from_numpy(s0).cuda()
        sro = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        st = torch.empty(1, dtype=torch.int32, device="cuda")
        args = (xp, torch.from_numpy(dest).cuda(), off_d, total)
        if staged:
            ws = torch.empty(mx.mxfp4_scatter_workspace_bytes(T, total, E, K), dtype=torch.uint8,
                             device="cuda")
            fn = (mx.mxfp4_quantize_grouped_scatter_ws_f16 if f16
                  else mx.mxfp4_quantize_grouped_scatter_ws)
            fn(*args, ws, codes, scales, sro, st)
        else:
            fn = mx.mxfp4_quantize_grouped_scatter_f16 if f16 else mx.mxfp4_quantize_grouped_scatter
            fn(*args, codes, scales, sro, st)
        torch.cuda.synchronize()
        assert int(st.item()) == rc == 0, staged
        assert np.array_equal(codes.cpu().numpy(), c_o), staged
        assert np.array_equal(scales.cpu().numpy(), s_o), staged
    # the NVFP4 experts quant of the same routing, a global scale per expert:
    # all distinct, one shared by every expert, or a few values repeated (a
    # token whose experts share one scale computes its bytes once)
    gs = (448.0 * 6.0 / np.exp(rng.uniform(-3, 8, E))).astype(np.float32)
    if seed % 3 == 1:
        gs[:] = gs[0]
    elif seed % 3 == 2:
        gs = gs[rng.integers(0, min(3, E), E)]
    nsb_nv = mx.mxfp4_nvfp4_grouped_scale_bytes_bound(total, E, K)
    s0_nv = rng.integers(0, 256, nsb_nv, dtype=np.uint8)
    rc_nv, cn_o, sn_o, _ = oracle.nvfp4_quantize_grouped_scatter(xb, dest, off, total, gs, c0,
                                                                 s0_nv, f16=f16)
    for staged in (False, True):
        codes = torch.from_numpy(c0).cuda()
        scales = torch.from_numpy(s0_nv).cuda()
        args = (xp, torch.from_numpy(dest).cuda(), off_d, total, torch.from_numpy(gs).cuda())
        if staged:
            ws = torch.empty(max(mx.mxfp4_nvfp4_scatter_workspace_bytes(total, E, K), 16),
                             dtype=torch.uint8, device="cuda")
            fn = (mx.mxfp4_quantize_nvfp4_grouped_scatter_ws_f16 if f16
                  else mx.mxfp4_quantize_nvfp4_grouped_scatter_ws)
            fn(*args, ws, codes, scales, sro, st)
        else:
            fn = (mx.mxfp4_quantize_nvfp4_grouped_scatter_f16 if f16
                  else mx.mxfp4_quantize_nvfp4_grouped_scatter)
            fn(*args, codes, scales, sro, st)
        torch.cuda.synchronize()
        assert int(st.item()) == rc_nv == 0, staged
        assert np.array_equal(codes.cpu().numpy(), cn_o), staged
        assert np.array_equal(scales.cpu().numpy(), sn_o), staged
    # gather (both kernels): dropped rows have index -1 -> zero rows, EINDEX
    rc_g, cg_o, sg_o, _ = oracle.quantize_grouped_gather(xb, row_tok, off, f16=f16)
    used = int(sro_o[-1]) * ((K // 32 + 3) // 4 * 4)
    for via in (True, False):
        c, s, r, stt = mx.quantize_grouped_gather(xp, torch.from_numpy(row_tok).cuda(), off_d,
                                                  via_scatter=via)
        torch.cuda.synchronize()
        assert int(stt.item()) == rc_g
        assert np.array_equal(c.cpu().numpy(), cg_o), via
        assert np.array_equal(s[:used].cpu().numpy(), sg_o[:used]), via


@pytest.mark.parametrize("seed", range(6 * SCALE))
def test_fuzz_nvfp4(mx, seed):
    rng = np.random.default_rng(300 + seed)
    M, K = int(rng.integers(1, 500)), 16 * int(rng.integers(1, 120))
    f16 = bool(seed % 2 == 1)
    x = _place(_random_x(rng, M, K, f16), rng)
    g = float(np.float32(448.0 * 6.0 / np.exp(rng.uniform(-3, 8))))
    g_t = torch.tensor([g], device="cuda")
    c, s = mx.quantize_nvfp4(x, g_t)
    c_o, s_o = oracle.nvfp4_quantize(_bits(x), g, f16=f16)
    assert np.array_equal(c.cpu().numpy(), c_o) and np.array_equal(s.cpu().numpy(), s_o)
    # its dequantize, into a 32-byte (wide kernel) or a 16-byte aligned output
    flat = torch.full((M * K + 16,), 7.0, dtype=torch.bfloat16, device="cuda")
    y = flat[8 * (seed % 2):][:M * K].view(M, K)
    mx.mxfp4_dequantize_nvfp4(c, s, g_t, M, K, y)
    y_o = oracle.nvfp4_dequantize(c_o, s_o, M, K, g)
    assert np.array_equal(_bits(y), y_o)
    if M > 1 and x.is_contiguous() and x.data_ptr() % 16 == 0:
        E = int(rng.integers(1, 9))
        off = _random_offsets(rng, E, M)
        gs = (448.0 * 6.0 / np.exp(rng.uniform(-3, 8, E))).astype(np.float32)
        cg, sg, sro, st = mx.quantize_nvfp4_grouped(x, torch.from_numpy(off).cuda(),
                                                    torch.from_numpy(gs).cuda())
        rc, cg_o, sg_o, sro_o = oracle.nvfp4_quantize_grouped(_bits(x), off, gs, f16=f16)
        torch.cuda.synchronize()
        assert int(st.item()) == rc == 0
        used = int(sro_o[-1]) * ((K // 16 + 3) // 4 * 4)
        assert np.array_equal(cg.cpu().numpy(), cg_o)
        assert np.array_equal(sg[:used].cpu().numpy(), sg_o[:used])


@pytest.mark.parametrize("seed", range(8 * SCALE))
def test_fuzz_route(mx, seed):
    """Random routings: token count, top_k, number of experts (up to the
    largest the call accepts), skewed expert popularity, dropped routes and
    ids outside [0, E); offsets, token -> rows, row -> token and the status
    word against the oracle, guard words after every output untouched."""
    rng = np.random.default_rng(900 + seed)
    T = int(rng.integers(0, 3000))
    k = int(rng.integers(1, 65))  # past 32 too: the routing call takes any top_k
    E = int(rng.choice([1, 2, 7, 64, 384, 1000, mx.MXFP4_ROUTE_MAX_EXPERTS]))
    popular = rng.zipf(1.5, (T, k)) - 1 if seed % 2 else rng.integers(0, E, (T, k))
    ids = (np.asarray(popular) % E).astype(np.int32)
    ids[rng.random((T, k)) < 0.05] = -1
    if seed % 4 == 3 and ids.size:
        ids.flat[int(rng.integers(0, ids.size))] = E + int(rng.integers(0, 5))  # invalid id
    with_rows = seed % 3 != 2
    g = torch.full((E + 1 + 64,), -5, dtype=torch.int32, device="cuda")
    dest = torch.full((T * k + 64,), -5, dtype=torch.int32, device="cuda")
    rows = torch.full((T * k + 64,), -5, dtype=torch.int32, device="cuda")
    st = torch.full((1,), -5, dtype=torch.int32, device="cuda")
    ws = torch.full((max(mx.mxfp4_route_workspace_bytes(T, k, E), 16),), 0x5A,
                    dtype=torch.uint8, device="cuda")
    mx.mxfp4_moe_route(torch.from_numpy(ids).cuda().view(T, k), E, ws, g[:E + 1],
                       dest[:T * k].view(T, k), rows[:T * k] if with_rows else None, st)
    torch.cuda.synchronize()
    rc, off_o, dest_o, rows_o = oracle.moe_route(ids, E)
    off_g, dest_g, rows_g = g.cpu().numpy(), dest.cpu().numpy(), rows.cpu().numpy()
    assert int(st.item()) == rc, (T, k, E)
    assert np.array_equal(off_g[:E + 1], off_o) and (off_g[E + 1:] == -5).all()
    assert np.array_equal(dest_g[:T * k].reshape(T, k), dest_o) and (dest_g[T * k:] == -5).all()
    n = int(off_o[-1])
    if with_rows:
        assert np.array_equal(rows_g[:n], rows_o) and (rows_g[n:] == -5).all()
    else:
        assert (rows_g == -5).all()


@pytest.mark.parametrize("seed", range(6 * SCALE))
def test_fuzz_swap_w13(mx, seed):
    """Random swaps: experts, 2N (even), K, flat or tiled scales, each bias
    present or absent (the w13 bias with non-finite and tie-rounding values);
    every output byte against the oracle, guard bytes after each output
    untouched."""
    rng = np.random.default_rng(1300 + seed)
    E = int(rng.integers(1, 9))
    two_n = 2 * int(rng.integers(1, 160))
    K = 32 * int(rng.integers(1, 70))
    tiled = int(seed % 2)
    codes = rng.integers(0, 256, (E, two_n, K // 2), dtype=np.uint16).astype(np.uint8)
    flat = rng.integers(0, 256, (E, two_n, K // 32), dtype=np.uint16).astype(np.uint8)
    scales = np.concatenate([oracle.tile(flat[e]) for e in range(E)]) if tiled else flat
    b13 = rng.standard_normal((E, two_n)).astype(np.float32) if seed % 3 != 1 else None
    if b13 is not None:
        b13.flat[0] = np.inf
        b13.flat[-1] = np.float32(1.0 + 2.0 ** -8)          # a BF16 tie: rounds to even
    b2 = rng.standard_normal(int(rng.integers(1, 3000))).astype(np.float32) if seed % 3 != 2 else None
    want = oracle.swap_w13(codes, scales, b13, E, two_n, K, tiled, b2)
    G = 64
    c_out = torch.full((codes.size + G,), 0xA5, dtype=torch.uint8, device="cuda")
    s_out = torch.full((scales.size + G,), 0xA5, dtype=torch.uint8, device="cuda")
    b13_out = torch.full((E * two_n + G,), 0x7E7E, dtype=torch.int16, device="cuda")
    b2_out = torch.full(((b2.size if b2 is not None else 0) + G,), 0x7E7E, dtype=torch.int16,
                        device="cuda")
    mx.mxfp4_swap_w13(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(),
                      torch.from_numpy(b13).cuda() if b13 is not None else None,
                      E, two_n, K, tiled, c_out[:codes.size], s_out[:scales.size],
                      b13_out[:E * two_n].view(torch.bfloat16) if b13 is not None else None,
                      torch.from_numpy(b2).cuda() if b2 is not None else None,
                      b2_out[:b2.size].view(torch.bfloat16) if b2 is not None else None)
    torch.cuda.synchronize()
    c, s = c_out.cpu().numpy(), s_out.cpu().numpy()
    assert np.array_equal(c[:codes.size], want[0].reshape(-1)) and (c[codes.size:] == 0xA5).all()
    assert np.array_equal(s[:scales.size], want[1].reshape(-1)) and (s[scales.size:] == 0xA5).all()
    b13g = b13_out.cpu().numpy().view(np.uint16)
    if b13 is not None:
        assert np.array_equal(b13g[:E * two_n], want[2].reshape(-1))
    assert (b13g[E * two_n if b13 is not None else 0:] == 0x7E7E).all()
    if b2 is not None:
        b2g = b2_out.cpu().numpy().view(np.uint16)
        assert np.array_equal(b2g[:b2.size], want[3].reshape(-1)) and (b2g[b2.size:] == 0x7E7E).all()
