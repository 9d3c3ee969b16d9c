"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle,
element by element, bit-exact for codes, every tiled scale byte (pad
included) and dequantized BF16.  Output buffers carry 0xA5 guard bands that
must survive every call."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 256  # bytes of 0xA5 on each side of every output


@pytest.fixture(scope="module")
def mx():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mxfp4_block_quantization_gb300 as m
    return m


# The full MoE batch (16384 tokens x top-8 over 384 experts, K = 7168; the
# grouped workload at its benchmark size) and the oracle's results for it,
# computed once per module with the unchanged single-threaded routines on
# ranges of experts over all host cores.
@pytest.fixture(scope="module")
def moe():
    return W.moe_grouped(seed=2, device="cuda")


@pytest.fixture(scope="module")
def moe_oracle(moe):
    rc, c, s, sro = oracle.quantize_grouped_threads(bits(moe.x), moe.offsets.cpu().numpy())
    assert rc == 0
    return c, s, sro


@pytest.fixture(scope="module")
def moe_nvfp4_oracle(moe):
    gs = _expert_gscales(moe.num_experts, 2)
    rc, c, s, sro = oracle.nvfp4_quantize_grouped_threads(bits(moe.x), moe.offsets.cpu().numpy(),
                                                          gs)
    assert rc == 0
    return gs, c, s, sro


def assert_full(got, want, what):
    """Every byte of a full-size output equal to the oracle's."""
    assert got.shape == want.shape, what
    assert np.array_equal(got, want), f"{what}: {_first_diff(got, want)}"


class Guarded:
    """A uint8 (or other dtype) device buffer framed by 0xA5 guard bands."""

    def __init__(self, nbytes, dtype=torch.uint8, shape=None):
        self.raw = torch.full((nbytes + 2 * GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
        self.nbytes = nbytes
        inner = self.raw[GUARD:GUARD + nbytes]
        self.t = inner.view(dtype)
        if shape is not None:
            self.t = self.t.view(shape)

    def check(self):
        head = self.raw[:GUARD].cpu().numpy()
        tail = self.raw[GUARD + self.nbytes:].cpu().numpy()
        assert (head == 0xA5).all() and (tail == 0xA5).all(), "guard band overwritten"


def bits(t):
    return W.bf16_bits(t)


def run_quantize(mx, x):
    M, K = x.shape
    codes = Guarded(M * (K // 2), shape=(M, K // 2))
    sb = mx.mxfp4_scale_bytes(M, K)
    scales = Guarded(sb)
    mx.mxfp4_quantize(x, codes.t, scales.t)
    torch.cuda.synchronize()
    codes.check()
    scales.check()
    return codes.t.cpu().numpy(), scales.t.cpu().numpy()


def run_dequantize(mx, codes, scales, M, K):
    y = Guarded(M * K * 2, torch.bfloat16, (M, K))
    mx.mxfp4_dequantize(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), M, K, y.t)
    torch.cuda.synchronize()
    y.check()
    return bits(y.t)


def assert_quant_parity(mx, x_dev):
    xb = bits(x_dev)
    M, K = xb.shape
    c_gpu, s_gpu = run_quantize(mx, x_dev)
    c_orc, s_orc = oracle.quantize(xb)
    assert np.array_equal(c_gpu, c_orc), _first_diff(c_gpu, c_orc)
    assert np.array_equal(s_gpu, s_orc), _first_diff(s_gpu, s_orc)
    y_gpu = run_dequantize(mx, c_gpu, s_gpu, M, K)
    y_orc = oracle.dequantize(c_orc, s_orc, M, K)
    assert np.array_equal(y_gpu, y_orc), _first_diff(y_gpu, y_orc)
    return c_orc, s_orc, y_orc


def _first_diff(a, b):
    idx = np.argwhere(a != b)
    if idx.size == 0:
        return "equal"
    i = tuple(idx[0])
    return f"{idx.shape[0]} mismatches, first at {i}: got {a[i]:#x} want {b[i]:#x}"


def rel_l2(xb, yb):
    x = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y = (yb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return float(np.linalg.norm(y - x) / np.linalg.norm(x))


# ------------------------------------------------------------------ dense
def test_small_matrix_128x256(mx):
    x = W.small_matrix(0).cuda()
    assert_quant_parity(mx, x)


def test_edge_cases_1000x2880(mx):
    x = W.edge_cases(4).cuda()
    c, s, y = assert_quant_parity(mx, x)
    print("edge-case rel-L2", rel_l2(bits(x), y))


def test_dense_activation_4096x7168(mx):
    x = W.dense_activation(1, device="cuda")
    c, s, y = assert_quant_parity(mx, x)
    print("dense rel-L2", rel_l2(bits(x), y))


@pytest.mark.parametrize("M", [1, 31, 127, 128, 129, 300])
@pytest.mark.parametrize("K", [32, 96, 160, 2880])
def test_ragged_shapes(mx, M, K):
    x = W.normal_bf16((M, K), seed=M * 1000 + K, device="cuda")
    assert_quant_parity(mx, x)


def test_strided_input(mx):
    """Row stride larger than K (a column slice of a wider matrix)."""
    wide = W.dense_activation(5, 300, 1024, device="cuda")
    x = wide[:, 128:128 + 640]
    assert x.stride(0) == 1024
    c_gpu, s_gpu = run_quantize(mx, x)
    c_orc, s_orc = oracle.quantize(bits(x.contiguous()))
    assert np.array_equal(c_gpu, c_orc) and np.array_equal(s_gpu, s_orc)


def test_empty(mx):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    codes, scales = mx.quantize(x)
    assert codes.numel() == 0 and scales.numel() == 0


def test_element_map_exhaustive(mx):
    """Every finite BF16 value under every reachable scale exponent: block b
    holds a max that fixes s (2^(s-125), or 0x7F7F for s = 253) followed by
    31 values of magnitude <= that max, enumerating all such BF16 patterns."""
    finite = np.arange(0x0000, 0x7F80, dtype=np.uint16)           # positive finite
    rows = []
    for s in range(1, 254):
        vmax = (s + 2) << 7 if s <= 252 else 0x7F7F                # bits of 2^(s-125)
        vals = finite[finite <= vmax]
        vals = np.concatenate([vals, vals | 0x8000])               # both signs
        pad = (-vals.size) % 31
        vals = np.concatenate([vals, np.zeros(pad, np.uint16)]).reshape(-1, 31)
        blocks = np.concatenate([np.full((vals.shape[0], 1), vmax, np.uint16), vals], axis=1)
        rows.append(blocks)
    blocks = np.concatenate(rows)
    pad = (-blocks.shape[0]) % 32
    blocks = np.concatenate([blocks, np.zeros((pad, 32), np.uint16)])
    xb = blocks.reshape(-1, 32 * 32)                               # K = 1024
    x = W.from_bits(xb, "cuda")
    c_gpu, s_gpu = run_quantize(mx, x)
    c_orc, s_orc = oracle.quantize(xb)
    assert np.array_equal(s_gpu, s_orc), _first_diff(s_gpu, s_orc)
    assert np.array_equal(c_gpu, c_orc), _first_diff(c_gpu, c_orc)


def test_dequant_all_codes_all_scales(mx):
    """All 16 codes x all 256 scale bytes (including 0 and the NaN 255)."""
    M, K = 256, 256                       # 2048 blocks: 8 per row
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 256, (M, K // 2), dtype=np.uint16).astype(np.uint8)
    codes[:16, :] = np.arange(256, dtype=np.uint16).astype(np.uint8)[None, :128]
    flat = (np.arange(M * (K // 32)) % 256).astype(np.uint8).reshape(M, K // 32)
    tiled = oracle.tile(flat)
    y_gpu = run_dequantize(mx, codes, tiled, M, K)
    y_orc = oracle.dequantize(codes, tiled, M, K)
    assert np.array_equal(y_gpu, y_orc), _first_diff(y_gpu, y_orc)


# ---------------------------------------------------------------- grouped
def run_grouped(mx, x, offsets):
    total, K = x.shape
    E = offsets.numel() - 1
    codes = Guarded(total * (K // 2), shape=(total, K // 2))
    bound = mx.mxfp4_grouped_scale_bytes_bound(total, E, K)
    scales = Guarded(bound)
    sro = Guarded(4 * (E + 1), torch.int32)
    status = Guarded(4, torch.int32)
    mx.mxfp4_quantize_grouped(x, offsets, codes.t, scales.t, sro.t, status.t)
    torch.cuda.synchronize()
    for g in (codes, scales, sro, status):
        g.check()
    return (codes.t.cpu().numpy(), scales.t.cpu().numpy(), sro.t.cpu().numpy(),
            int(status.t.cpu()[0]))


def test_grouped_small(mx):
    g = W.moe_grouped(seed=2, tokens=200, top_k=4, num_experts=12, K=288, device="cuda")
    c, s, sro, st = run_grouped(mx, g.x, g.offsets)
    rc, c_o, s_o, sro_o = oracle.quantize_grouped(bits(g.x), g.offsets.cpu().numpy())
    assert st == 0 and rc == 0
    assert np.array_equal(sro, sro_o)
    assert np.array_equal(c, c_o)
    pk = (288 // 32 + 3) // 4 * 4
    used = int(sro_o[-1]) * pk
    assert np.array_equal(s[:used], s_o[:used])
    assert (s[used:] == 0xA5).all(), "slack past P[E] must be untouched"


def test_grouped_empty_and_uniform_segments(mx):
    x = W.small_matrix(3, 512, 256).cuda()
    for off in ([0, 0, 130, 130, 130, 512, 512], [0, 128, 256, 384, 512], [0, 512]):
        o = torch.tensor(off, dtype=torch.int32, device="cuda")
        c, s, sro, st = run_grouped(mx, x, o)
        rc, c_o, s_o, sro_o = oracle.quantize_grouped(bits(x), np.array(off, np.int32))
        assert st == 0 and np.array_equal(sro, sro_o) and np.array_equal(c, c_o)
        used = int(sro_o[-1]) * 8
        assert np.array_equal(s[:used], s_o[:used])


@pytest.mark.parametrize("off", [[1, 10, 20], [0, 12, 8, 20], [0, 10, 19], [0, 10, 21]])
def test_grouped_bad_offsets(mx, off):
    x = W.small_matrix(3, 20, 64).cuda()
    o = torch.tensor(off, dtype=torch.int32, device="cuda")
    c, s, sro, st = run_grouped(mx, x, o)
    assert st == mx.MXFP4_EOFFSETS
    assert (sro == -1).all()
    assert (c == 0xA5).all() and (s == 0xA5).all(), "outputs must stay untouched"


def test_grouped_moe_full_size(mx, moe, moe_oracle):
    """131072 rows (16384 tokens x top-8 over 384 experts), K = 7168, against
    the oracle in full: every code byte, every scale byte of the 147,968
    padded rows (pad rows and pad columns included), every padded offset; the
    bound's slack past the last padded row and the guard bands untouched."""
    x, off = moe.x, moe.offsets
    total, K = x.shape
    E = off.numel() - 1
    bound = mx.mxfp4_grouped_scale_bytes_bound(total, E, K)
    codes = Guarded(total * (K // 2), shape=(total, K // 2))
    scales = Guarded(bound)
    sro = Guarded(4 * (E + 1), torch.int32)
    st = Guarded(4, torch.int32)
    mx.mxfp4_quantize_grouped(x, off, codes.t, scales.t, sro.t, st.t)
    torch.cuda.synchronize()
    for g in (codes, scales, sro, st):
        g.check()
    assert int(st.t.item()) == 0
    c_o, s_o, sro_o = moe_oracle
    assert_full(sro.t.cpu().numpy(), sro_o, "scale row offsets")
    assert_full(codes.t.cpu().numpy(), c_o, "codes")
    s_h = scales.t.cpu().numpy()
    assert_full(s_h[:s_o.size], s_o, "tiled scales")
    assert (s_h[s_o.size:] == 0xA5).all(), "slack past the last padded row was written"


def test_grouped_moe_full_size_dequantize(mx, moe, moe_oracle):
    """The dequantize of every expert segment of the full MoE batch (each
    segment its own matrix with its own tiled scales), all 131072 x 7168
    BF16 outputs against the oracle's dequantize of the same segments."""
    c_o, s_o, sro_o = moe_oracle
    total, K = moe.x.shape
    off_h = moe.offsets.cpu().numpy().astype(np.int64)
    pk = (K // 32 + 3) // 4 * 4
    codes = torch.from_numpy(c_o).cuda()
    scales = torch.from_numpy(s_o).cuda()
    y = Guarded(total * K * 2, torch.bfloat16, (total, K))
    E = off_h.size - 1
    for e in range(E):
        a, b = int(off_h[e]), int(off_h[e + 1])
        if b > a:
            p0 = int(sro_o[e]) * pk
            mx.mxfp4_dequantize(codes[a:b], scales[p0:p0 + mx.mxfp4_scale_bytes(b - a, K)],
                                b - a, K, y.t[a:b])
    torch.cuda.synchronize()
    y.check()
    want = np.zeros((total, K), np.uint16)

    def seg(e0, e1):
        for e in range(e0, e1):
            a, b = int(off_h[e]), int(off_h[e + 1])
            p0 = int(sro_o[e]) * pk
            want[a:b] = oracle.dequantize(c_o[a:b], s_o[p0:p0 + oracle.scale_bytes(b - a, K)],
                                          b - a, K)
    step = -(-E // oracle.host_threads())
    oracle._run_parts(seg, [(e, min(E, e + step)) for e in range(0, E, step)])
    assert_full(bits(y.t), want, "dequantized BF16")


# ------------------------------------------------------------------- swap
def run_swap(mx, codes, scales, b13, b2, E, two_n, K, tiled):
    c_in = torch.from_numpy(codes).cuda()
    s_in = torch.from_numpy(scales).cuda()
    b13_in = torch.from_numpy(b13).cuda() if b13 is not None else None
    b2_in = torch.from_numpy(b2).cuda() if b2 is not None else None
    c_out = Guarded(codes.size, shape=codes.shape)
    s_out = Guarded(scales.size, shape=scales.shape)
    b13_out = Guarded(b13.size * 2, torch.bfloat16, b13.shape) if b13 is not None else None
    b2_out = Guarded(b2.size * 2, torch.bfloat16, b2.shape) if b2 is not None else None
    mx.mxfp4_swap_w13(c_in, s_in, b13_in, E, two_n, K, tiled, c_out.t, s_out.t,
                      b13_out.t if b13_out else None, b2_in, b2_out.t if b2_out else None)
    torch.cuda.synchronize()
    for g in (c_out, s_out, b13_out, b2_out):
        if g is not None:
            g.check()
    return (c_out.t.cpu().numpy(), s_out.t.cpu().numpy(),
            bits(b13_out.t) if b13_out else None, bits(b2_out.t) if b2_out else None)


@pytest.mark.parametrize("tiled", [0, 1])
@pytest.mark.parametrize("E,two_n,K", [(3, 200, 160), (2, 256, 2048), (1, 4, 64), (5, 130, 2880)])
def test_swap_matches_oracle(mx, tiled, E, two_n, K):
    rng = np.random.default_rng(E * 100 + two_n + K)
    codes = rng.integers(0, 256, (E, two_n, K // 2), dtype=np.uint16).astype(np.uint8)
    flat = rng.integers(0, 256, (E, two_n, K // 32), dtype=np.uint16).astype(np.uint8)
    scales = np.concatenate([oracle.tile(flat[e]) for e in range(E)]) if tiled else flat
    b13 = rng.standard_normal((E, two_n)).astype(np.float32)
    b2 = rng.standard_normal((E, 37)).astype(np.float32)
    got = run_swap(mx, codes, scales, b13, b2, E, two_n, K, tiled)
    want = oracle.swap_w13(codes, scales, b13, E, two_n, K, tiled, b2)
    for g, w in zip(got, want):
        assert np.array_equal(g, w), _first_diff(g, w)


def test_swap_page_arange_layout(mx):
    """The PR #51038 test tensors in this library's layout: E = 1, 2N = 4,
    K = 64 (flat scales [1, 4, 2] = arange(8)); rows become (2, 3, 0, 1)."""
    codes = np.arange(128, dtype=np.uint8).reshape(1, 4, 32)
    scales = np.arange(8, dtype=np.uint8).reshape(1, 4, 2)
    b = np.arange(4, dtype=np.float32).reshape(1, 4)
    c, s, b13, b2 = run_swap(mx, codes, scales, b, b.copy(), 1, 4, 64, 0)
    assert np.array_equal(c[0], codes[0][[2, 3, 0, 1]])
    assert s.tolist() == [[[4, 5], [6, 7], [0, 1], [2, 3]]]
    assert b13.tolist() == [[0x4000, 0x4040, 0x0000, 0x3F80]]
    assert b2.tolist() == [[0x0000, 0x3F80, 0x4000, 0x4040]]


def test_expert_weights_full_size(mx):
    """128 experts: w13 [128, 1536, 2048] and w2 [128, 2048, 768] quantized
    as dense [E*rows, K] matrices (each expert a whole number of 128-row
    tiles, so its tiled scales are its own chunks), their dequantize, then
    the w13 swap of codes, tiled scales and both biases: every byte of every
    output against the oracle, guard bands intact."""
    w = W.expert_weights(3, device="cuda")
    E, two_n, H = w.w13.shape
    outs = {}
    for name, xw in (("w13", w.w13.view(E * two_n, H)), ("w2", w.w2.view(-1, w.w2.shape[2]))):
        M, K = xw.shape
        c = Guarded(M * (K // 2), shape=(M, K // 2))
        sc = Guarded(mx.mxfp4_scale_bytes(M, K))
        mx.mxfp4_quantize(xw, c.t, sc.t)
        y = Guarded(M * K * 2, torch.bfloat16, (M, K))
        mx.mxfp4_dequantize(c.t, sc.t, M, K, y.t)
        torch.cuda.synchronize()
        for g in (c, sc, y):
            g.check()
        c_o, s_o = oracle.quantize_threads(bits(xw))
        assert_full(c.t.cpu().numpy(), c_o, f"{name} codes")
        assert_full(sc.t.cpu().numpy(), s_o, f"{name} tiled scales")
        assert_full(bits(y.t), oracle.dequantize_threads(c_o, s_o, M, K), f"{name} dequantize")
        outs[name] = (c.t, sc.t, c_o, s_o)
    c13, s13, c13_o, s13_o = outs["w13"]
    c_sw, s_sw, b13_sw, b2_sw = run_swap(mx, c13_o.reshape(E, two_n, H // 2), s13_o,
                                         w.w13_bias.cpu().numpy(), w.w2_bias.cpu().numpy(), E,
                                         two_n, H, 1)
    want = oracle.swap_w13(c13_o.reshape(E, two_n, H // 2), s13_o, w.w13_bias.cpu().numpy(), E,
                           two_n, H, 1, w.w2_bias.cpu().numpy())
    assert_full(c_sw, want[0], "swapped codes")
    assert_full(s_sw, want[1], "swapped tiled scales")
    assert_full(b13_sw, want[2], "w13 bias (swapped, BF16)")
    assert_full(b2_sw, want[3], "w2 bias (BF16)")


# ------------------------------------------------- fused gather + grouped
def run_gather(mx, x, row_index, offsets):
    total = row_index.numel()
    K = x.shape[1]
    E = offsets.numel() - 1
    codes = Guarded(total * (K // 2), shape=(total, K // 2))
    scales = Guarded(mx.mxfp4_grouped_scale_bytes_bound(total, E, K))
    sro = Guarded(4 * (E + 1), torch.int32)
    status = Guarded(4, torch.int32)
    mx.mxfp4_quantize_grouped_gather(x, row_index, offsets, codes.t, scales.t, sro.t, status.t)
    torch.cuda.synchronize()
    for g in (codes, scales, sro, status):
        g.check()
    return (codes.t.cpu().numpy(), scales.t.cpu().numpy(), sro.t.cpu().numpy(),
            int(status.t.cpu()[0]))


def test_grouped_gather_small(mx):
    g = W.moe_grouped(seed=2, tokens=200, top_k=4, num_experts=12, K=288, device="cuda")
    c, s, sro, st = run_gather(mx, g.x_tokens, g.row_index, g.offsets)
    rc, c_o, s_o, sro_o = oracle.quantize_grouped_gather(bits(g.x_tokens), g.token_of_row.numpy(),
                                                         g.offsets.cpu().numpy())
    assert st == 0 and rc == 0 and np.array_equal(sro, sro_o)
    assert np.array_equal(c, c_o), _first_diff(c, c_o)
    used = int(sro_o[-1]) * 12
    assert np.array_equal(s[:used], s_o[:used])


def test_grouped_gather_strided_source(mx):
    g = W.moe_grouped(seed=5, tokens=150, top_k=2, num_experts=5, K=256, device="cuda")
    wide = torch.zeros((150, 384), dtype=torch.bfloat16, device="cuda")
    wide[:, 64:320] = g.x_tokens
    x = wide[:, 64:320]
    c, s, sro, st = run_gather(mx, x, g.row_index, g.offsets)
    rc, c_o, s_o, sro_o = oracle.quantize_grouped_gather(bits(g.x_tokens), g.token_of_row.numpy(),
                                                         g.offsets.cpu().numpy())
    assert st == 0 and np.array_equal(c, c_o)
    used = int(sro_o[-1]) * 8
    assert np.array_equal(s[:used], s_o[:used])


def test_grouped_gather_bad_index(mx):
    xt = W.small_matrix(3, 16, 64).cuda()
    idx = torch.tensor([0, 5, 99, 7, -1, 3], dtype=torch.int32, device="cuda")
    off = torch.tensor([0, 2, 6], dtype=torch.int32, device="cuda")
    c, s, sro, st = run_gather(mx, xt, idx, off)
    rc, c_o, s_o, sro_o = oracle.quantize_grouped_gather(bits(xt), idx.cpu().numpy(),
                                                         off.cpu().numpy())
    assert st == mx.MXFP4_EINDEX and rc == -7
    assert np.array_equal(c, c_o) and not c[2].any() and not c[4].any()
    used = int(sro_o[-1]) * 4
    assert np.array_equal(s[:used], s_o[:used])


def test_grouped_gather_moe_full_size(mx, moe, moe_oracle):
    """16384 tokens x top-8 over 384 experts, K = 7168: the fused gather
    equals the grouped quantize of the gathered matrix and the oracle, every
    byte."""
    g = moe
    c1, s1, sro1, st1 = mx.quantize_grouped_gather(g.x_tokens, g.row_index, g.offsets)
    c2, s2, sro2, st2 = mx.quantize_grouped(g.x, g.offsets)
    torch.cuda.synchronize()
    assert int(st1.cpu()[0]) == 0 and int(st2.cpu()[0]) == 0
    assert torch.equal(sro1, sro2) and torch.equal(c1, c2)
    used = int(sro1[-1].item()) * 224
    assert torch.equal(s1[:used], s2[:used])
    c_o, s_o, sro_o = moe_oracle
    assert_full(sro1.cpu().numpy(), sro_o, "scale row offsets")
    assert_full(c1.cpu().numpy(), c_o, "codes")
    assert_full(s1[:used].cpu().numpy(), s_o, "tiled scales")


# ------------------------------------------------- fused dispatch scatter
@pytest.fixture(params=[False, True], ids=["direct", "ws"])
def scatter_ws(request):
    """Every scatter case runs both forms: scale words stored per route
    (mxfp4_quantize_grouped_scatter) and staged in a workspace
    (mxfp4_quantize_grouped_scatter_ws)."""
    return request.param


def run_scatter(mx, x, dest, offsets, total, seed=0, ws=False):
    """Scatter form through the C ABI into guard-banded buffers whose inner
    bytes start random (the same bytes go to the oracle, so untouched rows
    and slack compare equal); returns the GPU and oracle results."""
    K = x.shape[1]
    E = offsets.numel() - 1
    rng = np.random.default_rng(seed)
    nsb = mx.mxfp4_grouped_scale_bytes_bound(total, E, K)
    c0 = rng.integers(0, 256, (total, K // 2), dtype=np.uint8)
    s0 = rng.integers(0, 256, nsb, dtype=np.uint8)
    codes = Guarded(total * (K // 2), shape=(total, K // 2))
    scales = Guarded(nsb)
    codes.t.copy_(torch.from_numpy(c0))
    scales.t.copy_(torch.from_numpy(s0))
    sro = Guarded(4 * (E + 1), torch.int32)
    status = Guarded(4, torch.int32)
    guards = [codes, scales, sro, status]
    if ws:
        work = Guarded(max(mx.mxfp4_scatter_workspace_bytes(x.shape[0], total, E, K), 16))
        work.t.fill_(0x5A)                            # contents on entry must not matter
        guards.append(work)
        mx.mxfp4_quantize_grouped_scatter_ws(x, dest, offsets, total, work.t, codes.t, scales.t,
                                             sro.t, status.t)
    else:
        mx.mxfp4_quantize_grouped_scatter(x, dest, offsets, total, codes.t, scales.t, sro.t,
                                          status.t)
    torch.cuda.synchronize()
    for g in guards:
        g.check()
    gpu = (codes.t.cpu().numpy(), scales.t.cpu().numpy(), sro.t.cpu().numpy(),
           int(status.t.cpu()[0]))
    rc, c_o, s_o, sro_o = oracle.quantize_grouped_scatter(
        bits(x.contiguous()), dest.cpu().numpy(), offsets.cpu().numpy(), total, c0, s0)
    return gpu, (c_o, s_o, sro_o, rc)


def assert_scatter_parity(gpu, orc, want_status=0):
    c, s, sro, st = gpu
    c_o, s_o, sro_o, rc = orc
    assert st == want_status and rc == want_status  # the oracle returns the ABI's codes
    assert np.array_equal(sro, sro_o)
    assert np.array_equal(c, c_o), _first_diff(c, c_o)
    assert np.array_equal(s, s_o), _first_diff(s, s_o)


def test_grouped_scatter_small(mx, scatter_ws):
    g = W.moe_grouped(seed=2, tokens=200, top_k=4, num_experts=12, K=288, device="cuda")
    gpu, orc = run_scatter(mx, g.x_tokens, g.dest_rows, g.offsets, g.row_index.numel(),
                           ws=scatter_ws)
    assert_scatter_parity(gpu, orc)
    c_g, s_g, sro_g, _ = run_gather(mx, g.x_tokens, g.row_index, g.offsets)
    used = int(sro_g[-1]) * 12
    assert np.array_equal(gpu[0], c_g) and np.array_equal(gpu[1][:used], s_g[:used])


@pytest.mark.parametrize("tokens,top_k,E,K", [
    (1, 1, 1, 32), (129, 3, 5, 160), (300, 2, 7, 2880), (64, 32, 40, 96), (257, 8, 16, 1056)])
def test_grouped_scatter_shapes(mx, tokens, top_k, E, K, scatter_ws):
    g = W.moe_grouped(seed=tokens + K, tokens=tokens, top_k=top_k, num_experts=E, K=K,
                      device="cuda")
    gpu, orc = run_scatter(mx, g.x_tokens, g.dest_rows, g.offsets, g.row_index.numel(), seed=K,
                           ws=scatter_ws)
    assert_scatter_parity(gpu, orc)


def test_grouped_scatter_dropped_routes(mx, scatter_ws):
    """20 % of the routes not dispatched (-1): their rows keep their previous
    bytes, codes and scale bytes alike; pad rows are zeroed."""
    g = W.moe_grouped(seed=6, tokens=300, top_k=4, num_experts=9, K=160, device="cuda")
    dst = g.dest_rows.clone()
    drop = torch.rand(dst.shape, generator=torch.Generator().manual_seed(1)) < 0.2
    dst[drop.cuda()] = -1
    gpu, orc = run_scatter(mx, g.x_tokens, dst, g.offsets, g.row_index.numel(), seed=3,
                           ws=scatter_ws)
    assert_scatter_parity(gpu, orc)


def test_grouped_scatter_empty_experts_and_no_tokens(mx, scatter_ws):
    x = W.small_matrix(4, 100, 256).cuda()
    off = torch.tensor([0, 0, 130, 130, 200, 200], dtype=torch.int32, device="cuda")
    perm = torch.randperm(200, generator=torch.Generator().manual_seed(2)).to(torch.int32)
    dst = perm.view(100, 2).cuda()
    gpu, orc = run_scatter(mx, x, dst, off, 200, seed=4, ws=scatter_ws)
    assert_scatter_parity(gpu, orc)
    # no tokens at all: every row untargeted, only the pad rows are written
    gpu, orc = run_scatter(mx, x[:0], dst[:0], off, 200, seed=5, ws=scatter_ws)
    assert_scatter_parity(gpu, orc)


def test_grouped_scatter_more_experts_than_shared_memory_holds(mx, scatter_ws):
    """600 experts (most of them empty at 900 routes): above the 511 segments
    the staged form's map CTAs keep in shared memory, so they search the
    offsets in global memory."""
    g = W.moe_grouped(seed=31, tokens=300, top_k=3, num_experts=600, K=96, device="cuda")
    gpu, orc = run_scatter(mx, g.x_tokens, g.dest_rows, g.offsets, g.row_index.numel(), seed=31,
                           ws=scatter_ws)
    assert_scatter_parity(gpu, orc)


def test_grouped_scatter_bad_entries(mx, scatter_ws):
    g = W.moe_grouped(seed=7, tokens=140, top_k=2, num_experts=3, K=64, device="cuda")
    total = g.row_index.numel()
    dst = g.dest_rows.clone()
    dst[3, 1] = total
    dst[7, 0] = -2
    dst[139, 1] = 1 << 30
    gpu, orc = run_scatter(mx, g.x_tokens, dst, g.offsets, total, seed=6, ws=scatter_ws)
    assert orc[3] == -7
    assert_scatter_parity(gpu, orc, want_status=mx.MXFP4_EINDEX)


@pytest.mark.parametrize("off", [[1, 10, 20], [0, 12, 8, 20], [0, 10, 19]])
def test_grouped_scatter_bad_offsets(mx, off, scatter_ws):
    x = W.small_matrix(3, 10, 64).cuda()
    dst = torch.arange(20, dtype=torch.int32, device="cuda").view(10, 2)
    o = torch.tensor(off, dtype=torch.int32, device="cuda")
    gpu, orc = run_scatter(mx, x, dst, o, 20, seed=7, ws=scatter_ws)
    assert orc[3] == -6 and gpu[3] == mx.MXFP4_EOFFSETS
    assert (gpu[2] == -1).all()
    assert np.array_equal(gpu[0], orc[0]) and np.array_equal(gpu[1], orc[1])  # untouched


def test_grouped_scatter_strided_and_16b_aligned(mx, scatter_ws):
    g = W.moe_grouped(seed=8, tokens=150, top_k=3, num_experts=6, K=256, device="cuda")
    wide = torch.zeros((150, 392), dtype=torch.bfloat16, device="cuda")
    wide[:, 8:264] = g.x_tokens
    for x in (wide[:, 8:264], offset16(g.x_tokens)):
        gpu, orc = run_scatter(mx, x, g.dest_rows, g.offsets, g.row_index.numel(), seed=8,
                               ws=scatter_ws)
        assert_scatter_parity(gpu, orc)


def test_grouped_scatter_moe_full_size(mx, moe, moe_oracle):
    """16384 tokens x top-8 over 384 experts, K = 7168: both scatter forms
    equal the fused gather (itself equal to the grouped quantize of the
    gathered matrix), and every byte equals the oracle."""
    g = moe
    c1, s1, sro1, st1 = mx.quantize_grouped_scatter(g.x_tokens, g.dest_rows, g.offsets)
    c2, s2, sro2, st2 = mx.quantize_grouped_gather(g.x_tokens, g.row_index, g.offsets)
    c3, s3, sro3, st3 = mx.quantize_grouped_scatter(g.x_tokens, g.dest_rows, g.offsets,
                                                    staged=False)
    torch.cuda.synchronize()
    assert int(st1.cpu()[0]) == 0 and int(st2.cpu()[0]) == 0 and int(st3.cpu()[0]) == 0
    assert torch.equal(sro1, sro2) and torch.equal(c1, c2) and torch.equal(c1, c3)
    used = int(sro1[-1].item()) * 224
    assert torch.equal(s1[:used], s2[:used]) and torch.equal(s1[:used], s3[:used])
    c_o, s_o, sro_o = moe_oracle
    assert_full(sro1.cpu().numpy(), sro_o, "scale row offsets")
    assert_full(c1.cpu().numpy(), c_o, "codes")
    assert_full(s1[:used].cpu().numpy(), s_o, "tiled scales")


# ----------------------- inputs aligned to 16 bytes but not to 32 bytes
def offset16(x):
    """The same values in a buffer whose base is 16 (not 32) bytes aligned:
    the kernels then take their two-16-byte-load path."""
    flat = torch.empty(x.numel() + 8, dtype=torch.bfloat16, device="cuda")
    y = flat[8:].view(x.shape)
    y.copy_(x)
    assert y.data_ptr() % 32 == 16
    return y


def test_dense_16b_aligned_input(mx):
    x = offset16(W.dense_activation(7, 300, 2880, device="cuda"))
    c_gpu, s_gpu = run_quantize(mx, x)
    c_orc, s_orc = oracle.quantize(bits(x))
    assert np.array_equal(c_gpu, c_orc) and np.array_equal(s_gpu, s_orc)


def test_dense_row_stride_16b(mx):
    """Row stride of 1032 elements (2064 bytes: a multiple of 16, not 32)."""
    wide = W.dense_activation(8, 200, 1032, device="cuda")
    x = wide[:, :1024]
    c_gpu, s_gpu = run_quantize(mx, x)
    c_orc, s_orc = oracle.quantize(bits(x.contiguous()))
    assert np.array_equal(c_gpu, c_orc) and np.array_equal(s_gpu, s_orc)


def test_grouped_16b_aligned_input(mx):
    g = W.moe_grouped(seed=6, tokens=120, top_k=3, num_experts=9, K=160, device="cuda")
    x = offset16(g.x)
    c, s, sro, st = run_grouped(mx, x, g.offsets)
    rc, c_o, s_o, sro_o = oracle.quantize_grouped(bits(g.x), g.offsets.cpu().numpy())
    assert st == 0 and np.array_equal(c, c_o) and np.array_equal(sro, sro_o)
    used = int(sro_o[-1]) * 8
    assert np.array_equal(s[:used], s_o[:used])


def test_grouped_gather_16b_aligned_input(mx):
    g = W.moe_grouped(seed=7, tokens=120, top_k=3, num_experts=9, K=160, device="cuda")
    x = offset16(g.x_tokens)
    c, s, sro, st = run_gather(mx, x, g.row_index, g.offsets)
    rc, c_o, s_o, sro_o = oracle.quantize_grouped_gather(bits(g.x_tokens), g.token_of_row.numpy(),
                                                         g.offsets.cpu().numpy())
    assert st == 0 and np.array_equal(c, c_o)
    used = int(sro_o[-1]) * 8
    assert np.array_equal(s[:used], s_o[:used])


# ------------------------------------------------------------- FP16 input
def f16_bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_quantize_f16(mx, x):
    M, K = x.shape
    codes = Guarded(M * (K // 2), shape=(M, K // 2))
    scales = Guarded(mx.mxfp4_scale_bytes(M, K))
    mx.mxfp4_quantize_f16(x, codes.t, scales.t)
    torch.cuda.synchronize()
    codes.check()
    scales.check()
    return codes.t.cpu().numpy(), scales.t.cpu().numpy()


@pytest.mark.parametrize("M,K", [(4096, 7168), (1000, 2880), (129, 160)])
def test_f16_dense(mx, M, K):
    x = W.dense_activation(13, M, K, device="cuda").float()
    x[::7, ::5] *= 2.0 ** -12                                    # FP16 subnormals too
    x = x.to(torch.float16)
    c, s = run_quantize_f16(mx, x)
    c_o, s_o = oracle.quantize_f16(f16_bits(x))
    assert np.array_equal(c, c_o), _first_diff(c, c_o)
    assert np.array_equal(s, s_o), _first_diff(s, s_o)


def test_f16_16b_aligned_input(mx):
    x = W.dense_activation(14, 200, 1024, device="cuda").to(torch.float16)
    flat = torch.empty(x.numel() + 8, dtype=torch.float16, device="cuda")
    y = flat[8:].view(x.shape)
    y.copy_(x)
    c, s = run_quantize_f16(mx, y)
    c_o, s_o = oracle.quantize_f16(f16_bits(x))
    assert np.array_equal(c, c_o) and np.array_equal(s, s_o)


def test_f16_element_map_exhaustive(mx):
    """Every finite FP16 value under every scale exponent FP16 block maxima
    reach (s = 101..141)."""
    finite = np.arange(0x0000, 0x7C00, dtype=np.uint16)
    rows = []
    for s in range(101, 142):
        e = s - 125                                                   # vmax = 2^e
        if s == 141:
            vmax = 0x7BFF                                             # 65504
        elif e >= -14:
            vmax = (e + 15) << 10
        else:
            vmax = 1 << (e + 24)                                      # subnormal power of two
        vals = finite[finite <= vmax]
        vals = np.concatenate([vals, vals | 0x8000])
        pad = (-vals.size) % 31
        vals = np.concatenate([vals, np.zeros(pad, np.uint16)]).reshape(-1, 31)
        rows.append(np.concatenate([np.full((vals.shape[0], 1), vmax, np.uint16), vals], axis=1))
    blocks = np.concatenate(rows)
    blocks = np.concatenate([blocks, np.zeros(((-blocks.shape[0]) % 32, 32), np.uint16)])
    hb = blocks.reshape(-1, 1024)
    x = torch.from_numpy(hb.view(np.int16)).view(torch.float16).cuda()
    c, s = run_quantize_f16(mx, x)
    c_o, s_o = oracle.quantize_f16(hb)
    assert np.array_equal(s, s_o), _first_diff(s, s_o)
    assert np.array_equal(c, c_o), _first_diff(c, c_o)


# ------------------------------------------------------------------ NVFP4
def run_nvfp4(mx, x, g):
    M, K = x.shape
    gs = torch.tensor([g], dtype=torch.float32, device="cuda")
    codes = Guarded(M * (K // 2), shape=(M, K // 2))
    scales = Guarded(mx.mxfp4_nvfp4_scale_bytes(M, K))
    mx.mxfp4_quantize_nvfp4(x, gs, codes.t, scales.t)
    torch.cuda.synchronize()
    codes.check()
    scales.check()
    c, s = codes.t.cpu().numpy(), scales.t.cpu().numpy()
    y = Guarded(M * K * 2, torch.bfloat16, (M, K))
    mx.mxfp4_dequantize_nvfp4(torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(), gs, M, K, y.t)
    torch.cuda.synchronize()
    y.check()
    return c, s, bits(y.t)


def assert_nvfp4_parity(mx, x, g):
    xb = bits(x)
    M, K = xb.shape
    c, s, y = run_nvfp4(mx, x, g)
    g32 = float(np.float32(g))
    c_o, s_o = oracle.nvfp4_quantize(xb, g32)
    assert np.array_equal(s, s_o), _first_diff(s, s_o)
    assert np.array_equal(c, c_o), _first_diff(c, c_o)
    y_o = oracle.nvfp4_dequantize(c_o, s_o, M, K, g32)
    assert np.array_equal(y, y_o), _first_diff(y, y_o)


@pytest.mark.parametrize("g", [1.0, 0.37, 2688.0 / 25.0])
def test_nvfp4_dense(mx, g):
    x = W.dense_activation(31, 1000, 2880, device="cuda")
    assert_nvfp4_parity(mx, x, g)


def test_nvfp4_full_size(mx):
    x = W.dense_activation(1, device="cuda")
    amax = float(x.float().abs().max())
    assert_nvfp4_parity(mx, x, 448.0 * 6.0 / amax)


@pytest.mark.parametrize("M", [1, 127, 129])
@pytest.mark.parametrize("K", [16, 48, 64, 80, 2880])
def test_nvfp4_ragged(mx, M, K):
    x = W.normal_bf16((M, K), seed=M * 7 + K, device="cuda")
    assert_nvfp4_parity(mx, x, 1.0)


def test_nvfp4_edge_cases_and_16b_aligned(mx):
    x = W.edge_cases(4).cuda()
    assert_nvfp4_parity(mx, x, 1.0)
    flat = torch.empty(x.numel() + 8, dtype=torch.bfloat16, device="cuda")
    y = flat[8:].view(x.shape)
    y.copy_(x)
    assert_nvfp4_parity(mx, y, 3.0)


def test_nvfp4_scale_sweep_every_bf16_max(mx):
    """Each 16-element block takes a different block max: every positive finite
    BF16 value (so g*vecMax/6 sweeps zero, subnormal, normal and saturated
    E4M3 scales), plus blocks whose scale lands exactly on an E4M3 midpoint."""
    rng = np.random.default_rng(9)
    vmax = np.arange(1, 0x7F80, dtype=np.uint16)
    grid = np.unique(np.abs([oracle.e4m3_to_double(i) for i in range(0x7F)]))
    mids = ((grid[:-1] + grid[1:]) / 2 * 6).astype(np.float32)
    mid_bits = (mids.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((mid_bits.astype(np.uint32) << 16).view(np.float32), mids)
    vmax = np.concatenate([vmax, mid_bits])
    rest = (rng.integers(0, 0x10000, (vmax.size, 15), dtype=np.uint32)).astype(np.uint16)
    rest = np.where((rest & 0x7FFF) <= vmax[:, None], rest, rest & 0x8000 | (vmax[:, None] >> 1))
    blocks = np.concatenate([vmax[:, None], rest], axis=1)
    blocks = np.concatenate([blocks, np.zeros(((-blocks.shape[0]) % 16, 16), np.uint16)])
    xb = blocks.reshape(-1, 256)
    assert_nvfp4_parity(mx, W.from_bits(xb, "cuda"), 1.0)


# ----------------------------------------------------- NVFP4, FP16 input
def run_nvfp4_f16(mx, x, g):
    M, K = x.shape
    gs = torch.tensor([g], dtype=torch.float32, device="cuda")
    codes = Guarded(M * (K // 2), shape=(M, K // 2))
    scales = Guarded(mx.mxfp4_nvfp4_scale_bytes(M, K))
    mx.mxfp4_quantize_nvfp4_f16(x, gs, codes.t, scales.t)
    torch.cuda.synchronize()
    codes.check()
    scales.check()
    return codes.t.cpu().numpy(), scales.t.cpu().numpy()


def assert_nvfp4_f16_parity(mx, x, g):
    c, s = run_nvfp4_f16(mx, x, g)
    c_o, s_o = oracle.nvfp4_quantize(f16_bits(x), float(np.float32(g)), f16=True)
    assert np.array_equal(s, s_o), _first_diff(s, s_o)
    assert np.array_equal(c, c_o), _first_diff(c, c_o)


@pytest.mark.parametrize("g", [1.0, 0.37, 2688.0 / 25.0])
def test_nvfp4_f16_dense(mx, g):
    x = W.dense_activation(33, 1000, 2880, device="cuda").float()
    x[::7, ::5] *= 2.0 ** -12                                    # FP16 subnormals too
    assert_nvfp4_f16_parity(mx, x.to(torch.float16), g)


@pytest.mark.parametrize("M,K", [(1, 16), (129, 80), (4096, 7168)])
def test_nvfp4_f16_ragged_and_full_size(mx, M, K):
    x = W.dense_activation(34, M, K, device="cuda").to(torch.float16)
    assert_nvfp4_f16_parity(mx, x, 448.0 * 6.0 / float(x.float().abs().max()))
    assert_nvfp4_f16_parity(mx, offset16_any(x), 1.0)


@pytest.mark.parametrize("g", [1.0, 4096.0])
def test_nvfp4_f16_scale_sweep_every_f16_max(mx, g):
    """Each 16-element block takes a different block max: every positive
    finite FP16 value, subnormals included.  With g = 1 the scales run from
    zero through E4M3 subnormals to saturation at 448; g = 4096 moves the
    FP16 subnormal maxima onto normal E4M3 scales."""
    rng = np.random.default_rng(19)
    vmax = np.arange(1, 0x7C00, dtype=np.uint16)
    rest = rng.integers(0, 0x10000, (vmax.size, 15), dtype=np.uint32).astype(np.uint16)
    rest = np.where((rest & 0x7FFF) <= vmax[:, None], rest, rest & 0x8000 | (vmax[:, None] >> 1))
    blocks = np.concatenate([vmax[:, None], rest], axis=1)
    blocks = np.concatenate([blocks, np.zeros(((-blocks.shape[0]) % 16, 16), np.uint16)])
    hb = blocks.reshape(-1, 256)
    x = torch.from_numpy(hb.view(np.int16)).view(torch.float16).cuda()
    assert_nvfp4_f16_parity(mx, x, g)


def test_nvfp4_grouped_f16_matches_oracle(mx):
    g = W.moe_grouped(seed=21, tokens=200, top_k=4, num_experts=12, K=288, device="cuda")
    gs = _expert_gscales(12, 21)
    xs = g.x.to(torch.float16)
    off = g.offsets
    rc, c_o, s_o, sro_o = oracle.nvfp4_quantize_grouped(f16_bits(xs), off.cpu().numpy(), gs,
                                                        f16=True)
    used = int(sro_o[-1]) * ((288 // 16 + 3) // 4 * 4)
    for xx in (xs, offset16_any(xs)):
        total, K = xx.shape
        E = off.numel() - 1
        codes = Guarded(total * (K // 2), shape=(total, K // 2))
        scales = Guarded(mx.mxfp4_nvfp4_grouped_scale_bytes_bound(total, E, K))
        sro = Guarded(4 * (E + 1), torch.int32)
        status = Guarded(4, torch.int32)
        mx.mxfp4_quantize_nvfp4_grouped_f16(xx, off, torch.from_numpy(gs).cuda(), codes.t,
                                            scales.t, sro.t, status.t)
        torch.cuda.synchronize()
        for t in (codes, scales, sro, status):
            t.check()
        assert int(status.t.cpu()[0]) == 0 and rc == 0
        assert np.array_equal(sro.t.cpu().numpy(), sro_o)
        c, s = codes.t.cpu().numpy(), scales.t.cpu().numpy()
        assert np.array_equal(c, c_o), _first_diff(c, c_o)
        assert np.array_equal(s[:used], s_o[:used]), _first_diff(s[:used], s_o[:used])
        assert (s[used:] == 0xA5).all(), "slack past P[E] must be untouched"
    # the high-level call dispatches on dtype
    c, s, sro, st = mx.quantize_nvfp4_grouped(xs, off, torch.from_numpy(gs).cuda())
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and np.array_equal(c.cpu().numpy(), c_o)


# ------------------------------------------------ streams, graphs, 64-bit
def test_non_default_stream(mx):
    x = W.dense_activation(41, 512, 1024, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        codes, scales = mx.quantize(x)
        y = mx.dequantize(codes, scales, 512, 1024)
    s.synchronize()
    c_o, s_o = oracle.quantize(bits(x))
    assert np.array_equal(codes.cpu().numpy(), c_o) and np.array_equal(scales.cpu().numpy(), s_o)
    assert np.array_equal(bits(y), oracle.dequantize(c_o, s_o, 512, 1024))


def test_cuda_graph_capture_and_replay(mx):
    """The launches (programmatic dependent launch included) can be captured
    in a CUDA graph and replayed on new input contents."""
    M, K = 512, 2048
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    codes = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(mx.mxfp4_scale_bytes(M, K), dtype=torch.uint8, device="cuda")
    y = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    x.copy_(W.dense_activation(42, M, K, device="cuda"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):                       # warm-up outside the capture
        mx.mxfp4_quantize(x, codes, scales)
        mx.mxfp4_dequantize(codes, scales, M, K, y)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mx.mxfp4_quantize(x, codes, scales)
        mx.mxfp4_dequantize(codes, scales, M, K, y)
    for seed in (43, 44):
        x.copy_(W.dense_activation(seed, M, K, device="cuda"))
        g.replay()
        torch.cuda.synchronize()
        c_o, s_o = oracle.quantize(bits(x))
        assert np.array_equal(codes.cpu().numpy(), c_o)
        assert np.array_equal(scales.cpu().numpy(), s_o)
        assert np.array_equal(bits(y), oracle.dequantize(c_o, s_o, M, K))



def test_cuda_graph_of_the_moe_path(mx):
    """Routing, the staged MXFP4 scatter, the gather through a workspace and
    the staged NVFP4 scatter captured in one CUDA graph (memsets and
    programmatic dependent launches included), then replayed on new token
    values and new expert ids: every output against the oracle, so no
    decision of the calls depends on the contents seen at capture time."""
    T, k, E, K = 512, 4, 16, 512
    total = T * k
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    x = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
    gs = torch.empty(E, dtype=torch.float32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    dest = torch.empty((T, k), dtype=torch.int32, device="cuda")
    rows = torch.empty(total, dtype=torch.int32, device="cuda")
    st = [torch.empty(1, dtype=torch.int32, device="cuda") for _ in range(4)]
    u8 = lambda n: torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")  # noqa: E731
    r_ws = u8(mx.mxfp4_route_workspace_bytes(T, k, E))
    s_ws = u8(mx.mxfp4_scatter_workspace_bytes(T, total, E, K))
    g_ws = u8(mx.mxfp4_gather_workspace_bytes(T, total, E, K))
    n_ws = u8(mx.mxfp4_nvfp4_scatter_workspace_bytes(total, E, K))
    bound, nv_bound = (mx.mxfp4_grouped_scale_bytes_bound(total, E, K),
                       mx.mxfp4_nvfp4_grouped_scale_bytes_bound(total, E, K))
    c1, s1, c2, s2 = u8(total * K // 2).view(-1)[:total * K // 2], u8(bound), \
        u8(total * K // 2).view(-1)[:total * K // 2], u8(bound)
    c3, s3 = u8(total * K // 2).view(-1)[:total * K // 2], u8(nv_bound)
    sro = [torch.empty(E + 1, dtype=torch.int32, device="cuda") for _ in range(3)]

    def path():
        mx.mxfp4_moe_route(ids, E, r_ws, off, dest, rows, st[0])
        mx.mxfp4_quantize_grouped_scatter_ws(x, dest, off, total, s_ws, c1, s1, sro[0], st[1])
        mx.mxfp4_quantize_grouped_gather_ws(x, rows, off, g_ws, c2, s2, sro[1], st[2])
        mx.mxfp4_quantize_nvfp4_grouped_scatter_ws(x, dest, off, total, gs, n_ws, c3, s3, sro[2],
                                                   st[3])

    def fill(seed):
        rng = np.random.default_rng(seed)
        ids.copy_(torch.from_numpy(rng.integers(0, E, (T, k)).astype(np.int32)))
        x.copy_(W.dense_activation(seed, T, K, device="cuda"))
        gs.copy_(torch.from_numpy((448.0 * 6.0 / np.exp(rng.uniform(-2, 6, E))).astype(np.float32)))

    fill(70)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                    # warm-up outside the capture
        path()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        path()
    for seed in (71, 72):
        fill(seed)
        graph.replay()
        torch.cuda.synchronize()
        ids_h, xb, g_h = ids.cpu().numpy(), bits(x), gs.cpu().numpy()
        rc, off_o, dest_o, rows_o = oracle.moe_route(ids_h, E)
        assert rc == 0 and [int(t.item()) for t in st] == [0, 0, 0, 0]
        assert np.array_equal(off.cpu().numpy(), off_o)
        assert np.array_equal(dest.cpu().numpy(), dest_o)
        assert np.array_equal(rows.cpu().numpy(), rows_o)
        rc, c_o, s_o, sro_o = oracle.quantize_grouped_scatter(xb, dest_o, off_o, total)
        used = int(sro_o[-1]) * ((K // 32 + 3) // 4 * 4)
        assert rc == 0 and np.array_equal(sro[0].cpu().numpy(), sro_o)
        for c, sc in ((c1, s1), (c2, s2)):           # the scatter and the gather
            assert np.array_equal(c.cpu().numpy().reshape(c_o.shape), c_o)
            assert np.array_equal(sc[:used].cpu().numpy(), s_o[:used])
        rc, c_o, s_o, sro_o = oracle.nvfp4_quantize_grouped_scatter(xb, dest_o, off_o, total, g_h)
        used = int(sro_o[-1]) * ((K // 16 + 3) // 4 * 4)
        assert rc == 0 and np.array_equal(sro[2].cpu().numpy(), sro_o)
        assert np.array_equal(c3.cpu().numpy().reshape(c_o.shape), c_o)
        assert np.array_equal(s3[:used].cpu().numpy(), s_o[:used])


def test_calls_on_concurrent_streams(mx):
    """The library keeps no state between calls (the no-allocation gather's
    fixed scratch excepted): the dense quantize and dequantize on one stream
    and the routing plus staged scatter on another, enqueued interleaved and
    running at the same time, give the oracle's bytes."""
    M, K = 2048, 2048
    T, k, E = 1024, 8, 32
    total = T * k
    xa = W.dense_activation(81, M, K, device="cuda")
    xb = W.dense_activation(82, T, K, device="cuda")
    rng = np.random.default_rng(83)
    ids = torch.from_numpy(rng.integers(0, E, (T, k)).astype(np.int32)).cuda()
    ca = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    sa = torch.empty(mx.mxfp4_scale_bytes(M, K), dtype=torch.uint8, device="cuda")
    ya = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    ws_r = torch.empty(mx.mxfp4_route_workspace_bytes(T, k, E), dtype=torch.uint8, device="cuda")
    ws_s = torch.empty(mx.mxfp4_scatter_workspace_bytes(T, total, E, K), dtype=torch.uint8,
                       device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    dest = torch.empty((T, k), dtype=torch.int32, device="cuda")
    cb = torch.empty((total, K // 2), dtype=torch.uint8, device="cuda")
    sb = torch.empty(mx.mxfp4_grouped_scale_bytes_bound(total, E, K), dtype=torch.uint8,
                     device="cuda")
    sro = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    st = torch.empty(1, dtype=torch.int32, device="cuda")
    s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()
    s_a.wait_stream(torch.cuda.current_stream())
    s_b.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        mx.mxfp4_quantize(xa, ca, sa, s_a)
        mx.mxfp4_moe_route(ids, E, ws_r, off, dest, None, None, s_b)
        mx.mxfp4_dequantize(ca, sa, M, K, ya, s_a)
        mx.mxfp4_quantize_grouped_scatter_ws(xb, dest, off, total, ws_s, cb, sb, sro, st, s_b)
    torch.cuda.synchronize()
    c_o, s_o = oracle.quantize(bits(xa))
    assert np.array_equal(ca.cpu().numpy(), c_o) and np.array_equal(sa.cpu().numpy(), s_o)
    assert np.array_equal(bits(ya), oracle.dequantize(c_o, s_o, M, K))
    rc, off_o, dest_o, _ = oracle.moe_route(ids.cpu().numpy(), E)
    assert rc == 0 and np.array_equal(dest.cpu().numpy(), dest_o)
    rc, cq, sq, sro_o = oracle.quantize_grouped_scatter(bits(xb), dest_o, off_o, total)
    used = int(sro_o[-1]) * ((K // 32 + 3) // 4 * 4)
    assert rc == 0 and int(st.item()) == 0
    assert np.array_equal(cb.cpu().numpy(), cq) and np.array_equal(sb[:used].cpu().numpy(), sq[:used])

def test_more_than_4gib_input(mx):
    """33000 x 65536 BF16 (4.3 GB): byte offsets beyond 2^32; the first and
    last 128-row tiles (and one in the middle) checked against the oracle,
    then the same tiles of its dequantize (a 4.3 GB output)."""
    M, K = 33000, 65536
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    for r0 in range(0, M, 4096):
        r1 = min(M, r0 + 4096)
        x[r0:r1] = W.normal_bf16((r1 - r0, K), seed=r0 + 1, device="cuda")
    codes, scales = mx.quantize(x)
    torch.cuda.synchronize()
    per_tile = mx.mxfp4_scale_bytes(128, K)
    for t in (0, 128, (M - 1) // 128):
        r0 = t * 128
        r1 = min(M, r0 + 128)
        c_o, s_o = oracle.quantize(bits(x[r0:r1]))
        assert np.array_equal(codes[r0:r1].cpu().numpy(), c_o), t
        assert np.array_equal(scales[t * per_tile:(t + 1) * per_tile].cpu().numpy(), s_o), t
    # and its dequantize: a 4.3 GB BF16 output, the same tiles against the oracle
    del x
    torch.cuda.empty_cache()
    y = mx.dequantize(codes, scales, M, K)
    torch.cuda.synchronize()
    for t in (0, 128, (M - 1) // 128):
        r0 = t * 128
        r1 = min(M, r0 + 128)
        c_t = codes[r0:r1].cpu().numpy()
        s_t = scales[t * per_tile:(t + 1) * per_tile].cpu().numpy()
        assert np.array_equal(bits(y[r0:r1]), oracle.dequantize(c_t, s_t, r1 - r0, K)), t
    del y, codes, scales
    torch.cuda.empty_cache()


def test_grouped_and_scatter_beyond_4gib(mx):
    """The grouped quantize, the staged scatter, the gather, the NVFP4 experts
    quant and its staged scatter over a 33000 x 65536 BF16 batch (4.3 GB; row byte offsets
    past 2^32) in five uneven segments, one empty: the first and last 128-row
    tiles of the first and last segments against the oracle (the scatter's
    rows through a random permutation of the tokens; the gather of the same
    rows equal to the scatter)."""
    M, K = 33000, 65536
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    for r0 in range(0, M, 4096):
        r1 = min(M, r0 + 4096)
        x[r0:r1] = W.normal_bf16((r1 - r0, K), seed=r0 + 7, device="cuda")
    off_h = np.array([0, 7000, 7000, 20000, 26001, M], dtype=np.int32)
    off = torch.from_numpy(off_h).cuda()
    E = off_h.size - 1
    per_tile = mx.mxfp4_scale_bytes(128, K)

    def check(codes, scales, sro, rows_of):
        for e in (0, E - 1):
            n = int(off_h[e + 1] - off_h[e])
            for t in (0, (n - 1) // 128):
                r0 = int(off_h[e]) + 128 * t
                r1 = min(int(off_h[e + 1]), r0 + 128)
                c_o, s_o = oracle.quantize(bits(x[rows_of(r0, r1)]))
                assert np.array_equal(codes[r0:r1].cpu().numpy(), c_o), (e, t)
                c0 = (int(sro[e]) // 128 + t) * per_tile
                assert np.array_equal(scales[c0:c0 + per_tile].cpu().numpy(), s_o), (e, t)

    codes, scales, sro, st = mx.quantize_grouped(x, off)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check(codes, scales, sro.cpu().numpy(), lambda r0, r1: slice(r0, r1))
    del codes, scales
    perm = torch.randperm(M, generator=torch.Generator().manual_seed(5)).to(torch.int32)
    dest = perm.view(M, 1).cuda()                   # token t -> row perm[t]
    inv = torch.empty_like(perm)
    inv[perm.long()] = torch.arange(M, dtype=torch.int32)
    codes, scales, sro, st = mx.quantize_grouped_scatter(x, dest, off)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check(codes, scales, sro.cpu().numpy(), lambda r0, r1: inv[r0:r1].long().cuda())
    # the same rows as a gather (row -> token), which must equal the scatter
    codes_g, scales_g, sro_g, st = mx.quantize_grouped_gather(x, inv.cuda(), off)
    torch.cuda.synchronize()
    used = int(sro[-1]) * ((K // 32 + 3) // 4 * 4)
    assert int(st.item()) == 0 and torch.equal(sro_g, sro)
    assert torch.equal(codes_g, codes) and torch.equal(scales_g[:used], scales[:used])
    del codes, scales, codes_g, scales_g
    # the NVFP4 experts quant, a global scale per expert
    gs = torch.tensor([448.0 * 6.0 / v for v in (3.0, 5.0, 7.0, 4.0, 6.0)], device="cuda")
    codes, scales, sro, st = mx.quantize_nvfp4_grouped(x, off, gs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    per_tile = mx.mxfp4_nvfp4_scale_bytes(128, K)
    sro_h = sro.cpu().numpy()
    for e in (0, E - 1):
        n = int(off_h[e + 1] - off_h[e])
        for t in (0, (n - 1) // 128):
            r0 = int(off_h[e]) + 128 * t
            r1 = min(int(off_h[e + 1]), r0 + 128)
            c_o, s_o = oracle.nvfp4_quantize(bits(x[r0:r1]), float(gs[e]))
            assert np.array_equal(codes[r0:r1].cpu().numpy(), c_o), (e, t)
            c0 = (int(sro_h[e]) // 128 + t) * per_tile
            assert np.array_equal(scales[c0:c0 + per_tile].cpu().numpy(), s_o), (e, t)
    del codes, scales
    # and the staged NVFP4 scatter through the permutation
    codes, scales, sro, st = mx.quantize_nvfp4_grouped_scatter(x, dest, off, gs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    sro_h = sro.cpu().numpy()
    for e in (0, E - 1):
        n = int(off_h[e + 1] - off_h[e])
        for t in (0, (n - 1) // 128):
            r0 = int(off_h[e]) + 128 * t
            r1 = min(int(off_h[e + 1]), r0 + 128)
            c_o, s_o = oracle.nvfp4_quantize(bits(x[inv[r0:r1].long().cuda()]), float(gs[e]))
            assert np.array_equal(codes[r0:r1].cpu().numpy(), c_o), (e, t)
            c0 = (int(sro_h[e]) // 128 + t) * per_tile
            assert np.array_equal(scales[c0:c0 + per_tile].cpu().numpy(), s_o), (e, t)
    del x, codes, scales
    torch.cuda.empty_cache()

def test_grouped_many_skewed_experts(mx):
    """3000 experts (the offsets scan spans three 1024-wide chunks) with
    Zipf-like segment sizes, many empty: the segment estimate misses and the
    binary-search fallback runs.  Plain grouped and fused gather both match
    the oracle."""
    rng = np.random.default_rng(12)
    E = 3000
    sizes = np.minimum((rng.zipf(1.6, E) - 1) * 3, 900).astype(np.int64)
    sizes[rng.random(E) < 0.3] = 0
    total = int(sizes.sum())
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    K = 160
    T = 700
    x_tok = W.normal_bf16((T, K), seed=13, device="cuda")
    row_index = torch.from_numpy(rng.integers(0, T, total).astype(np.int32)).cuda()
    x = x_tok.index_select(0, row_index.long())
    off_d = torch.from_numpy(off).cuda()
    c, s, sro, st = run_grouped(mx, x, off_d)
    rc, c_o, s_o, sro_o = oracle.quantize_grouped(bits(x), off)
    assert st == 0 and rc == 0 and np.array_equal(sro, sro_o)
    assert np.array_equal(c, c_o)
    used = int(sro_o[-1]) * 8
    assert np.array_equal(s[:used], s_o[:used])
    c2, s2, sro2, st2 = run_gather(mx, x_tok, row_index, off_d)
    assert st2 == 0 and np.array_equal(sro2, sro_o) and np.array_equal(c2, c_o)
    assert np.array_equal(s2[:used], s_o[:used])


# ----------------------------------------- non-finite input: no fault, finite blocks exact
def _with_nonfinite(x, seed):
    """x with +-Inf / NaN planted in ~2 % of its 32-element blocks; returns
    (tensor, boolean mask of the blocks left finite)."""
    xb = bits(x).copy()
    M, K = xb.shape
    rng = np.random.default_rng(seed)
    nb = K // 32
    hit = rng.random((M, nb)) < 0.02
    for r, b in zip(*np.nonzero(hit)):
        xb[r, b * 32 + rng.integers(0, 32)] = rng.choice(
            np.array([0x7F80, 0xFF80, 0x7FC0, 0xFFC1], np.uint16))
    t = W.from_bits(xb).to(x.device)
    return t, ~hit


def _blocks_equal(c1, s1, c2, s2, M, K, ok):
    """Codes and (untiled) scales of the blocks marked ok agree."""
    f1 = oracle.untile(s1, M, K // 32)
    f2 = oracle.untile(s2, M, K // 32)
    assert np.array_equal(f1[ok], f2[ok])
    n1 = c1.reshape(M, K // 32, 16)
    n2 = c2.reshape(M, K // 32, 16)
    assert np.array_equal(n1[ok], n2[ok])


def test_nonfinite_inputs_do_not_fault(mx):
    M, K = 300, 2880
    x, ok = _with_nonfinite(W.dense_activation(11, M, K, device="cuda"), 1)
    c, s = run_quantize(mx, x)                                  # guard bands checked
    c_o, s_o = oracle.quantize(bits(x))
    _blocks_equal(c, s, c_o, s_o, M, K, ok)
    # FP16, NVFP4 and the grouped forms run without error on the same data
    x16 = x.to(torch.float16)
    cc = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    ss = torch.empty(mx.mxfp4_scale_bytes(M, K), dtype=torch.uint8, device="cuda")
    mx.mxfp4_quantize_f16(x16, cc, ss)
    mx.quantize_nvfp4(x, torch.tensor([1.0], device="cuda"))
    off = torch.tensor([0, 100, 100, 300], dtype=torch.int32, device="cuda")
    _, _, _, st = mx.quantize_grouped(x, off)
    dst = torch.randperm(M, generator=torch.Generator().manual_seed(3)).to(torch.int32)
    _, _, _, st2 = mx.quantize_grouped_scatter(x, dst.view(M, 1).cuda(), off)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0


# -------------------------------------------------- NVFP4 experts quant
def run_nvfp4_grouped(mx, x, offsets, gs):
    total, K = x.shape
    E = offsets.numel() - 1
    codes = Guarded(total * (K // 2), shape=(total, K // 2))
    scales = Guarded(mx.mxfp4_nvfp4_grouped_scale_bytes_bound(total, E, K))
    sro = Guarded(4 * (E + 1), torch.int32)
    status = Guarded(4, torch.int32)
    mx.mxfp4_quantize_nvfp4_grouped(x, offsets, gs, codes.t, scales.t, sro.t, status.t)
    torch.cuda.synchronize()
    for g in (codes, scales, sro, status):
        g.check()
    return (codes.t.cpu().numpy(), scales.t.cpu().numpy(), sro.t.cpu().numpy(),
            int(status.t.cpu()[0]))


def _expert_gscales(E, seed):
    rng = np.random.default_rng(seed)
    return np.float32(448.0 * 6.0) / np.exp(rng.uniform(0.0, 3.0, E)).astype(np.float32)


@pytest.mark.parametrize("tokens,top_k,E,K", [(200, 4, 12, 288), (130, 2, 5, 80),
                                              (64, 3, 9, 2880), (1, 1, 3, 16)])
def test_nvfp4_grouped_matches_oracle(mx, tokens, top_k, E, K):
    g = W.moe_grouped(seed=tokens + K, tokens=tokens, top_k=top_k, num_experts=E, K=K,
                      device="cuda")
    gs = _expert_gscales(E, K)
    c, s, sro, st = run_nvfp4_grouped(mx, g.x, g.offsets, torch.from_numpy(gs).cuda())
    rc, c_o, s_o, sro_o = oracle.nvfp4_quantize_grouped(bits(g.x), g.offsets.cpu().numpy(), gs)
    assert st == 0 and rc == 0 and np.array_equal(sro, sro_o)
    assert np.array_equal(c, c_o), _first_diff(c, c_o)
    used = int(sro_o[-1]) * ((K // 16 + 3) // 4 * 4)
    assert np.array_equal(s[:used], s_o[:used]), _first_diff(s[:used], s_o[:used])
    assert (s[used:] == 0xA5).all(), "slack past P[E] must be untouched"


def test_nvfp4_grouped_empty_segments_16b_input_and_bad_offsets(mx):
    x = W.small_matrix(6, 400, 192).cuda()
    gs = torch.tensor([1.0, 3.0, 0.5, 9.0, 2.0], device="cuda")
    off = torch.tensor([0, 0, 129, 129, 400, 400], dtype=torch.int32, device="cuda")
    for xx in (x, offset16(x)):
        c, s, sro, st = run_nvfp4_grouped(mx, xx, off, gs)
        rc, c_o, s_o, sro_o = oracle.nvfp4_quantize_grouped(bits(x), off.cpu().numpy(),
                                                            gs.cpu().numpy())
        used = int(sro_o[-1]) * 12
        assert st == 0 and np.array_equal(c, c_o) and np.array_equal(s[:used], s_o[:used])
    bad = torch.tensor([0, 300, 200, 200, 400, 400], dtype=torch.int32, device="cuda")
    c, s, sro, st = run_nvfp4_grouped(mx, x, bad, gs)
    assert st == mx.MXFP4_EOFFSETS and (sro == -1).all()
    assert (c == 0xA5).all() and (s == 0xA5).all()


def test_nvfp4_grouped_moe_full_size(mx, moe, moe_nvfp4_oracle):
    """131,072 x 7168 expert-sorted rows, 384 experts with their own global
    scales, against the oracle in full: every code byte, every E4M3 scale
    byte of the padded rows, every padded offset, the slack untouched."""
    gs, c_o, s_o, sro_o = moe_nvfp4_oracle
    total, K = moe.x.shape
    E = moe.num_experts
    codes = Guarded(total * (K // 2), shape=(total, K // 2))
    scales = Guarded(mx.mxfp4_nvfp4_grouped_scale_bytes_bound(total, E, K))
    sro = Guarded(4 * (E + 1), torch.int32)
    st = Guarded(4, torch.int32)
    mx.mxfp4_quantize_nvfp4_grouped(moe.x, moe.offsets, torch.from_numpy(gs).cuda(), codes.t,
                                    scales.t, sro.t, st.t)
    torch.cuda.synchronize()
    for g in (codes, scales, sro, st):
        g.check()
    assert int(st.t.item()) == 0
    assert_full(sro.t.cpu().numpy(), sro_o, "scale row offsets")
    assert_full(codes.t.cpu().numpy(), c_o, "codes")
    s_h = scales.t.cpu().numpy()
    assert_full(s_h[:s_o.size], s_o, "E4M3 tiled scales")
    assert (s_h[s_o.size:] == 0xA5).all(), "slack past the last padded row was written"


# ------------------------------------ NVFP4 experts quant, dispatch as scatter
def run_nvfp4_scatter(mx, x, dest, offsets, total, gs, seed=0, ws=False):
    """The NVFP4 scatter through the C ABI into guard-banded buffers with a
    random prefill (the oracle gets the same bytes); returns GPU and oracle
    results."""
    K = x.shape[1]
    E = offsets.numel() - 1
    f16 = x.dtype == torch.float16
    rng = np.random.default_rng(seed)
    nsb = mx.mxfp4_nvfp4_grouped_scale_bytes_bound(total, E, K)
    c0 = rng.integers(0, 256, (total, K // 2), dtype=np.uint8)
    s0 = rng.integers(0, 256, nsb, dtype=np.uint8)
    codes = Guarded(total * (K // 2), shape=(total, K // 2))
    scales = Guarded(nsb)
    codes.t.copy_(torch.from_numpy(c0))
    scales.t.copy_(torch.from_numpy(s0))
    sro = Guarded(4 * (E + 1), torch.int32)
    status = Guarded(4, torch.int32)
    guards = [codes, scales, sro, status]
    g_d = torch.from_numpy(gs).cuda()
    if ws:
        work = Guarded(max(mx.mxfp4_nvfp4_scatter_workspace_bytes(total, E, K), 16))
        work.t.fill_(0x5A)                            # contents on entry must not matter
        guards.append(work)
        fn = (mx.mxfp4_quantize_nvfp4_grouped_scatter_ws_f16 if f16
              else mx.mxfp4_quantize_nvfp4_grouped_scatter_ws)
        fn(x, dest, offsets, total, g_d, work.t, codes.t, scales.t, sro.t, status.t)
    else:
        fn = (mx.mxfp4_quantize_nvfp4_grouped_scatter_f16 if f16
              else mx.mxfp4_quantize_nvfp4_grouped_scatter)
        fn(x, dest, offsets, total, g_d, codes.t, scales.t, sro.t, status.t)
    torch.cuda.synchronize()
    for g in guards:
        g.check()
    gpu = (codes.t.cpu().numpy(), scales.t.cpu().numpy(), sro.t.cpu().numpy(),
           int(status.t.cpu()[0]))
    xb = (x.contiguous().cpu().view(torch.int16).numpy().view(np.uint16) if f16
          else bits(x.contiguous()))
    rc, c_o, s_o, sro_o = oracle.nvfp4_quantize_grouped_scatter(
        xb, dest.cpu().numpy(), offsets.cpu().numpy(), total, gs, c0, s0, f16=f16)
    return gpu, (c_o, s_o, sro_o, rc)


@pytest.mark.parametrize("tokens,top_k,E,K", [
    (1, 1, 1, 16), (129, 3, 5, 80), (300, 2, 7, 2880), (64, 32, 40, 96), (257, 8, 16, 1056)])
def test_nvfp4_scatter_shapes(mx, tokens, top_k, E, K, scatter_ws):
    g = W.moe_grouped(seed=tokens + K + 5, tokens=tokens, top_k=top_k, num_experts=E, K=K,
                      device="cuda")
    gs = _expert_gscales(E, K)
    gpu, orc = run_nvfp4_scatter(mx, g.x_tokens, g.dest_rows, g.offsets, g.row_index.numel(),
                                 gs, seed=K, ws=scatter_ws)
    assert_scatter_parity(gpu, orc)


@pytest.mark.parametrize("f16", [False, True])
def test_nvfp4_scatter_dropped_routes_strided_and_aligned(mx, f16, scatter_ws):
    g = W.moe_grouped(seed=51, tokens=300, top_k=4, num_experts=9, K=160, device="cuda")
    dst = g.dest_rows.clone()
    drop = torch.rand(dst.shape, generator=torch.Generator().manual_seed(5)) < 0.2
    dst[drop.cuda()] = -1
    gs = _expert_gscales(9, 51)
    xt = g.x_tokens.to(torch.float16) if f16 else g.x_tokens
    wide = torch.zeros((300, 184), dtype=xt.dtype, device="cuda")
    wide[:, 8:168] = xt
    for x in (xt, wide[:, 8:168], offset16_any(xt)):
        gpu, orc = run_nvfp4_scatter(mx, x, dst, g.offsets, g.row_index.numel(), gs, seed=52,
                                     ws=scatter_ws)
        assert_scatter_parity(gpu, orc)


def test_nvfp4_scatter_bad_entries_offsets_and_no_tokens(mx, scatter_ws):
    g = W.moe_grouped(seed=53, tokens=140, top_k=2, num_experts=3, K=64, device="cuda")
    total = g.row_index.numel()
    gs = np.array([1.0, 7.5, 0.3], np.float32)
    dst = g.dest_rows.clone()
    dst[3, 1] = total
    dst[7, 0] = -2
    gpu, orc = run_nvfp4_scatter(mx, g.x_tokens, dst, g.offsets, total, gs, seed=54,
                                 ws=scatter_ws)
    assert orc[3] == -7
    assert_scatter_parity(gpu, orc, want_status=mx.MXFP4_EINDEX)
    gpu, orc = run_nvfp4_scatter(mx, g.x_tokens[:0], dst[:0], g.offsets, total, gs, seed=55,
                                 ws=scatter_ws)
    assert_scatter_parity(gpu, orc)
    bad = torch.tensor([0, 200, 100, total], dtype=torch.int32, device="cuda")
    gpu, orc = run_nvfp4_scatter(mx, g.x_tokens, g.dest_rows, bad, total, gs, seed=56,
                                 ws=scatter_ws)
    assert orc[3] == -6 and gpu[3] == mx.MXFP4_EOFFSETS and (gpu[2] == -1).all()
    assert np.array_equal(gpu[0], orc[0]) and np.array_equal(gpu[1], orc[1])  # untouched


@pytest.mark.parametrize("f16", [False, True])
def test_nvfp4_scatter_shared_global_scales(mx, f16, scatter_ws):
    """Experts that share a global scale (all of them, then runs of equal and
    distinct scales, with dropped routes in between): a token's routes to
    such experts get equal codes and scale bytes, the rest their own; every
    byte against the oracle, over several passes and a ragged tail."""
    g = W.moe_grouped(seed=57, tokens=300, top_k=6, num_experts=12, K=2880 + 32,
                      device="cuda")
    dst = g.dest_rows.clone()
    drop = torch.rand(dst.shape, generator=torch.Generator().manual_seed(7)) < 0.15
    dst[drop.cuda()] = -1
    xt = g.x_tokens.to(torch.float16) if f16 else g.x_tokens
    shared = np.full(12, 448.0 * 6.0 / 5.0, np.float32)
    runs = np.array([1.0, 1.0, 3.0, 3.0, 1.0, 0.5, 0.5, 0.5, 7.0, 1.0, 1.0, 3.0], np.float32)
    for gs in (shared, runs * np.float32(448.0 * 6.0 / 20.0)):
        gpu, orc = run_nvfp4_scatter(mx, xt, dst, g.offsets, g.row_index.numel(), gs, seed=58,
                                     ws=scatter_ws)
        assert_scatter_parity(gpu, orc)


def test_nvfp4_scatter_moe_full_size(mx, moe, moe_nvfp4_oracle):
    """16384 tokens x top-8 over 384 experts with their own global scales,
    K = 7168: both scatter forms equal the NVFP4 experts quant of the
    gathered batch byte for byte, and every byte equals the oracle."""
    g = moe
    gs_h, c_o, s_o, sro_o = moe_nvfp4_oracle
    gs = torch.from_numpy(gs_h).cuda()
    c1, s1, sro1, st1 = mx.quantize_nvfp4_grouped_scatter(g.x_tokens, g.dest_rows, g.offsets, gs)
    c2, s2, sro2, st2 = mx.quantize_nvfp4_grouped(g.x, g.offsets, gs)
    c3, s3, sro3, st3 = mx.quantize_nvfp4_grouped_scatter(g.x_tokens, g.dest_rows, g.offsets, gs,
                                                          staged=False)
    torch.cuda.synchronize()
    assert int(st1.item()) == int(st2.item()) == int(st3.item()) == 0
    assert torch.equal(sro1, sro2) and torch.equal(sro1, sro3)
    used = int(sro1[-1].item()) * (7168 // 16)
    assert torch.equal(c1, c2) and torch.equal(s1[:used], s2[:used])
    assert torch.equal(c1, c3) and torch.equal(s1[:used], s3[:used])
    assert_full(sro1.cpu().numpy(), sro_o, "scale row offsets")
    assert_full(c1.cpu().numpy(), c_o, "codes")
    assert_full(s1[:used].cpu().numpy(), s_o, "E4M3 tiled scales")


def test_nvfp4_scatter_moe_full_size_one_global_scale(mx, moe):
    """The same batch with one global scale for every expert (each token's
    routes then share their bytes and codes): both scatter forms equal the
    NVFP4 experts quant of the gathered batch, and that equals the oracle in
    full."""
    g = moe
    E = g.num_experts
    gs = torch.full((E,), 448.0 * 6.0 / 5.0, device="cuda")
    c2, s2, sro2, st2 = mx.quantize_nvfp4_grouped(g.x, g.offsets, gs)
    for staged in (True, False):
        c1, s1, sro1, st1 = mx.quantize_nvfp4_grouped_scatter(g.x_tokens, g.dest_rows, g.offsets,
                                                              gs, staged=staged)
        torch.cuda.synchronize()
        assert int(st1.item()) == int(st2.item()) == 0
        assert torch.equal(sro1, sro2)
        used = int(sro1[-1].item()) * (7168 // 16)
        assert torch.equal(c1, c2) and torch.equal(s1[:used], s2[:used]), staged
    rc, c_o, s_o, sro_o = oracle.nvfp4_quantize_grouped_threads(
        bits(g.x), g.offsets.cpu().numpy(), gs.cpu().numpy())
    assert rc == 0
    assert_full(sro2.cpu().numpy(), sro_o, "scale row offsets")
    assert_full(c2.cpu().numpy(), c_o, "codes")
    assert_full(s2[:s_o.size].cpu().numpy(), s_o, "E4M3 tiled scales")


# ------------------------------------ NVFP4 at the ends of the global scale
# g * vecMax / 6 overflowing to +inf (the E4M3 byte saturates at 448, the
# products x * g / 448 overflow and the codes saturate at +-6), g below the
# point where any block gets a nonzero E4M3 byte (byte 0, zero codes), and a
# subnormal g; every step is the float32 arithmetic both sides share.  The
# results are specified for g < 2^119 (g / float(byte) finite for every
# nonzero byte); 6.5e35 is just below that bound.
EXTREME_G = [6.5e35, 1.0e30, 1.0e-3, 1.0e-30, 1.0e-40]


@pytest.mark.parametrize("g", EXTREME_G)
def test_nvfp4_extreme_global_scale(mx, g):
    """Dense NVFP4 quantize of the edge-case matrix (heavy tails, zero and
    subnormal blocks) bit-exact against the oracle; the dequantize too where
    1/g is finite (for a subnormal g, 1/g = +inf and a zero code gives
    0 * inf = NaN, whose payload the two sides need not share)."""
    x = W.edge_cases(4).cuda()
    M, K = x.shape
    c, s, y = run_nvfp4(mx, x, g)
    g32 = np.float32(g)
    c_o, s_o = oracle.nvfp4_quantize(bits(x), float(g32))
    assert np.array_equal(s, s_o), _first_diff(s, s_o)
    assert np.array_equal(c, c_o), _first_diff(c, c_o)
    if g >= 1.0e30:
        assert (s_o == 0x7E).sum() > s_o.size // 2          # saturated E4M3 bytes
        assert ((c_o & 0x77) == 0x77).any()                 # and saturated codes
    if g <= 1.0e-30:
        assert not s_o.any() and not c_o.any()              # no block reaches 2^-9
    with np.errstate(divide="ignore", over="ignore"):
        inv_finite = np.isfinite(np.float32(1.0) / g32)
    if inv_finite:
        y_o = oracle.nvfp4_dequantize(c_o, s_o, M, K, float(g32))
        assert np.array_equal(y, y_o), _first_diff(y, y_o)


@pytest.mark.parametrize("g", [1.0, 0.37, 1.0e30, 1.0e-30])
def test_nvfp4_dequantize_every_code_and_scale_byte(mx, g):
    """All 16 codes x all 256 E4M3 scale bytes (negative, subnormal and the
    NaN bytes, whose blocks give 0x7FC0), both store widths, against the
    oracle."""
    M, K = 256, 256
    flat = (np.arange(M * (K // 16)) % 256).astype(np.uint8).reshape(M, K // 16)
    nib = np.tile(np.arange(16), M * K // 16).reshape(M, K)
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    tiled = oracle.tile(flat)
    want = oracle.nvfp4_dequantize(codes, tiled, M, K, float(np.float32(g)))
    gs = torch.tensor([g], dtype=torch.float32, device="cuda")
    for off in (0, 8):                  # 32-byte and only 16-byte aligned outputs
        y = Guarded(M * K * 2 + 16, torch.bfloat16, None)
        out = y.t[off:off + M * K].view(M, K)
        mx.mxfp4_dequantize_nvfp4(torch.from_numpy(codes).cuda(), torch.from_numpy(tiled).cuda(),
                                  gs, M, K, out)
        torch.cuda.synchronize()
        y.check()
        assert np.array_equal(bits(out), want), _first_diff(bits(out), want)


def test_nvfp4_global_scale_beyond_its_range(mx):
    """g = 3e38, past 2^119: a block of BF16 subnormals gets a small E4M3
    byte, g / float(byte) overflows to +inf and its zero elements give
    0 * inf = NaN, whose E2M1 code is unspecified.  The call must not fault,
    the guard bands hold, every scale byte is exact, and so is every code
    except those NaN products'."""
    x = W.edge_cases(4).cuda()
    M, K = x.shape
    g32 = np.float32(3.0e38)
    c, s, _ = run_nvfp4(mx, x, float(g32))
    xb = bits(x)
    c_o, s_o = oracle.nvfp4_quantize(xb, float(g32))
    assert np.array_equal(s, s_o), _first_diff(s, s_o)
    byte = oracle.untile(s_o, M, K // 16)                    # [M, K/16] block bytes
    sfv = np.array([oracle.e4m3_to_double(b) for b in range(256)], np.float32)[byte]
    with np.errstate(divide="ignore", over="ignore"):
        inv_inf = np.isinf(g32 / np.where(sfv > 0, sfv, np.float32(1)))
    nan_el = ((xb & 0x7FFF) == 0) & np.repeat(inv_inf & (byte != 0), 16, axis=1)
    assert nan_el.any(), "the case must occur"
    keep = np.ones((M, K), bool)
    keep[nan_el] = False
    nib = lambda c_: np.stack([c_ & 0xF, c_ >> 4], axis=2).reshape(M, K)  # noqa: E731
    assert np.array_equal(nib(c)[keep], nib(c_o)[keep])


@pytest.mark.parametrize("shared", [False, True], ids=["per_expert", "shared"])
def test_nvfp4_grouped_and_scatter_extreme_global_scales(mx, scatter_ws, shared):
    """The experts quant and both scatter forms with global scales at the
    ends of float32: one of EXTREME_G per expert (and 1.0), or the largest
    shared by every expert (the scatter's one-scale path)."""
    g = W.moe_grouped(seed=9, tokens=300, top_k=4, num_experts=6, K=320, device="cuda")
    total = g.row_index.numel()
    gs = (np.full(6, EXTREME_G[0], np.float32) if shared
          else np.array(EXTREME_G[:2] + [1.0] + EXTREME_G[2:], np.float32))
    c, s, sro, st = run_nvfp4_grouped(mx, g.x, g.offsets, torch.from_numpy(gs).cuda())
    rc, c_o, s_o, sro_o = oracle.nvfp4_quantize_grouped(bits(g.x), g.offsets.cpu().numpy(), gs)
    assert st == 0 and rc == 0 and np.array_equal(sro, sro_o)
    assert np.array_equal(c, c_o), _first_diff(c, c_o)
    used = int(sro_o[-1]) * 20
    assert np.array_equal(s[:used], s_o[:used]), _first_diff(s[:used], s_o[:used])
    gpu, orc = run_nvfp4_scatter(mx, g.x_tokens, g.dest_rows, g.offsets, total, gs, seed=9,
                                 ws=scatter_ws)
    assert_scatter_parity(gpu, orc)


# --------------------------------------- wide rows and a single expert
@pytest.mark.parametrize("K", [32768, 16 * 1027])
def test_every_form_on_wide_rows(mx, K, scatter_ws):
    """Rows of 32,768 elements (256 k-tiles: 16 tile-kernel CTAs per tile, 64
    passes per token row) and of 16,432 (an NVFP4 width with a ragged last
    k-tile): dense MXFP4 and NVFP4 quantize and dequantize, the grouped
    quantize, and the dispatch as gather and as scatter (MXFP4 and NVFP4),
    all against the oracle."""
    g = W.moe_grouped(seed=K % 97, tokens=40, top_k=3, num_experts=5, K=K, device="cuda")
    total = g.row_index.numel()
    if K % 32 == 0:
        assert_quant_parity(mx, g.x_tokens[:33].contiguous())
        c, s, sro, st = run_grouped(mx, g.x, g.offsets)
        rc, c_o, s_o, sro_o = oracle.quantize_grouped(bits(g.x), g.offsets.cpu().numpy())
        assert st == rc == 0 and np.array_equal(sro, sro_o) and np.array_equal(c, c_o)
        used = int(sro_o[-1]) * ((K // 32 + 3) // 4 * 4)
        assert np.array_equal(s[:used], s_o[:used])
        _gather_oracle_check(run_gather_ws(mx, g.x_tokens, g.row_index, g.offsets),
                             bits(g.x_tokens), g.row_index.cpu().numpy(),
                             g.offsets.cpu().numpy(), K)
        assert_scatter_parity(*run_scatter(mx, g.x_tokens, g.dest_rows, g.offsets, total,
                                           seed=K, ws=scatter_ws))
    assert_nvfp4_parity(mx, g.x_tokens[:33].contiguous(), 2688.0 / 25.0)
    gs = _expert_gscales(5, K)
    assert_scatter_parity(*run_nvfp4_scatter(mx, g.x_tokens, g.dest_rows, g.offsets, total, gs,
                                             seed=K, ws=scatter_ws))


def test_every_grouped_form_with_one_expert(mx, scatter_ws):
    """E = 1: every row in one segment (its own scale tiles), top_k = 1."""
    g = W.moe_grouped(seed=77, tokens=300, top_k=1, num_experts=1, K=640, device="cuda")
    total = g.row_index.numel()
    c, s, sro, st = run_grouped(mx, g.x, g.offsets)
    rc, c_o, s_o, sro_o = oracle.quantize_grouped(bits(g.x), g.offsets.cpu().numpy())
    assert st == rc == 0 and sro.tolist() == [0, 384] and np.array_equal(c, c_o)
    assert np.array_equal(s[:384 * 20], s_o[:384 * 20])
    _gather_oracle_check(run_gather_ws(mx, g.x_tokens, g.row_index, g.offsets),
                         bits(g.x_tokens), g.row_index.cpu().numpy(), g.offsets.cpu().numpy(),
                         640)
    assert_scatter_parity(*run_scatter(mx, g.x_tokens, g.dest_rows, g.offsets, total, seed=77,
                                       ws=scatter_ws))
    assert_scatter_parity(*run_nvfp4_scatter(mx, g.x_tokens, g.dest_rows, g.offsets, total,
                                             np.array([3.5], np.float32), seed=77,
                                             ws=scatter_ws))


# ----------------------------------------------- FP16 input, grouped forms
def _f16(t):
    return t.to(torch.float16)


def _h_bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def test_f16_grouped_gather_scatter_match_oracle(mx):
    g = W.moe_grouped(seed=12, tokens=180, top_k=4, num_experts=10, K=288, device="cuda")
    xt = _f16(g.x_tokens)
    xs = _f16(g.x)
    off = g.offsets
    rc, c_o, s_o, sro_o = oracle.quantize_grouped(_h_bits(xs), off.cpu().numpy(), f16=True)
    used = int(sro_o[-1]) * 12
    for label, (c, s, sro, st) in (
            ("grouped", mx.quantize_grouped(xs, off)),
            ("grouped 16B", mx.quantize_grouped(offset16_any(xs), off)),
            ("gather", mx.quantize_grouped_gather(xt, g.row_index, off)),
            ("scatter", mx.quantize_grouped_scatter(xt, g.dest_rows, off))):
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and rc == 0, label
        assert np.array_equal(sro.cpu().numpy(), sro_o), label
        assert np.array_equal(c.cpu().numpy(), c_o), label
        assert np.array_equal(s[:used].cpu().numpy(), s_o[:used]), label


def offset16_any(x):
    flat = torch.empty(x.numel() + 8, dtype=x.dtype, device=x.device)
    y = flat[8:].view(x.shape)
    y.copy_(x)
    assert y.data_ptr() % 32 == 16
    return y


def test_f16_dispatch_full_size(mx):
    """The MoE batch in FP16: the scatter and gather forms equal the grouped
    quantize of the permuted FP16 matrix byte for byte; two experts also
    against the oracle."""
    g = W.moe_grouped(seed=2, device="cuda")
    xt = _f16(g.x_tokens)
    xs = _f16(g.x)
    c1, s1, sro1, st1 = mx.quantize_grouped(xs, g.offsets)
    c2, s2, sro2, st2 = mx.quantize_grouped_gather(xt, g.row_index, g.offsets)
    c3, s3, sro3, st3 = mx.quantize_grouped_scatter(xt, g.dest_rows, g.offsets)
    torch.cuda.synchronize()
    assert int(st1.item()) == int(st2.item()) == int(st3.item()) == 0
    used = int(sro1[-1].item()) * 224
    assert torch.equal(c1, c2) and torch.equal(c1, c3)
    assert torch.equal(s1[:used], s2[:used]) and torch.equal(s1[:used], s3[:used])
    off_h = g.offsets.cpu().numpy()
    for e in (3, 200):
        a, b = int(off_h[e]), int(off_h[e + 1])
        c_o, s_o = oracle.quantize_f16(_h_bits(xs[a:b]))
        assert np.array_equal(c1[a:b].cpu().numpy(), c_o)
        p0 = int(sro1[e].item()) * 224
        assert np.array_equal(s1[p0:p0 + s_o.size].cpu().numpy(), s_o)


# -------------------------------------- fused gather through the scatter path
def run_gather_ws(mx, x, row_index, offsets, f16=False):
    total = row_index.numel()
    K = x.shape[1]
    E = offsets.numel() - 1
    codes = Guarded(total * (K // 2), shape=(total, K // 2))
    scales = Guarded(mx.mxfp4_grouped_scale_bytes_bound(total, E, K))
    sro = Guarded(4 * (E + 1), torch.int32)
    status = Guarded(4, torch.int32)
    ws = Guarded(mx.mxfp4_gather_workspace_bytes(x.shape[0], total, E, K))
    ws.t.fill_(0x5A)                                  # contents on entry must not matter
    fn = mx.mxfp4_quantize_grouped_gather_ws_f16 if f16 else mx.mxfp4_quantize_grouped_gather_ws
    fn(x, row_index, offsets, ws.t, codes.t, scales.t, sro.t, status.t)
    torch.cuda.synchronize()
    for g in (codes, scales, sro, status, ws):
        g.check()
    return (codes.t.cpu().numpy(), scales.t.cpu().numpy(), sro.t.cpu().numpy(),
            int(status.t.cpu()[0]))


def _gather_oracle_check(got, xb, idx, off, K, f16=False):
    c, s, sro, st = got
    rc, c_o, s_o, sro_o = oracle.quantize_grouped_gather(xb, idx, off, f16=f16)
    assert st == rc and np.array_equal(sro, sro_o)
    assert np.array_equal(c, c_o), _first_diff(c, c_o)
    used = int(sro_o[-1]) * ((K // 32 + 3) // 4 * 4)
    assert np.array_equal(s[:used], s_o[:used]), _first_diff(s[:used], s_o[:used])


def test_gather_ws_small_strided_and_aligned(mx):
    g = W.moe_grouped(seed=2, tokens=200, top_k=4, num_experts=12, K=288, device="cuda")
    xb = bits(g.x_tokens)
    idx = g.token_of_row.numpy().astype(np.int32)
    off = g.offsets.cpu().numpy()
    _gather_oracle_check(run_gather_ws(mx, g.x_tokens, g.row_index, g.offsets), xb, idx, off, 288)
    wide = torch.zeros((200, 320), dtype=torch.bfloat16, device="cuda")
    wide[:, 16:304] = g.x_tokens
    _gather_oracle_check(run_gather_ws(mx, wide[:, 16:304], g.row_index, g.offsets), xb, idx, off,
                         288)
    _gather_oracle_check(run_gather_ws(mx, offset16(g.x_tokens), g.row_index, g.offsets), xb, idx,
                         off, 288)


def test_gather_ws_bad_index_heavy_and_unused_tokens(mx):
    """Out-of-range indices give zero rows; one token taken by 70 rows (32 in
    its bucket, 38 on the overflow list); most tokens taken by none."""
    xt = W.small_matrix(3, 40, 64).cuda()
    rng = np.random.default_rng(9)
    idx = rng.integers(0, 5, 300).astype(np.int32)     # only tokens 0..4 are used
    idx[rng.permutation(300)[:70]] = 7                  # token 7: 70 rows
    idx[[5, 17, 250]] = [-1, 40, 1 << 20]               # out of range
    off = np.array([0, 33, 33, 160, 300], np.int32)
    got = run_gather_ws(mx, xt, torch.from_numpy(idx).cuda(), torch.from_numpy(off).cuda())
    assert got[3] == mx.MXFP4_EINDEX
    _gather_oracle_check(got, bits(xt), idx, off, 64)
    assert not got[0][[5, 17, 250]].any()


def test_gather_ws_more_experts_than_shared_memory_holds(mx):
    """3000 experts: above the 2048 segments the map kernel keeps in shared
    memory, so every row's segment is searched in global memory."""
    g = W.moe_grouped(seed=32, tokens=400, top_k=5, num_experts=3000, K=64, device="cuda")
    _gather_oracle_check(run_gather_ws(mx, g.x_tokens, g.row_index, g.offsets),
                         bits(g.x_tokens), g.token_of_row.numpy().astype(np.int32),
                         g.offsets.cpu().numpy(), 64)


def test_gather_ws_long_overflow_list(mx):
    """5000 rows from 3 tokens: all but 96 rows go to the overflow list, more
    entries than overflow warps, so each of those warps takes several."""
    xt = W.small_matrix(4, 3, 256).cuda()
    rng = np.random.default_rng(11)
    idx = rng.integers(0, 3, 5000).astype(np.int32)
    off = np.array([0, 1000, 1000, 3100, 5000], np.int32)
    _gather_oracle_check(run_gather_ws(mx, xt, torch.from_numpy(idx).cuda(),
                                       torch.from_numpy(off).cuda()), bits(xt), idx, off, 256)


def test_gather_per_row_kernel_many_tiles(mx):
    """K = 64 leaves too few code bytes to lend a workspace: the call without
    one runs the per-row gather kernel, here over 32,768 rows in 64 segments
    (hundreds of padded tiles), every byte against the oracle."""
    g = W.moe_grouped(seed=63, tokens=4096, top_k=8, num_experts=64, K=64, device="cuda")
    total = g.row_index.numel()
    ws = mx.mxfp4_gather_workspace_bytes(4096, total, 64, 64)
    assert -(-ws // 32) * 4 > total  # more than a quarter of the rows' codes: no borrowing
    got = run_gather(mx, g.x_tokens, g.row_index, g.offsets)
    _gather_oracle_check(got, bits(g.x_tokens), g.token_of_row.numpy().astype(np.int32),
                         g.offsets.cpu().numpy(), 64)


@pytest.mark.parametrize("f16", [False, True])
def test_gather_without_workspace_borrows_its_codes_tail(mx, f16):
    """The gather without a workspace, large enough to run through the scatter
    path in the last rows of its own codes output (2048 tokens x top-8, K =
    1024: 1104 of 16384 rows borrowed): against the oracle, with out-of-range
    indices in the borrowed tail and in the body; rejected offsets leave the
    codes, tail included, untouched."""
    g = W.moe_grouped(seed=61, tokens=2048, top_k=8, num_experts=64, K=1024, device="cuda")
    xt = g.x_tokens.to(torch.float16) if f16 else g.x_tokens
    hb = (xt.cpu().view(torch.int16).numpy().view(np.uint16) if f16 else bits(xt))
    idx = g.token_of_row.numpy().astype(np.int32)
    total = idx.size
    idx[[5, 9000, total - 1, total - 700]] = [-1, 2048, -3, 1 << 20]
    off = g.offsets
    E = off.numel() - 1
    codes = Guarded(total * 512, shape=(total, 512))
    scales = Guarded(mx.mxfp4_grouped_scale_bytes_bound(total, E, 1024))
    sro = Guarded(4 * (E + 1), torch.int32)
    status = Guarded(4, torch.int32)
    fn = mx.mxfp4_quantize_grouped_gather_f16 if f16 else mx.mxfp4_quantize_grouped_gather
    fn(xt, torch.from_numpy(idx).cuda(), off, codes.t, scales.t, sro.t, status.t)
    torch.cuda.synchronize()
    for t in (codes, scales, sro, status):
        t.check()
    got = (codes.t.cpu().numpy(), scales.t.cpu().numpy(), sro.t.cpu().numpy(),
           int(status.t.cpu()[0]))
    _gather_oracle_check(got, hb, idx, off.cpu().numpy(), 1024, f16=f16)
    assert got[3] == mx.MXFP4_EINDEX
    assert not got[0][[5, 9000, total - 1, total - 700]].any()
    # rejected offsets: nothing written, the borrowed tail included
    bad = off.clone()
    bad[3] = bad[4] + 1
    codes2 = Guarded(total * 512, shape=(total, 512))
    fn(xt, torch.from_numpy(idx).cuda(), bad, codes2.t, scales.t, sro.t, status.t)
    torch.cuda.synchronize()
    codes2.check()
    assert int(status.t.cpu()[0]) == mx.MXFP4_EOFFSETS
    assert (codes2.t == 0xA5).all()


def test_gather_ws_bad_offsets_write_nothing(mx):
    xt = W.small_matrix(3, 16, 64).cuda()
    idx = torch.arange(20, dtype=torch.int32, device="cuda") % 16
    off = torch.tensor([0, 12, 8, 20], dtype=torch.int32, device="cuda")
    c, s, sro, st = run_gather_ws(mx, xt, idx, off)
    assert st == mx.MXFP4_EOFFSETS and (sro == -1).all()
    assert (c == 0xA5).all() and (s == 0xA5).all()


def test_gather_ws_fp16_and_full_size(mx):
    g = W.moe_grouped(seed=13, tokens=130, top_k=3, num_experts=6, K=96, device="cuda")
    x16 = g.x_tokens.to(torch.float16)
    hb = x16.cpu().view(torch.int16).numpy().view(np.uint16)
    _gather_oracle_check(run_gather_ws(mx, x16, g.row_index, g.offsets, f16=True), hb,
                         g.token_of_row.numpy().astype(np.int32), g.offsets.cpu().numpy(), 96,
                         f16=True)
    G = W.moe_grouped(seed=2, device="cuda")
    c1, s1, sro1, st1 = mx.quantize_grouped_gather(G.x_tokens, G.row_index, G.offsets)
    c2, s2, sro2, st2 = mx.quantize_grouped_gather(G.x_tokens, G.row_index, G.offsets,
                                                   via_scatter=False)
    torch.cuda.synchronize()
    assert int(st1.item()) == 0 and int(st2.item()) == 0 and torch.equal(sro1, sro2)
    used = int(sro1[-1].item()) * 224
    assert torch.equal(c1, c2) and torch.equal(s1[:used], s2[:used])
