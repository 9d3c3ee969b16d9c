"""GPU parity of the dispatch permutation (mxfp4_moe_route) against the
oracle, through the C ABI: every output word, at chunk boundaries, with
dropped (-1) and invalid ids, one expert and the most experts, no tokens,
the full 16384-token top-8 routing over 384 experts, and routed straight
into the fused scatter quantize."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mxfp4_block_quantization_gb300 as m
    return m


def run_route(mx, ids_np, E, with_rows=True):
    ids = torch.from_numpy(ids_np).cuda()
    T, k = ids_np.shape
    off = torch.full((E + 1 + 64,), -5, dtype=torch.int32, device="cuda")   # + guard words
    dest = torch.full((T * k + 64,), -5, dtype=torch.int32, device="cuda")
    rows = torch.full((T * k + 64,), -5, dtype=torch.int32, device="cuda")
    st = torch.full((1,), -5, dtype=torch.int32, device="cuda")
    ws = torch.full((max(mx.mxfp4_route_workspace_bytes(T, k, E), 16),), 0x5A,
                    dtype=torch.uint8, device="cuda")                     # contents irrelevant
    mx.mxfp4_moe_route(ids, E, ws, off[:E + 1], dest[:T * k].view(T, k),
                       rows[:T * k] if with_rows else None, st)
    torch.cuda.synchronize()
    off, dest, rows = off.cpu().numpy(), dest.cpu().numpy(), rows.cpu().numpy()
    assert (off[E + 1:] == -5).all() and (dest[T * k:] == -5).all() and (rows[T * k:] == -5).all()
    n_rows = int(off[E])
    if not with_rows:
        assert (rows == -5).all()
    return off[:E + 1], dest[:T * k].reshape(T, k), rows[:n_rows], int(st.item()), rows


def assert_route_parity(mx, ids_np, E, with_rows=True):
    off, dest, rows, st, raw = run_route(mx, ids_np, E, with_rows)
    rc, off_o, dest_o, rows_o = oracle.moe_route(ids_np, E)
    assert st == rc
    assert np.array_equal(off, off_o)
    assert np.array_equal(dest, dest_o), np.argwhere(dest != dest_o)[:5]
    if with_rows:
        assert np.array_equal(rows, rows_o)
        assert (raw[int(off_o[-1]):] == -5).all(), "row_index past the rows was written"


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (128, 8, 384), (1024, 1, 7), (1025, 1, 7),
                                   (341, 3, 5), (2047, 4, 100), (500, 32, 9),
                                   (64, 2, 8192)])
def test_route_random_ids(mx, T, k, E):
    rng = np.random.default_rng(T * 31 + k * 7 + E)
    ids = rng.integers(0, E, (T, k)).astype(np.int32)
    ids[rng.random((T, k)) < 0.03] = -1
    assert_route_parity(mx, ids, E)


def test_route_skewed_invalid_and_without_row_index(mx):
    rng = np.random.default_rng(5)
    ids = np.where(rng.random((3000, 6)) < 0.7, 3, rng.integers(0, 40, (3000, 6))).astype(np.int32)
    assert_route_parity(mx, ids, 40)                         # one expert takes most routes
    ids[::97, 1] = 40                                        # out of range
    ids[5, 0] = -3
    assert_route_parity(mx, ids, 40)
    assert_route_parity(mx, ids, 40, with_rows=False)
    ids[:] = -1                                              # nothing dispatched
    assert_route_parity(mx, ids, 40)


def test_route_no_tokens(mx):
    off, dest, rows, st, _ = run_route(mx, np.zeros((0, 8), np.int32), 12)
    assert st == 0 and (off == 0).all() and dest.size == 0


def test_route_moe_full_size(mx):
    """16384 tokens x top-8 over 384 experts (the MoE workload's routing):
    the device routing equals the oracle and the workload generator's own
    permutation, which sorts with torch."""
    g = W.moe_grouped(seed=2, device="cpu", K=32)
    off = g.offsets.numpy()
    dest = g.dest_rows.numpy()
    ids = (np.searchsorted(off, dest, side="right") - 1).astype(np.int32)
    assert_route_parity(mx, ids, 384)
    o, d, r, st, _ = run_route(mx, ids, 384)
    assert st == 0 and np.array_equal(o, off) and np.array_equal(d, dest)
    assert np.array_equal(r, g.row_index.numpy())


def test_route_then_scatter_quantize(mx):
    """Router ids straight to the grouped MXFP4 batch: moe_route, then the
    scatter quantize with a workspace, equals the oracle's route and scatter."""
    rng = np.random.default_rng(11)
    T, k, E, K = 700, 4, 23, 320
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    x = W.normal_bf16((T, K), 12, device="cuda")
    off, dest, rows, st = mx.moe_route(torch.from_numpy(ids).cuda(), E)
    codes, scales, sro, st2 = mx.quantize_grouped_scatter(x, dest, off)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    rc, off_o, dest_o, _ = oracle.moe_route(ids, E)
    rc2, c_o, s_o, sro_o = oracle.quantize_grouped_scatter(W.bf16_bits(x), dest_o, off_o,
                                                           T * k)
    assert rc == rc2 == 0 and np.array_equal(sro.cpu().numpy(), sro_o)
    assert np.array_equal(codes.cpu().numpy(), c_o)
    used = int(sro_o[-1]) * 12
    assert np.array_equal(scales[:used].cpu().numpy(), s_o[:used])
