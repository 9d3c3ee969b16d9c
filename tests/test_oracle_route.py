"""Pins of the oracle's dispatch permutation (router expert ids -> rows
sorted by expert, then by entry index): a hand-derived example, numpy's
stable argsort on random ids, dropped (-1) and invalid ids, and the MoE
workload generator, which sorts with torch."""
import numpy as np
import pytest


def test_route_hand_example(orc):
    # entries (t, j): t0 -> 2, 0; t1 -> 0, 1; t2 -> 2, 2 (twice); t3 -> not dispatched, 1
    ids = np.array([[2, 0], [0, 1], [2, 2], [-1, 1]], np.int32)
    rc, off, dest, rows = orc.moe_route(ids, 3)
    assert rc == 0
    assert off.tolist() == [0, 2, 4, 7]
    assert dest.tolist() == [[4, 0], [1, 2], [5, 6], [-1, 3]]
    assert rows.tolist() == [0, 1, 1, 3, 0, 2, 2]


def _numpy_route(ids, E):
    flat = ids.ravel()
    ok = (flat >= 0) & (flat < E)
    idx = np.nonzero(ok)[0]
    order = idx[np.argsort(flat[idx], kind="stable")]
    dest = np.full(flat.size, -1, np.int64)
    dest[order] = np.arange(order.size)
    off = np.concatenate([[0], np.cumsum(np.bincount(flat[ok], minlength=E))])
    return off, dest.reshape(ids.shape), order // ids.shape[1]


@pytest.mark.parametrize("T,top_k,E", [(1, 1, 1), (97, 3, 5), (500, 8, 384), (64, 32, 7000)])
def test_route_equals_a_stable_sort(orc, T, top_k, E):
    rng = np.random.default_rng(T * 7 + E)
    ids = rng.integers(0, E, (T, top_k)).astype(np.int32)
    ids[rng.random((T, top_k)) < 0.05] = -1                  # some routes not dispatched
    rc, off, dest, rows = orc.moe_route(ids, E)
    off_n, dest_n, rows_n = _numpy_route(ids, E)
    assert rc == 0
    assert np.array_equal(off, off_n) and np.array_equal(dest, dest_n)
    assert np.array_equal(rows, rows_n)


def test_route_invalid_ids_are_dropped_and_reported(orc):
    ids = np.array([[0, 3], [5, -1], [-2, 1], [2, 2]], np.int32)
    rc, off, dest, rows = orc.moe_route(ids, 3)
    assert rc == -7
    assert off.tolist() == [0, 1, 2, 4]
    assert dest.tolist() == [[0, -1], [-1, -1], [-1, 1], [2, 3]]
    assert rows.tolist() == [0, 2, 3, 3]
    rc, *_ = orc.moe_route(np.array([[-1, -1]], np.int32), 3)
    assert rc == 0                                            # -1 alone is not an error


def test_route_reproduces_the_moe_workload(orc):
    """The workload generator routes each token to distinct experts and
    stable-sorts the entries with torch; the expert of every entry, read
    back from its row's segment, routes to the very same permutation."""
    import workloads as W
    g = W.moe_grouped(seed=2, tokens=2000, top_k=8, num_experts=384, K=32)
    off = g.offsets.numpy()
    dest = g.dest_rows.numpy()
    ids = (np.searchsorted(off, dest, side="right") - 1).astype(np.int32)
    rc, off_o, dest_o, rows_o = orc.moe_route(ids, 384)
    assert rc == 0
    assert np.array_equal(off_o, off) and np.array_equal(dest_o, dest)
    assert np.array_equal(rows_o, g.row_index.numpy())
