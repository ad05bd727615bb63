"""GPU planner parity: row intervals, Full/Partial/Empty CSR lists in q2k and
k2q order and the longest-work-first tile order must equal the oracle's
bit for bit; the backward work items must partition the k2q lists by
q-chunk in chunk-major order."""
import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

COST_FULL, COST_MASK = 4, 5


@pytest.fixture(scope="module")
def ffa():
    import torch
    assert torch.cuda.is_available()
    import __graft_entry__
    __graft_entry__.build()
    import flexible_mask_flashattention_gb300 as m
    return m


def check_bwd_items(plan, k2q):
    """The backward work items partition every k-tile's k2q blocks into pieces
    that each lie inside one q-chunk, one piece per (k-tile, chunk) pair with
    blocks, ordered by chunk and then by the k-tiles' longest-work-first rank."""
    fo, fi, mo, mi, order = k2q
    info = plan.info()
    C = info["bwd_chunk_tiles"]
    items = plan.bwd_items().astype(np.int64)
    assert C > 0 and C & (C - 1) == 0 and len(items) == info["bwd_items"]
    n_rt = len(fo) - 1
    rank = np.empty(n_rt, np.int64)
    rank[order] = np.arange(n_rt)
    kt, f0, m0 = items[:, 0], items[:, 1], items[:, 2]
    nf, nm = items[:, 3] & 0xffff, items[:, 3] >> 16
    assert np.all(nf + nm > 0)
    assert np.all((fo[kt] <= f0) & (f0 + nf <= fo[kt + 1]) & (mo[kt] <= m0) & (m0 + nm <= mo[kt + 1]))
    # every block of both lists is covered exactly once
    for idx, start, cnt in ((fi, f0, nf), (mi, m0, nm)):
        cover = np.zeros(len(idx) + 1, np.int64)
        np.add.at(cover, start, 1)
        np.add.at(cover, start + cnt, -1)
        assert np.all(np.cumsum(cover)[:len(idx)] == 1)
    # each item lies in one chunk (lists ascend inside a k-tile: first and last decide)
    chunk = np.where(nf > 0, fi[np.minimum(f0, max(len(fi) - 1, 0))] // C if len(fi) else -1,
                     mi[np.minimum(m0, max(len(mi) - 1, 0))] // C if len(mi) else -1).astype(np.int64)
    for idx, start, cnt in ((fi, f0, nf), (mi, m0, nm)):
        has = cnt > 0
        if np.any(has):
            assert np.all(idx[start[has]] // C == chunk[has])
            assert np.all(idx[start[has] + cnt[has] - 1] // C == chunk[has])
    # one item per (k-tile, chunk) pair with blocks
    kt_all = np.concatenate([np.repeat(np.arange(n_rt), np.diff(fo)), np.repeat(np.arange(n_rt), np.diff(mo))])
    q_all = np.concatenate([fi, mi]).astype(np.int64)
    pairs = np.unique(kt_all * (1 << 32) + q_all // C)
    got = np.sort(kt * (1 << 32) + chunk)
    np.testing.assert_array_equal(got, pairs)
    # chunk-major, then longest-work-first rank
    key = chunk * (1 << 32) + rank[kt]
    assert np.all(np.diff(key) > 0)


def check_plan(ffa, slices, sq, sk, bm, bn, dense=None, bwd=None):
    """bm x bn: forward (q2k) tiles; bwd: the backward (k2q) tiles, default the same."""
    bbm, bbn = bwd if bwd is not None else (bm, bn)
    plan = ffa.Plan(slices, sq, sk, bm, bn, bwd_block_m=bbm, bwd_block_n=bbn)
    info = plan.info()
    assert info["mask_area"] == O.slices_area(slices)
    assert info["plan_launches"] >= (0 if sq == 0 else 1)
    assert (info["fwd_bm"], info["fwd_bn"], info["bwd_bm"], info["bwd_bn"]) == (bm, bn, bbm, bbn)
    assert info["m_tiles"] == -(-sq // bm) and info["n_tiles"] == -(-sk // bn)
    assert info["bwd_m_tiles"] == -(-sq // bbm) and info["bwd_n_tiles"] == -(-sk // bbn)
    for direction in ("q2k", "k2q"):
        tm, tn = (bm, bn) if direction == "q2k" else (bbm, bbn)
        counts = O.block_counts_from_intervals(slices, sq, sk, tm, tn)
        want = O.block_csr_from_intervals(slices, sq, sk, tm, tn, direction, counts=counts)
        got = plan.csr(direction)
        for name, a, b in zip(("full_off", "full_idx", "mask_off", "mask_idx"), want, got[:4]):
            np.testing.assert_array_equal(b, a, err_msg=f"{direction} {name}")
        np.testing.assert_array_equal(got[4], O.lpt_order(want[0], want[2], COST_FULL, COST_MASK),
                                      err_msg=f"{direction} order")
        if direction == "k2q":
            check_bwd_items(plan, got)
        if dense:
            cls = O.classify_blocks_dense(slices, sq, sk, tm, tn, direction)
            for a, b in zip(O.csr_from_classes(cls, direction), got[:4]):
                np.testing.assert_array_equal(b, a)
    if dense:   # one query interval per (slice, key column the slice allows to some row)
        kiv = sum(int(O.mask_block([s], np.arange(sq), np.arange(sk)).any(axis=0).sum())
                  for s in O.slice_tuples(slices))
        assert info["key_intervals"] == kiv
    row, lo, hi = O.row_intervals(slices, sq)
    assert info["row_intervals"] == len(row)
    off, iv = plan.row_intervals()
    np.testing.assert_array_equal(off, np.searchsorted(row, np.arange(sq + 1)))
    np.testing.assert_array_equal(iv[:, 0], lo)
    np.testing.assert_array_equal(iv[:, 1], hi)
    plan.check_status()
    plan.destroy()


@pytest.mark.parametrize("seed", range(24))
def test_random_slices_random_tiles(ffa, seed):
    rng = np.random.default_rng(seed)
    sq, sk = int(rng.integers(1, 700)), int(rng.integers(1, 700))
    bm, bn = int(2 ** rng.integers(3, 8)), int(2 ** rng.integers(3, 8))
    bwd = (int(2 ** rng.integers(3, 8)), int(2 ** rng.integers(3, 8))) if seed % 2 else None
    sl = W.random_slices(seed, sq, sk, max_segments=6, max_pieces=6)
    check_plan(ffa, sl, sq, sk, bm, bn, dense=True, bwd=bwd)


@pytest.mark.parametrize("seed", range(6))
def test_random_slices_random_tiles_general_path(ffa, seed):
    """Sizes above the one-launch path for small plans (2048 rows or columns),
    so that the general multi-kernel path is checked on random slice lists too."""
    rng = np.random.default_rng(1000 + seed)
    sq, sk = int(rng.integers(2049, 4500)), int(rng.integers(300, 4500))
    if seed % 2:
        sq, sk = sk, sq
    bm, bn = int(2 ** rng.integers(3, 8)), int(2 ** rng.integers(3, 8))
    bwd = (int(2 ** rng.integers(3, 8)), int(2 ** rng.integers(3, 8))) if seed % 3 else None
    sl = W.random_slices(seed + 50, sq, sk, max_segments=6, max_pieces=6)
    check_plan(ffa, sl, sq, sk, bm, bn, dense=True, bwd=bwd)


def test_edge_cases(ffa):
    check_plan(ffa, [], 300, 200, 128, 128, dense=True)                       # no slices: every row empty
    check_plan(ffa, [(0, 1, 0, 1, O.FULL)], 1, 1, 128, 128, dense=True)       # one token
    check_plan(ffa, [(5, 5, 0, 9, O.FULL), (0, 3, 4, 4, O.CAUSAL), (0, 2, 0, 5, O.BI_CAUSAL)], 9, 9, 8, 8,
               dense=True)                                                    # zero-area slices only
    check_plan(ffa, [(0, 1000, 0, 1000, O.CAUSAL)], 1000, 1000, 128, 128, dense=True)   # ragged causal
    check_plan(ffa, [(0, 256, 0, 256, O.FULL)], 256, 256, 128, 128, dense=True)         # all Full
    check_plan(ffa, [(0, 200, 0, 600, O.FULL)], 200, 600, 16, 1024, dense=True)          # one wide tile
    check_plan(ffa, [(0, 3000, 0, 40, O.INV_CAUSAL), (0, 3000, 40, 41, O.FULL)], 3000, 41, 8, 8)


def test_many_intervals_per_row(ffa):
    # 300 one-key FULL slices per row: exercises rows with many intervals.
    sl = [(0, 256, 3 * j, 3 * j + 1, O.FULL) for j in range(300)]
    check_plan(ffa, sl, 256, 900, 128, 128)


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
def test_workload_plans(ffa, name):
    w = W.workload(name)
    check_plan(ffa, w.slices, w.seqlen, w.seqlen, 128, 128, dense=w.seqlen <= 4096)


def test_square_causal_closed_form(ffa):
    for m in (1, 3, 17):
        L = 128 * m
        plan = ffa.Plan([(0, L, 0, L, O.CAUSAL)], L, L)
        info = plan.info()
        assert info["q2k_full"] == m * (m - 1) // 2 and info["q2k_mask"] == m
        assert info["k2q_full"] == m * (m - 1) // 2 and info["k2q_mask"] == m
        assert info["mask_area"] == L * (L + 1) // 2
