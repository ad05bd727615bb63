"""The library's dispatch solver (host code, no GPU) against the oracle's
chunk areas and min-heap greedy: bit-exact on random slice lists and on the
named workloads, the hand-worked area fixtures, and its argument checks."""
import os

import numpy as np
import pytest

import oracle as O
import workloads as W
from conftest import golden_lines

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ffa():
    import flexible_mask_flashattention_gb300 as m
    try:
        m.load_library()
    except m.FFAError:
        pytest.skip("library not built")
    return m


def check(ffa, slices, sq, sk, chunk, cp):
    bucket, carea, barea = ffa.dispatch_solve(slices, sq, sk, chunk, cp)
    want_area = O.chunk_areas(slices, sq, chunk)
    want_bucket, want_load = O.dispatch_greedy(want_area, cp)
    np.testing.assert_array_equal(carea, want_area)
    np.testing.assert_array_equal(bucket, want_bucket)
    np.testing.assert_array_equal(barea, want_load)


def test_area_fixtures(ffa):
    n = 0
    for toks in golden_lines("dispatch.txt"):
        if toks[0] != "areas":
            continue
        sl = [tuple(int(x) for x in t.split(",")) for t in toks[1].split(";")]
        sq, sk, chunk = int(toks[3]), int(toks[5]), int(toks[7])
        want = [int(x) for x in toks[-1].split(",")]
        _, carea, _ = ffa.dispatch_solve(sl, sq, sk, chunk, 1)
        assert carea.tolist() == want, sl
        n += 1
    assert n >= 8


@pytest.mark.parametrize("seed", range(20))
def test_random_slices(ffa, seed):
    rng = np.random.default_rng(900 + seed)
    cp = int(rng.integers(1, 6))
    chunk = int(rng.integers(1, 40))
    sq = cp * chunk * int(rng.integers(1, 8))
    sk = int(rng.integers(1, 500))
    sl = W.random_slices(seed + 1000, sq, sk, max_segments=6, max_pieces=6)
    check(ffa, sl, sq, sk, chunk, cp)


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
@pytest.mark.parametrize("chunk,cp", [(512, 4), (2048, 8)])
def test_workloads(ffa, name, chunk, cp):
    w = W.workload(name)
    if w.seqlen % (chunk * cp):
        pytest.skip("sequence length not divisible")
    check(ffa, w.slices, w.seqlen, w.seqlen, chunk, cp)


def test_argument_checks(ffa):
    with pytest.raises(ffa.FFAError):
        ffa.dispatch_solve([(0, 10, 0, 10, O.FULL)], 10, 10, 4, 2)          # 10 % (2 * 4) != 0
    with pytest.raises(ffa.FFAError):
        ffa.dispatch_solve([(0, 9, 0, 11, O.FULL)], 8, 10, 2, 2)           # slice beyond seqlen_q
    with pytest.raises(ffa.FFAError):
        ffa.dispatch_solve([(0, 8, 0, 8, O.FULL), (0, 4, 2, 3, O.FULL)], 8, 8, 2, 2)   # double coverage
    with pytest.raises(ffa.FFAError):
        ffa.dispatch_solve([], 8, 8, 0, 2)                                  # chunk size 0
    bucket, carea, barea = ffa.dispatch_solve([], 8, 8, 2, 2)               # empty mask: all areas 0
    # equal loads go to the lower bucket until it is full
    assert carea.tolist() == [0, 0, 0, 0] and barea.tolist() == [0, 0] and bucket.tolist() == [0, 0, 1, 1]
