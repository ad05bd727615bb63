"""GPU parity of Range-Gather and Range-Scatter-Reduce against the oracle:
gather bit-exact; scatter-reduce bit-exact on disjoint fp32 ranges (one add
per element), within fp32 summation order on overlapping ones, and within
one bf16 rounding per add in bf16."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from ffa_testlib import to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffa():
    assert torch.cuda.is_available()
    import __graft_entry__
    __graft_entry__.build()
    import flexible_mask_flashattention_gb300 as m
    return m


def random_ranges(rng, rows, n, allow_overlap):
    out = []
    if allow_overlap:
        for _ in range(n):
            s = int(rng.integers(0, rows))
            out.append((s, int(rng.integers(s, min(rows, s + 200) + 1))))
    else:
        cuts = sorted(set(rng.integers(0, rows + 1, 2 * n).tolist()))
        pairs = list(zip(cuts[0::2], cuts[1::2]))
        out = [pairs[i] for i in rng.permutation(len(pairs))]
    return out


@pytest.mark.parametrize("seed", range(6))
def test_range_gather(ffa, seed):
    rng = np.random.default_rng(seed)
    rows, h, d = int(rng.integers(1, 3000)), [1, 4, 8][seed % 3], [64, 128][seed % 2]
    t = W.make_tensors(rows, h, h, d, seed, with_dout=False)["k"]
    ranges = random_ranges(rng, rows, int(rng.integers(0, 40)), allow_overlap=True) + [(0, 0), (rows, rows)]
    got = ffa.range_gather(t.cuda(), ranges)
    want = O.range_gather(t.float().numpy(), ranges)
    assert got.shape[0] == want.shape[0]
    np.testing.assert_array_equal(to_np(got), want)


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_range_scatter_reduce(ffa, overlap, dtype):
    rng = np.random.default_rng(17 + overlap)
    rows, h, d = 2500, 4, 128
    ranges = random_ranges(rng, rows, 30, allow_overlap=overlap)
    total = sum(e - s for s, e in ranges)
    g = torch.Generator().manual_seed(3)
    dst = torch.randn(rows, h, d, generator=g).to(dtype)
    src = torch.randn(total, h, d, generator=g).to(dtype)
    want = O.range_scatter_reduce(src.float().numpy(), ranges, dst.float().numpy())
    got = ffa.range_scatter_reduce(src.cuda(), ranges, dst.cuda())
    torch.cuda.synchronize()
    got = to_np(got).astype(np.float64)
    if dtype == torch.float32 and not overlap:
        # one fp32 add per element: the fp32 rounding of the exact sum
        np.testing.assert_array_equal(got, want.astype(np.float32).astype(np.float64))
    else:
        # k rounded adds into an element: |err| <= k u sum |terms| (u the unit roundoff)
        cover = np.zeros(rows, np.int64)
        for s, e in ranges:
            cover[s:e] += 1
        k = np.maximum(cover, 1)[:, None, None]
        u = 2.0 ** -24 if dtype == torch.float32 else 2.0 ** -8
        abs_sum = O.range_scatter_reduce(np.abs(src.float().numpy()), ranges, np.abs(dst.float().numpy()))
        assert np.all(np.abs(got - want) <= k * u * abs_sum)


@pytest.mark.parametrize("width", [4, 64])
def test_range_gather_long_table(ffa, width):
    # more ranges than travel in the launch's parameters: the table goes through device memory.
    # With 16-byte rows (width 4 fp32) one 64 KB gather tile spans hundreds of ranges.
    rng = np.random.default_rng(40 + width)
    rows = 5000
    x = torch.randn(rows, width, generator=torch.Generator().manual_seed(5))
    ranges = random_ranges(rng, rows, 700, allow_overlap=True)
    got = ffa.range_gather(x.cuda(), ranges)
    np.testing.assert_array_equal(to_np(got), O.range_gather(x.numpy(), ranges))
    # and just below the parameter limit, on the same data
    few = ranges[:256]
    np.testing.assert_array_equal(to_np(ffa.range_gather(x.cuda(), few)), O.range_gather(x.numpy(), few))


def test_range_scatter_reduce_long_table(ffa):
    rng = np.random.default_rng(41)
    rows = 6000
    ranges = random_ranges(rng, rows, 400, allow_overlap=False)
    assert len(ranges) > 256
    total = sum(e - s for s, e in ranges)
    g = torch.Generator().manual_seed(6)
    dst = torch.randn(rows, 2, 8, generator=g)
    src = torch.randn(total, 2, 8, generator=g)
    want = O.range_scatter_reduce(src.numpy(), ranges, dst.numpy())
    got = to_np(ffa.range_scatter_reduce(src.cuda(), ranges, dst.cuda())).astype(np.float64)
    np.testing.assert_array_equal(got, want.astype(np.float32).astype(np.float64))


def test_argument_errors(ffa):
    x = torch.zeros(10, 4, dtype=torch.float32, device="cuda")
    with pytest.raises(ffa.FFAError):
        ffa.range_gather(x, [(5, 11)])                                      # beyond the rows
    with pytest.raises(ffa.FFAError):
        ffa.range_gather(torch.zeros(10, 3, dtype=torch.float32, device="cuda"), [(0, 2)])   # 12-byte rows
    with pytest.raises(ffa.FFAError):
        ffa.range_scatter_reduce(torch.zeros(2, 4, device="cuda"), [(3, 2)], x)             # start > end
