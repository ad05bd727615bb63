"""GPU parity of the LSE merge of partial results: ffa_fwd_accumulate (the
forward merged into an existing (out, lse)) and ffa_lse_combine (two partial
results merged element by element), against the oracle's union forward /
backward and its lse_merge.

Tolerances.
- ffa_fwd_accumulate: the tests scale v by 0.5, so that |out| < 2. The result
  then carries at most two bf16 roundings (of the input partial and of the
  output) of at most 2^-8 each, and the standard out / lse tolerances apply.
- ffa_lse_combine: the result is one fp32 weighted sum rounded once to bf16,
  so |err| <= 2^-8 |ref| + 1e-5 (half a bf16 ulp, with room for the fp32
  exp / log of the weights), and lse |err| <= 1e-4.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from ffa_testlib import check_grad, check_out_lse, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffa():
    import torch
    assert torch.cuda.is_available()
    import __graft_entry__
    __graft_entry__.build()
    import flexible_mask_flashattention_gb300 as m
    return m


def tensors(S, hq, hkv, d, seed):
    t = W.make_tensors(S, hq, hkv, d, seed)
    t["v"] = (t["v"].float() * 0.5).to(t["v"].dtype)   # exact: a power-of-two scale of bf16 values
    return t


def split_cases():
    cases = []
    for seed in range(6):
        rng = np.random.default_rng(300 + seed)
        S = int(rng.integers(100, 700))
        sl = W.random_slices(seed + 400, S, S, max_segments=5, max_pieces=5)
        cases.append((f"random{seed}", S, sl[0::2], sl[1::2]))
    # one causal document split by keys: the first 200 keys, then the rest (two bottom-right causal
    # pieces with the same q-range give the whole causal triangle only together)
    S = 500
    a = [(0, S, 0, 200, O.FULL)]
    cases.append(("keys_split", S, [(200, S, 0, 200, O.FULL)], [(200, S, 200, S, O.CAUSAL)]))
    cases.append(("disjoint_rows", S, [(0, 250, 0, S, O.FULL)], [(250, S, 0, S, O.CAUSAL)]))   # no row in both
    cases.append(("empty_second", S, [(0, S, 0, S, O.CAUSAL)], []))
    cases.append(("empty_first", S, [], a))
    return cases


@pytest.mark.parametrize("case", split_cases(), ids=lambda c: c[0])
def test_fwd_accumulate_equals_union(ffa, case):
    import torch
    name, S, sa, sb = case
    hq, hkv, d = 4, 2, 128
    t = tensors(S, hq, hkv, d, 11)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    scale = 1.0 / np.sqrt(d)
    pa, pb = ffa.Plan(sa, S, S), ffa.Plan(sb, S, S)
    out, lse = ffa.fwd(q, k, v, pa, scale)
    ffa.fwd_accumulate(q, k, v, pb, scale, out, lse)
    pa.check_status()
    pb.check_status()
    torch.cuda.synchronize()
    r_out, r_lse = O.attention_forward(t["q"], t["k"], t["v"], list(sa) + list(sb), scale)
    check_out_lse(to_np(out), to_np(lse), r_out, r_lse, name)


def test_fwd_accumulate_three_parts_head_dim_64(ffa):
    import torch
    S, hq, hkv, d = 389, 3, 3, 64
    sl = W.random_slices(77, S, S, max_segments=4, max_pieces=6)
    parts = [sl[i::3] for i in range(3)]
    t = tensors(S, hq, hkv, d, 3)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    scale = 0.125
    plans = [ffa.Plan(p, S, S) for p in parts]
    out, lse = ffa.fwd(q, k, v, plans[0], scale)
    for p in plans[1:]:
        ffa.fwd_accumulate(q, k, v, p, scale, out, lse)
    torch.cuda.synchronize()
    r_out, r_lse = O.attention_forward(t["q"], t["k"], t["v"], sl, scale)
    check_out_lse(to_np(out), to_np(lse), r_out, r_lse, "three parts d=64")


def combine_ref(a, b):
    return O.lse_merge([(O.to_f64(a["out"]), O.to_f64(a["lse"])), (O.to_f64(b["out"]), O.to_f64(b["lse"]))])


def check_combine(out, lse, ref_out, ref_lse, what):
    out, lse = to_np(out).astype(np.float64), to_np(lse).astype(np.float64)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse)), what
    fin = np.isfinite(ref_lse)
    assert np.abs(lse[fin] - ref_lse[fin]).max(initial=0.0) <= 1e-4, what
    assert np.all(np.abs(out - ref_out) <= 2.0 ** -8 * np.abs(ref_out) + 1e-5), what


@pytest.mark.parametrize("S,hq,d", [(1, 1, 128), (1000, 4, 128), (777, 3, 64), (4099, 16, 128)])
def test_lse_combine_matches_oracle(ffa, S, hq, d):
    import torch
    a = W.make_partials(S, hq, d, seed=S + hq)
    b = W.make_partials(S, hq, d, seed=S + hq + 1, empty_frac=0.3)
    # rows empty in both parts, and rows with equal lse
    b["lse"][:, ::7] = a["lse"][:, ::7]
    b["lse"][0, ::5] = -np.inf
    a["lse"][0, ::5] = -np.inf
    ref_out, ref_lse = combine_ref(a, b)
    ga = {n: x.cuda() for n, x in a.items()}
    gb = {n: x.cuda() for n, x in b.items()}
    out, lse = ffa.lse_combine(ga["out"], ga["lse"], gb["out"], gb["lse"])
    torch.cuda.synchronize()
    check_combine(out, lse, ref_out, ref_lse, f"S={S} hq={hq} d={d}")
    # in place into a
    ffa.lse_combine(ga["out"], ga["lse"], gb["out"], gb["lse"], out=ga["out"], lse=ga["lse"])
    torch.cuda.synchronize()
    check_combine(ga["out"], ga["lse"], ref_out, ref_lse, "in place")


def test_fragment_backward_with_merged_result_equals_union(ffa):
    """The backward of a merged forward: each part's ffa_bwd, given the merged (out, lse), yields
    that part's share of dq / dk / dv; their sums equal the union's gradients."""
    import torch
    S, hq, hkv, d = 600, 4, 2, 128
    sl = W.random_slices(91, S, S, max_segments=4, max_pieces=5)
    sa, sb = sl[0::2], sl[1::2]
    t = tensors(S, hq, hkv, d, 21)
    g = {n: x.cuda() for n, x in t.items()}
    scale = 1.0 / np.sqrt(d)
    pa, pb = ffa.Plan(sa, S, S), ffa.Plan(sb, S, S)
    out, lse = ffa.fwd(g["q"], g["k"], g["v"], pa, scale)
    ffa.fwd_accumulate(g["q"], g["k"], g["v"], pb, scale, out, lse)
    ga = ffa.bwd(g["q"], g["k"], g["v"], out, lse, g["dout"], pa, scale)
    gb = ffa.bwd(g["q"], g["k"], g["v"], out, lse, g["dout"], pb, scale)
    torch.cuda.synchronize()
    ref = O.attention_backward(t["q"], t["k"], t["v"], t["dout"], sl, scale)
    for name, x, y, r in zip(("dq", "dk", "dv"), ga, gb, ref):
        check_grad(to_np(x).astype(np.float64) + to_np(y), r, name)


def test_argument_errors(ffa):
    import torch
    x = torch.zeros(10, 2, 96, dtype=torch.bfloat16, device="cuda")
    l = torch.zeros(2, 10, dtype=torch.float32, device="cuda")
    with pytest.raises(ffa.FFAError):
        ffa.lse_combine(x, l, x, l)                                  # head dim 96
    y = torch.zeros(10, 2, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ffa.FFAError):
        ffa.lse_combine(y, l, y, torch.zeros(2, 9, dtype=torch.float32, device="cuda"))   # lse shape
