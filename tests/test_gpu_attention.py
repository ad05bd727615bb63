"""GPU forward / backward parity against the fp64 oracle on small and ragged
cases, element by element: every mask type, GQA and MHA head layouts (odd head
counts included), head dims 64 and 128, empty rows, empty slice lists,
lengths that are not multiples of the 128 tile, overlapping q-ranges."""
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


def run(ffa, slices, sq, sk, hq, hkv, d, seed, backward=True, scale=None):
    import torch
    scale = scale if scale is not None else 1.0 / np.sqrt(d)
    t = W.make_tensors(max(sq, sk), hq, hkv, d, seed)
    t = {"q": t["q"][:sq].contiguous(), "k": t["k"][:sk].contiguous(), "v": t["v"][:sk].contiguous(),
         "dout": t["dout"][:sq].contiguous()}
    dev = {n: x.cuda() for n, x in t.items()}
    plan = ffa.Plan(slices, sq, sk)
    out, lse = ffa.fwd(dev["q"], dev["k"], dev["v"], plan, scale)
    res = {"out": out, "lse": lse}
    if backward:
        res["dq"], res["dk"], res["dv"] = ffa.bwd(dev["q"], dev["k"], dev["v"], out, lse, dev["dout"], plan, scale)
    plan.check_status()
    torch.cuda.synchronize()
    return t, {n: to_np(x) for n, x in res.items()}, scale


def compare(t, g, slices, scale, backward=True, what=""):
    r_out, r_lse = O.attention_forward(t["q"], t["k"], t["v"], slices, scale)
    check_out_lse(g["out"], g["lse"], r_out, r_lse, what)
    if backward:
        r_dq, r_dk, r_dv = O.attention_backward(t["q"], t["k"], t["v"], t["dout"], slices, scale)
        check_grad(g["dq"], r_dq, what + " dq")
        check_grad(g["dk"], r_dk, what + " dk")
        check_grad(g["dv"], r_dv, what + " dv")


@pytest.mark.parametrize("mtype", [O.FULL, O.CAUSAL, O.INV_CAUSAL, O.BI_CAUSAL])
@pytest.mark.parametrize("shape", [(256, 256), (200, 333), (333, 200), (130, 130)])
def test_single_slice_each_type(ffa, mtype, shape):
    sq, sk = shape
    sl = [(0, sq, 0, sk, mtype)]
    t, g, sc = run(ffa, sl, sq, sk, 2, 1, 128, 7 + mtype)
    compare(t, g, sl, sc, what=f"type {mtype} {shape}")


@pytest.mark.parametrize("seed", range(12))
def test_random_slices(ffa, seed):
    rng = np.random.default_rng(100 + seed)
    sq, sk = int(rng.integers(1, 600)), int(rng.integers(1, 600))
    hq, hkv = [(1, 1), (2, 2), (3, 1), (4, 2), (6, 2), (4, 1), (5, 5), (8, 2)][seed % 8]
    sl = W.random_slices(seed + 50, sq, sk, max_segments=5, max_pieces=5)
    t, g, sc = run(ffa, sl, sq, sk, hq, hkv, 128, seed)
    compare(t, g, sl, sc, what=f"seed {seed}")


@pytest.mark.parametrize("hq,hkv", [(2, 2), (3, 3), (4, 1)])
def test_head_dim_64(ffa, hq, hkv):
    sq = sk = 389
    sl = W.random_slices(77, sq, sk, max_segments=4, max_pieces=4)
    t, g, sc = run(ffa, sl, sq, sk, hq, hkv, 64, 3)
    compare(t, g, sl, sc, what="d=64")


@pytest.mark.parametrize("mtype", [O.FULL, O.CAUSAL, O.INV_CAUSAL, O.BI_CAUSAL])
def test_head_dim_64_each_type(ffa, mtype):
    # GQA, ragged lengths, non-square slices: the backward's 64-dim path end to end
    sq, sk = 300, 420
    sl = [(0, sq, 0, sk, mtype)]
    t, g, sc = run(ffa, sl, sq, sk, 8, 2, 64, 11 + mtype)
    compare(t, g, sl, sc, what=f"d=64 type {mtype}")


def test_tiny_mixed_workload(ffa):
    w = W.workload("tiny_mixed")
    t, g, sc = run(ffa, w.slices, w.seqlen, w.seqlen, w.hq, w.hkv, w.d, w.seed)
    compare(t, g, w.slices, sc, what="tiny_mixed")


def test_empty_slice_list(ffa):
    t, g, sc = run(ffa, [], 300, 300, 2, 2, 128, 1)
    assert np.all(g["out"] == 0) and np.all(np.isneginf(g["lse"]))
    assert np.all(g["dq"] == 0) and np.all(g["dk"] == 0) and np.all(g["dv"] == 0)


def test_partly_covered_rows_and_keys(ffa):
    # rows 0..99 and 250..299 have no keys; keys 0..49 are never attended
    sl = [(100, 250, 50, 300, O.FULL)]
    t, g, sc = run(ffa, sl, 300, 300, 2, 1, 128, 2)
    compare(t, g, sl, sc, what="partial coverage")
    assert np.all(g["out"][:100] == 0) and np.all(np.isneginf(g["lse"][:, :100]))
    assert np.all(g["dk"][:50] == 0) and np.all(g["dv"][:50] == 0)


def test_overlapping_q_ranges_sink_window(ffa):
    sl = W.sink_window_slices(3, 320, 64, 96)
    t, g, sc = run(ffa, sl, 960, 960, 4, 4, 128, 4)
    compare(t, g, sl, sc, what="sink+window")


def test_varlen_causal_equals_per_document_runs(ffa):
    lengths = [130, 1, 257, 64, 300]
    S = sum(lengths)
    sl = W.varlen_slices(lengths)
    t, g, sc = run(ffa, sl, S, S, 2, 1, 128, 5)
    compare(t, g, sl, sc, what="varlen")
    start = 0
    for L in lengths:
        tt = {n: x[start:start + L] for n, x in t.items()}
        import torch
        plan = ffa.Plan([(0, L, 0, L, O.CAUSAL)], L, L)
        out, lse = ffa.fwd(*(tt[n].contiguous().cuda() for n in ("q", "k", "v")), plan, sc)
        # the packed run tiles the documents differently, so the two agree to rounding only
        check_out_lse(g["out"][start:start + L], g["lse"][:, start:start + L], to_np(out).astype(np.float64),
                      to_np(lse).astype(np.float64), f"doc of {L}")
        start += L


@pytest.mark.parametrize("order", ["rising", "mixed"])
@pytest.mark.parametrize("hq,hkv", [(2, 2), (2, 1), (3, 3)])
def test_running_max_raised_often(ffa, order, hq, hkv):
    """Keys scaled block by block, so that a row's max over a 128-key block
    exceeds its running max by far more than the lazy-rescale threshold on
    most blocks: O and the row sum are rescaled again and again, and on head
    pairs that load their own K / V tiles the speculative exponentials of a
    Full block are redone against the raised max."""
    import torch
    sq, sk, d = 200, 1000, 128
    t = W.make_tensors(sk, hq, hkv, d, 21)
    blocks = (sk + 127) // 128
    f = 1.0 + 4.0 * np.arange(blocks)
    if order == "mixed":
        f = f[np.random.default_rng(5).permutation(blocks)]
    scale_rows = torch.from_numpy(np.repeat(f, 128)[:sk]).float()[:, None, None]
    t["k"] = (t["k"].float() * scale_rows).to(torch.bfloat16)
    # Rows this peaked take their output from one or two keys, so |out| reaches
    # |v|; v is scaled by 1/4 to keep |out| < 2, where the bf16 rounding of the
    # output alone stays well inside the out bound (in [4, 8) it is 0.0156).
    t["v"] = (t["v"].float() * 0.25).to(torch.bfloat16)
    t = {"q": t["q"][:sq].contiguous(), "k": t["k"], "v": t["v"], "dout": t["dout"][:sq].contiguous()}
    sl = [(0, sq, 0, sk - 300, O.FULL), (0, sq, sk - 300, sk, O.CAUSAL)]
    dev = {n: x.cuda() for n, x in t.items()}
    sc = 1.0 / np.sqrt(d)
    plan = ffa.Plan(sl, sq, sk)
    out, lse = ffa.fwd(dev["q"], dev["k"], dev["v"], plan, sc)
    dq, dk, dv = ffa.bwd(dev["q"], dev["k"], dev["v"], out, lse, dev["dout"], plan, sc)
    plan.check_status()
    torch.cuda.synchronize()
    g = {"out": to_np(out), "lse": to_np(lse), "dq": to_np(dq), "dk": to_np(dk), "dv": to_np(dv)}
    compare(t, g, sl, sc, what=f"raised max {order} {hq}/{hkv}")


SWEEP_HEADS = [(2, 2), (4, 4), (4, 2), (6, 2), (3, 3), (8, 1)]


@pytest.mark.parametrize("case", range(40))
def test_random_sweep(ffa, case):
    """Random slice lists on random ragged, non-square shapes over six head
    layouts and both head dims; every fourth case with keys scaled block by
    block, so that the running max is raised on most blocks."""
    import torch
    rng = np.random.default_rng(2026 + case)
    sq, sk = int(rng.integers(200, 1600)), int(rng.integers(200, 1600))
    hq, hkv = SWEEP_HEADS[case % len(SWEEP_HEADS)]
    d = 64 if case % 3 == 0 else 128
    sl = W.random_slices(1000 + case, sq, sk)
    t = W.make_tensors(max(sq, sk), hq, hkv, d, 500 + case)
    t = {"q": t["q"][:sq].contiguous(), "k": t["k"][:sk].contiguous(), "v": t["v"][:sk].contiguous(),
         "dout": t["dout"][:sq].contiguous()}
    if case % 4 == 1:
        f = 1.0 + 3.0 * np.arange((sk + 127) // 128)
        rows = torch.from_numpy(np.repeat(f, 128)[:sk]).float()[:, None, None]
        t["k"] = (t["k"].float() * rows).to(torch.bfloat16)
        t["v"] = (t["v"].float() * 0.25).to(torch.bfloat16)   # keeps |out| < 2 (output rounding)
    dev = {n: x.cuda() for n, x in t.items()}
    sc = 1.0 / np.sqrt(d)
    plan = ffa.Plan(sl, sq, sk)
    out, lse = ffa.fwd(dev["q"], dev["k"], dev["v"], plan, sc)
    dq, dk, dv = ffa.bwd(dev["q"], dev["k"], dev["v"], out, lse, dev["dout"], plan, sc)
    plan.check_status()
    torch.cuda.synchronize()
    g = {"out": to_np(out), "lse": to_np(lse), "dq": to_np(dq), "dk": to_np(dk), "dv": to_np(dv)}
    compare(t, g, sl, sc, what=f"sweep {case} ({sq}x{sk}, {hq}/{hkv}, d={d})")


def test_single_token_and_long_row(ffa):
    t, g, sc = run(ffa, [(0, 1, 0, 1, O.FULL)], 1, 1, 1, 1, 128, 9)
    compare(t, g, [(0, 1, 0, 1, O.FULL)], sc, what="1 token")
    sl = [(0, 3, 0, 5000, O.FULL)]
    t, g, sc = run(ffa, sl, 3, 5000, 2, 1, 128, 10)
    compare(t, g, sl, sc, what="long rows")


def test_argument_errors(ffa):
    import torch
    q = torch.zeros(256, 2, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(256, 2, 128, dtype=torch.bfloat16, device="cuda")
    plan = ffa.Plan([(0, 256, 0, 256, O.CAUSAL)], 256, 256)
    with pytest.raises(ffa.FFAError):
        ffa.fwd(q[:255], k, k, plan, 1.0)                         # seqlen mismatch with the plan
    with pytest.raises(ffa.FFAError):
        ffa.fwd(torch.zeros(256, 3, 128, dtype=torch.bfloat16, device="cuda"), k, k, plan, 1.0)   # 3 % 2 != 0
    with pytest.raises(ffa.FFAError):
        ffa.fwd(torch.zeros(256, 2, 96, dtype=torch.bfloat16, device="cuda"),
                torch.zeros(256, 2, 96, dtype=torch.bfloat16, device="cuda"),
                torch.zeros(256, 2, 96, dtype=torch.bfloat16, device="cuda"), plan, 1.0)      # head dim 96
    small = ffa.Plan([(0, 256, 0, 256, O.CAUSAL)], 256, 256, 64, 64)
    with pytest.raises(ffa.FFAError):
        ffa.fwd(q, k, k, small, 1.0)                              # tiles must be 128 x 128
    plan.check_status()
