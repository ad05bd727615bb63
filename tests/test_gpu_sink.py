"""GPU parity of the attention sink (ffa_fwd_sink, ffa_bwd_sink) against the
fp64 oracle: every row's softmax also holds a per-head logit with a zero value
vector.  out / lse use the forward tolerances; dq / dk / dv and the sink
gradient the relative Frobenius bound of the gradients."""
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


def run(ffa, slices, S, hq, hkv, d, seed, sink, backward=True):
    import torch
    t = W.make_tensors(S, hq, hkv, d, seed)
    g = {n: x.cuda() for n, x in t.items()}
    sk = torch.tensor(sink, dtype=torch.float32, device="cuda")
    scale = 1.0 / np.sqrt(d)
    plan = ffa.Plan(slices, S, S)
    out, lse = ffa.fwd_sink(g["q"], g["k"], g["v"], plan, scale, sk)
    res = {"out": to_np(out), "lse": to_np(lse)}
    if backward:
        dq, dk, dv, ds = ffa.bwd_sink(g["q"], g["k"], g["v"], out, lse, g["dout"], plan, scale, sk)
        res.update(dq=to_np(dq), dk=to_np(dk), dv=to_np(dv), dsink=to_np(ds))
    plan.check_status()
    torch.cuda.synchronize()
    sink64 = np.asarray(sink, dtype=np.float64)
    r_out, r_lse = O.attention_forward(t["q"], t["k"], t["v"], slices, scale, sink=sink64)
    check_out_lse(res["out"], res["lse"], r_out, r_lse, "sink forward")
    if backward:
        rq, rk, rv = O.attention_backward(t["q"], t["k"], t["v"], t["dout"], slices, scale, sink=sink64)
        rs = O.sink_gradient(t["q"], t["k"], t["v"], t["dout"], slices, scale, sink64)
        check_grad(res["dq"], rq, "dq")
        check_grad(res["dk"], rk, "dk")
        check_grad(res["dv"], rv, "dv")
        check_grad(res["dsink"], rs, "dsink")
    return res


@pytest.mark.parametrize("mtype", [O.FULL, O.CAUSAL, O.INV_CAUSAL, O.BI_CAUSAL])
def test_sink_each_mask_type(ffa, mtype):
    S = 333
    run(ffa, [(0, S, 0, S - 40, mtype)], S, 4, 2, 128, 5 + mtype, [0.5, -1.0, 3.0, -30.0])


@pytest.mark.parametrize("seed", range(4))
def test_sink_random_slices(ffa, seed):
    rng = np.random.default_rng(500 + seed)
    S = int(rng.integers(50, 700))
    hq, hkv = [(2, 1), (4, 4), (6, 2), (3, 3)][seed]
    sl = W.random_slices(seed + 600, S, S, max_segments=5, max_pieces=5)
    run(ffa, sl, S, hq, hkv, 128, seed, list(rng.normal(0, 3, hq)))


def test_sink_dominates_and_vanishes(ffa):
    S = 257
    sl = W.varlen_slices([100, 57, 100])
    res = run(ffa, sl, S, 2, 2, 128, 9, [40.0, -60.0])
    assert np.abs(res["out"][:, 0]).max() < 1e-6          # sink 40 takes every row's weight
    assert np.allclose(res["lse"][0], 40.0, atol=1e-3)


def test_sink_head_dim_64(ffa):
    S = 389
    sl = W.random_slices(77, S, S, max_segments=4, max_pieces=4)
    run(ffa, sl, S, 3, 3, 64, 3, [0.0, 1.0, -2.0])


def test_sink_with_no_keys_at_all(ffa):
    import torch
    S, hq, d = 200, 2, 128
    t = W.make_tensors(S, hq, hq, d, 1)
    g = {n: x.cuda() for n, x in t.items()}
    sk = torch.tensor([1.5, -0.5], dtype=torch.float32, device="cuda")
    plan = ffa.Plan([], S, S)
    out, lse = ffa.fwd_sink(g["q"], g["k"], g["v"], plan, 0.1, sk)
    dq, dk, dv, ds = ffa.bwd_sink(g["q"], g["k"], g["v"], out, lse, g["dout"], plan, 0.1, sk)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(lse == sk[:, None])
    assert torch.all(dq == 0) and torch.all(dk == 0) and torch.all(dv == 0) and torch.all(ds == 0)
