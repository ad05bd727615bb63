"""The persistent kernels' scheduling and the plan's per-direction tiles, on a GB300.

* Each CTA of the forward and backward main kernel starts with unit
  blockIdx.x and then pops units from one counter.  The per-CTA trace
  (ffa_plan_enable_cta_trace) shows every CTA's units and blocks: over all
  CTAs they must add up to exactly the plan's work (each unit taken once),
  with one CTA per SM at most, and the results must still match the oracle.
* ffa_tile_cfg: a plan whose backward tiles are not 128 x 128 still serves
  the forward; the backward refuses it, and so does the forward for
  non-128 forward tiles.
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


@pytest.mark.parametrize("hq,hkv", [(8, 2), (6, 6), (5, 1)])
def test_every_unit_taken_once(ffa, hq, hkv):
    import torch
    S, d = 3000, 128
    lengths = W.doc_lengths(S, 200, 1500, "uniform", 11)
    sl = W.varlen_slices(lengths)
    t = W.make_tensors(S, hq, hkv, d, 12)
    dev = {n: x.cuda() for n, x in t.items()}
    plan = ffa.Plan(sl, S, S)
    plan.enable_cta_trace(True)
    scale = 1.0 / np.sqrt(d)
    out, lse = ffa.fwd(dev["q"], dev["k"], dev["v"], plan, scale)
    dq, dk, dv = ffa.bwd(dev["q"], dev["k"], dev["v"], out, lse, dev["dout"], plan, scale)
    plan.check_status()
    torch.cuda.synchronize()
    info = plan.info()
    sms = torch.cuda.get_device_properties(0).multi_processor_count

    # forward units: (q-tile, head pair) with at least one block
    fo, fi, mo, mi, _ = plan.csr("q2k")
    blocks_per_tile = np.diff(fo) + np.diff(mo)
    pairs = (hq + 1) // 2
    tr = plan.read_cta_trace("fwd").astype(np.int64)
    assert 0 < len(tr) <= sms and len(tr) == min(info["m_tiles"] * pairs, sms)
    assert np.all(tr[:, 1] >= tr[:, 0])
    assert tr[:, 2].sum() == np.count_nonzero(blocks_per_tile) * pairs
    assert tr[:, 3].sum() == blocks_per_tile.sum() * pairs

    # backward units: (work item, kv head); blocks counted once per q head of the group
    items = plan.bwd_items()
    item_blocks = (items[:, 3] & 0xffff) + (items[:, 3] >> 16)
    tr = plan.read_cta_trace("bwd_main").astype(np.int64)
    assert 0 < len(tr) <= sms and len(tr) == min(len(items) * hkv, sms)
    assert np.all(tr[:, 1] >= tr[:, 0])
    assert tr[:, 2].sum() == len(items) * hkv
    assert tr[:, 3].sum() == item_blocks.sum() * hkv * (hq // hkv)
    k2q = plan.csr("k2q")
    assert item_blocks.sum() == len(k2q[1]) + len(k2q[3])

    # and the results are the oracle's
    r_out, r_lse = O.attention_forward(t["q"], t["k"], t["v"], sl, scale)
    check_out_lse(to_np(out), to_np(lse), r_out, r_lse, "traced forward")
    r_dq, r_dk, r_dv = O.attention_backward(t["q"], t["k"], t["v"], t["dout"], sl, scale)
    for name, g, r in (("dq", dq, r_dq), ("dk", dk, r_dk), ("dv", dv, r_dv)):
        check_grad(to_np(g), r, f"traced {name}")
    plan.enable_cta_trace(False)
    assert len(plan.read_cta_trace("fwd")) == 0


def test_every_unit_taken_once_head_pair_major(ffa):
    """From 2048 q-tiles on, the forward orders its units head pair by head
    pair; the trace must still add up to the plan's work, and sampled rows of
    every head must match the oracle."""
    import torch
    from oracle import rows_c as R
    S, hq, hkv, d = 2048 * 128, 6, 2, 128
    lengths = W.doc_lengths(S, 300, 6000, "uniform", 31)
    sl = W.varlen_slices(lengths)
    dev = W.make_tensors(S, hq, hkv, d, 32, device="cuda", with_dout=False)
    plan = ffa.Plan(sl, S, S)
    assert plan.info()["m_tiles"] >= 2048
    plan.enable_cta_trace(True)
    scale = 1.0 / np.sqrt(d)
    out, lse = ffa.fwd(dev["q"], dev["k"], dev["v"], plan, scale)
    plan.check_status()
    torch.cuda.synchronize()
    fo, fi, mo, mi, _ = plan.csr("q2k")
    blocks_per_tile = np.diff(fo) + np.diff(mo)
    pairs = (hq + 1) // 2
    tr = plan.read_cta_trace("fwd").astype(np.int64)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert len(tr) == sms
    assert tr[:, 2].sum() == np.count_nonzero(blocks_per_tile) * pairs
    assert tr[:, 3].sum() == blocks_per_tile.sum() * pairs
    rows = W.sample_rows(S, 256, 33)
    ridx = torch.tensor(rows, device="cuda")
    g_out, g_lse = to_np(out[ridx]), to_np(lse[:, ridx])
    host = {n: x.cpu() for n, x in dev.items()}
    r_out, r_lse, _ = R.attention_rows(host["q"], host["k"], host["v"], sl, scale, rows)
    check_out_lse(g_out, g_lse, r_out, r_lse, "head-pair-major forward")
    plan.enable_cta_trace(False)


def test_head_dim_64_at_2048_q_tiles(ffa):
    """Head dim 64 on the paths large problems take: head-pair-major forward
    units (2048 q-tiles), the speculative exponentials of head pairs with their
    own K / V (MHA), and backward units that hold all of their k-tile's blocks
    (short documents) storing dK / dV.  Sampled rows and keys of every head
    against the row-by-row oracle."""
    import torch
    from oracle import rows_c as R
    S, hq, hkv, d = 2048 * 128, 4, 4, 64
    lengths = W.doc_lengths(S, 200, 3000, "uniform", 41)
    sl = W.varlen_slices(lengths)
    dev = W.make_tensors(S, hq, hkv, d, 42, device="cuda", with_dout=True)
    scale = 1.0 / np.sqrt(d)
    plan = ffa.Plan(sl, S, S)
    out, lse = ffa.fwd(dev["q"], dev["k"], dev["v"], plan, scale)
    dq, dk, dv = ffa.bwd(dev["q"], dev["k"], dev["v"], out, lse, dev["dout"], plan, scale)
    plan.check_status()
    torch.cuda.synchronize()
    rows = W.sample_rows(S, 512, 43, slices=sl[:4], edge=8)
    # every key of the second document and of the last one
    keys = list(range(sl[1].k_start, sl[1].k_end)) + list(range(sl[-1].k_start, sl[-1].k_end))
    ridx, kidx = torch.tensor(rows, device="cuda"), torch.tensor(keys, device="cuda")
    g = {"out": to_np(out[ridx]), "lse": to_np(lse[:, ridx]), "dq": to_np(dq[ridx]),
         "dk": to_np(dk[kidx]), "dv": to_np(dv[kidx])}
    host = {n: x.cpu() for n, x in dev.items()}
    r_out, r_lse, r_dq = R.attention_rows(host["q"], host["k"], host["v"], sl, scale, rows, dout=host["dout"])
    r_dk, r_dv = R.attention_keys(host["q"], host["k"], host["v"], host["dout"], sl, scale, keys)
    check_out_lse(g["out"], g["lse"], r_out, r_lse, "d=64, 2048 q-tiles")
    check_grad(g["dq"], r_dq, "d=64, 2048 q-tiles dq")
    check_grad(g["dk"], r_dk, "d=64, 2048 q-tiles dk")
    check_grad(g["dv"], r_dv, "d=64, 2048 q-tiles dv")


def test_trace_is_off_by_default(ffa):
    import torch
    S = 256
    t = W.make_tensors(S, 2, 2, 64, 3, with_dout=False)
    plan = ffa.Plan([(0, S, 0, S, O.CAUSAL)], S, S)
    ffa.fwd(t["q"].cuda(), t["k"].cuda(), t["v"].cuda(), plan, 0.125)
    torch.cuda.synchronize()
    assert len(plan.read_cta_trace("fwd")) == 0 and len(plan.read_cta_trace("bwd_main")) == 0


def test_tiles_per_direction(ffa):
    import torch
    S, hq, hkv, d = 700, 4, 2, 128
    sl = W.random_slices(4, S, S)
    t = W.make_tensors(S, hq, hkv, d, 9)
    dev = {n: x.cuda() for n, x in t.items()}
    scale = 1.0 / np.sqrt(d)
    # backward tiles other than 128 x 128: the forward runs, the backward is refused
    plan = ffa.Plan(sl, S, S, 128, 128, bwd_block_m=64, bwd_block_n=256)
    info = plan.info()
    assert (info["fwd_bm"], info["fwd_bn"], info["bwd_bm"], info["bwd_bn"]) == (128, 128, 64, 256)
    out, lse = ffa.fwd(dev["q"], dev["k"], dev["v"], plan, scale)
    torch.cuda.synchronize()
    r_out, r_lse = O.attention_forward(t["q"], t["k"], t["v"], sl, scale)
    check_out_lse(to_np(out), to_np(lse), r_out, r_lse, "forward of a plan with 64 x 256 backward tiles")
    with pytest.raises(ffa.FFAError) as e:
        ffa.bwd(dev["q"], dev["k"], dev["v"], out, lse, dev["dout"], plan, scale)
    assert e.value.code == 4   # FFA_ERR_UNSUPPORTED
    # forward tiles other than 128 x 128: the forward is refused
    plan2 = ffa.Plan(sl, S, S, 64, 128, bwd_block_m=128, bwd_block_n=128)
    with pytest.raises(ffa.FFAError) as e:
        ffa.fwd(dev["q"], dev["k"], dev["v"], plan2, scale)
    assert e.value.code == 4
    plan.check_status()
    plan2.check_status()
