"""Parity at the workloads' full sizes, in the launch configuration the bench
times (one plan, one ffa_fwd, one ffa_bwd over all heads).

The fp64 oracle cannot redo a 1M-token problem, so it checks sampled outputs:
out / lse / dq on 1024 random rows plus the first and last 16 rows of every
slice's q-range, and dk / dv on keys few rows attend (whole short documents,
the last keys of the longest one).  On the GQA workloads the oracle takes one
kv-head group (the last), on the MHA ones the last two heads.  The same
tolerances as on small cases apply.
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


def doc_ranges(w):
    """Distinct q-ranges of the slices, as (start, end) pairs."""
    return sorted({(s.q_start, s.q_end) for s in w.slices})


def key_sample(w):
    """Keys for the dk / dv check, chosen so that few rows attend them."""
    docs = doc_ranges(w)
    if w.name.startswith("varlen"):
        by_len = sorted(docs, key=lambda r: r[1] - r[0])
        keys = [k for a, b in by_len[:2] for k in range(a, b)]
        a, b = by_len[-1]
        keys += list(range(b - 256, b))
        return sorted(set(keys))
    if w.name.startswith("video"):
        return list(range(w.seqlen - 256, w.seqlen))
    # sink + window: the last keys of the first document (window keys only;
    # the sink keys, which every row of a document attends, are checked on the
    # small sink-and-window case of the attention tests)
    return list(range(32768 - 256, 32768))


def oracle_heads(w):
    """The q-head and kv-head ranges the oracle recomputes: one kv group for
    GQA (all its q heads, since dk / dv sum over them), the last two heads for MHA."""
    G = w.hq // w.hkv
    if G > 1:
        g = w.hkv - 1
        return slice(g * G, (g + 1) * G), slice(g, g + 1)
    return slice(w.hq - 2, w.hq), slice(w.hkv - 2, w.hkv)


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
def test_workload_parity(ffa, name):
    import torch
    w = W.workload(name)
    S = w.seqlen
    if name == "tiny_mixed":
        t = W.make_tensors(S, w.hq, w.hkv, w.d, w.seed, with_dout=False)
        dev = {n: x.cuda() for n, x in t.items()}
    else:
        dev = W.make_tensors(S, w.hq, w.hkv, w.d, w.seed, device="cuda", with_dout=w.backward)
    plan = ffa.Plan(w.slices, S, S)
    out, lse = ffa.fwd(dev["q"], dev["k"], dev["v"], plan, w.scale)
    if w.backward:
        dq, dk, dv = ffa.bwd(dev["q"], dev["k"], dev["v"], out, lse, dev["dout"], plan, w.scale)
    plan.check_status()
    torch.cuda.synchronize()

    if name == "tiny_mixed":
        r_out, r_lse = O.attention_forward(t["q"], t["k"], t["v"], w.slices, w.scale)
        check_out_lse(to_np(out), to_np(lse), r_out, r_lse, name)
        return

    hs, ks = oracle_heads(w)
    host = {n: x[:, hs if n in ("q", "dout") else ks].cpu() for n, x in dev.items()}

    rows = W.sample_rows(S, 1024, w.seed + 17, slices=w.slices, edge=16)
    r_out, r_lse = O.attention_forward(host["q"], host["k"], host["v"], w.slices, w.scale, rows=rows)
    g_out = to_np(out[rows][:, hs])
    g_lse = to_np(lse[hs][:, rows])
    check_out_lse(g_out, g_lse, r_out, r_lse, f"{name} (rows {len(rows)})")

    keys = key_sample(w)
    r_dq, r_dk, r_dv = O.attention_backward(host["q"], host["k"], host["v"], host["dout"], w.slices, w.scale,
                                            rows=rows, keys=keys)
    check_grad(to_np(dq[rows][:, hs]), r_dq, f"{name} dq")
    check_grad(to_np(dk[keys][:, ks]), r_dk, f"{name} dk")
    check_grad(to_np(dv[keys][:, ks]), r_dv, f"{name} dv")
    # every key without any query has zero gradient; no NaN anywhere
    for x in (out, lse, dq, dk, dv):
        assert not torch.isnan(x).any()
