"""Parity at the workloads' full sizes, in the launch configuration the bench
times (one plan, one ffa_fwd, one ffa_bwd over all heads).

A dense fp64 oracle cannot redo a 1M-token problem, so the row-by-row C
oracle (``oracle/rows_c.py``, pinned in test_oracle_rows.py) checks sampled
outputs, on every head:
  * out, lse and dq on 4096 random rows plus the first and last 64 rows of
    every slice's q-range;
  * dk and dv, for every kv head, on keys whose rows the oracle can afford:
      varlen causal    every key of the two shortest documents and the last
                       256 keys of the longest one;
      video            the first 128 keys of the last frame block and the
                       last 128 keys of the sequence;
      sink + window    the 1024 sink keys of the first document (every row of
                       the document attends them) and its last 256 keys.
The tiny workload is checked whole against the numpy oracle.  The 64K varlen
workload is also checked against the GPU's own per-document runs.  The same
tolerances as on small cases apply to each sampled set.
"""
import time

import numpy as np
import pytest

import oracle as O
import workloads as W
from ffa_testlib import check_grad, check_out_lse, to_np
from oracle import rows_c as R

pytestmark = pytest.mark.gpu

RANDOM_ROWS = 4096
EDGE_ROWS = 64


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
    """Keys for the dk / dv check."""
    S = w.seqlen
    if w.name.startswith("varlen"):
        by_len = sorted(doc_ranges(w), key=lambda r: (r[1] - r[0], r[0]))
        keys = [k for a, b in by_len[:2] for k in range(a, b)]
        a, b = by_len[-1]
        keys += list(range(b - 256, b))
        return sorted(set(keys))
    if w.name.startswith("video"):
        return list(range(S - 4096, S - 4096 + 128)) + list(range(S - 128, S))
    # sink + window: the first document's sink keys and last keys
    return list(range(0, 1024)) + list(range(32768 - 256, 32768))


def run_gpu(ffa, w, dev, slices=None):
    plan = ffa.Plan(w.slices if slices is None else slices, w.seqlen, w.seqlen)
    out, lse = ffa.fwd(dev["q"], dev["k"], dev["v"], plan, w.scale)
    grads = None
    if w.backward:
        grads = ffa.bwd(dev["q"], dev["k"], dev["v"], out, lse, dev["dout"], plan, w.scale)
    plan.check_status()
    return out, lse, grads


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
def test_workload_parity(ffa, name):
    import torch
    w = W.workload(name)
    S = w.seqlen
    if name == "tiny_mixed":
        t = W.make_tensors(S, w.hq, w.hkv, w.d, w.seed, with_dout=False)
        dev = {n: x.cuda() for n, x in t.items()}
        out, lse, _ = run_gpu(ffa, w, dev)
        torch.cuda.synchronize()
        r_out, r_lse = O.attention_forward(t["q"], t["k"], t["v"], w.slices, w.scale)
        check_out_lse(to_np(out), to_np(lse), r_out, r_lse, name)
        return

    dev = W.make_tensors(S, w.hq, w.hkv, w.d, w.seed, device="cuda", with_dout=w.backward)
    out, lse, (dq, dk, dv) = run_gpu(ffa, w, dev)
    torch.cuda.synchronize()
    for x in (out, lse, dq, dk, dv):
        assert not torch.isnan(x).any()

    rows = W.sample_rows(S, RANDOM_ROWS, w.seed + 17, slices=w.slices, edge=EDGE_ROWS)
    keys = key_sample(w)
    ridx = torch.tensor(rows, device="cuda")
    kidx = torch.tensor(keys, device="cuda")
    g_out, g_lse, g_dq = to_np(out[ridx]), to_np(lse[:, ridx]), to_np(dq[ridx])
    g_dk, g_dv = to_np(dk[kidx]), to_np(dv[kidx])
    host = {n: x.cpu() for n, x in dev.items()}
    del dev, out, lse, dq, dk, dv
    torch.cuda.empty_cache()

    t0 = time.time()
    r_out, r_lse, r_dq = R.attention_rows(host["q"], host["k"], host["v"], w.slices, w.scale, rows, dout=host["dout"])
    t1 = time.time()
    r_dk, r_dv = R.attention_keys(host["q"], host["k"], host["v"], host["dout"], w.slices, w.scale, keys)
    t2 = time.time()
    print(f"\n{name}: oracle rows {len(rows)} x {w.hq} heads {t1 - t0:.1f} s, "
          f"keys {len(keys)} x {w.hkv} kv heads {t2 - t1:.1f} s")
    check_out_lse(g_out, g_lse, r_out, r_lse, f"{name} (rows {len(rows)}, all heads)")
    check_grad(g_dq, r_dq, f"{name} dq (rows {len(rows)}, all heads)")
    check_grad(g_dk, r_dk, f"{name} dk (keys {len(keys)}, all kv heads)")
    check_grad(g_dv, r_dv, f"{name} dv (keys {len(keys)}, all kv heads)")


def test_varlen_equals_gpu_per_document(ffa):
    """The 64K varlen-causal result equals the GPU's runs over each document alone
    (its slice alone, on the same packed tensors)."""
    import torch
    w = W.workload("varlen_causal_64k")
    dev = W.make_tensors(w.seqlen, w.hq, w.hkv, w.d, w.seed, device="cuda", with_dout=True)
    out, lse, (dq, dk, dv) = run_gpu(ffa, w, dev)
    for s in w.slices:
        r = slice(s.q_start, s.q_end)
        o1, l1, (dq1, dk1, dv1) = run_gpu(ffa, w, dev, slices=[s])
        torch.cuda.synchronize()
        check_out_lse(to_np(out[r]), to_np(lse[:, r]), to_np(o1[r]).astype(np.float64),
                      to_np(l1[:, r]).astype(np.float64), f"doc {s.q_start}")
        check_grad(to_np(dq[r]), to_np(dq1[r]).astype(np.float64), f"doc {s.q_start} dq")
        check_grad(to_np(dk[r]), to_np(dk1[r]).astype(np.float64), f"doc {s.q_start} dk")
        check_grad(to_np(dv[r]), to_np(dv1[r]).astype(np.float64), f"doc {s.q_start} dv")
