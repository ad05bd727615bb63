"""Pins of the oracle's row-by-row C implementation (``oracle/rows_c.py``).

It is checked against what does not depend on it:
  * torch's fp64 scaled_dot_product_attention (no mask, is_causal, explicit
    boolean masks from random slice lists) for out, torch.logsumexp of the
    masked scores for lse;
  * fp64 torch autograd of dense masked attention (GQA, rows without keys)
    for dq / dk / dv;
  * varlen causal equal to per-document causal attention;
  * the numpy oracle (``oracle.ffa_oracle``), itself pinned in test_oracle.py,
    on random slice lists of every mask type, ragged and non-square;
and rejects bad rows and keys.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from oracle import rows_c as R


def tensors(sq, hq, hkv, d, seed, sk=None):
    t = W.make_tensors(sq, hq, hkv, d, seed)
    if sk is not None and sk != sq:
        t2 = W.make_tensors(sk, hq, hkv, d, seed + 1000)
        t["k"], t["v"] = t2["k"], t2["v"]
    return t


def dense_reference(t, mask, scale):
    """fp64 torch attention over a dense boolean mask: out and lse (library
    routines: SDPA for out, logsumexp for lse), rows without keys give 0 / -inf."""
    q = torch.from_numpy(O.to_f64(t["q"])).permute(1, 0, 2)
    k = torch.from_numpy(O.to_f64(t["k"])).permute(1, 0, 2)
    v = torch.from_numpy(O.to_f64(t["v"])).permute(1, 0, 2)
    rep = q.shape[0] // k.shape[0]
    k, v = k.repeat_interleave(rep, 0), v.repeat_interleave(rep, 0)
    m = torch.from_numpy(mask)
    live = m.any(dim=1)
    safe = m | ~live[:, None]   # keep SDPA finite on empty rows; they are overwritten below
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=safe, scale=scale)
    out = torch.where(live[None, :, None], out, torch.zeros_like(out))
    s = scale * torch.einsum("hid,hjd->hij", q, k)
    lse = torch.logsumexp(torch.where(m[None], s, torch.tensor(-math.inf, dtype=torch.float64)), dim=-1)
    return out.permute(1, 0, 2).numpy(), lse.numpy()


def test_full_equals_sdpa():
    t = tensors(96, 4, 2, 16, 0)
    out, lse, _ = R.attention_rows(t["q"], t["k"], t["v"], [(0, 96, 0, 96, O.FULL)], 0.3, range(96))
    ref, rlse = dense_reference(t, np.ones((96, 96), dtype=bool), 0.3)
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, rlse, atol=1e-12, rtol=0)


def test_square_causal_equals_sdpa_is_causal():
    t = tensors(80, 2, 2, 8, 1)
    out, _, _ = R.attention_rows(t["q"], t["k"], t["v"], [(0, 80, 0, 80, O.CAUSAL)], 0.5, range(80))
    q, k, v = (torch.from_numpy(O.to_f64(t[n])).permute(1, 0, 2) for n in ("q", "k", "v"))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=0.5)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), atol=1e-12, rtol=0)


@pytest.mark.parametrize("seed", range(8))
def test_random_slices_equal_sdpa_masked(seed):
    sq, sk = 45 + 3 * seed, 61 - seed
    t = tensors(sq, 4, 2 if seed % 2 else 1, 8, seed, sk=sk)
    sl = W.random_slices(seed + 100, sq, sk)
    m = O.dense_mask(sl, sq, sk)
    out, lse, _ = R.attention_rows(t["q"], t["k"], t["v"], sl, 0.35, range(sq))
    ref, rlse = dense_reference(t, m, 0.35)
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)
    assert np.array_equal(np.isneginf(lse), np.isneginf(rlse))
    fin = np.isfinite(rlse)
    np.testing.assert_allclose(lse[fin], rlse[fin], atol=1e-12, rtol=0)


def test_varlen_causal_equals_per_document_attention():
    lengths = W.doc_lengths(300, 20, 90, "uniform", 7)
    S = sum(lengths)
    t = tensors(S, 2, 2, 8, 3)
    out, _, _ = R.attention_rows(t["q"], t["k"], t["v"], W.varlen_slices(lengths), 0.4, range(S))
    start = 0
    for L in lengths:
        seg = slice(start, start + L)
        q, k, v = (torch.from_numpy(O.to_f64(t[n][seg])).permute(1, 0, 2) for n in ("q", "k", "v"))
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=0.4)
        np.testing.assert_allclose(out[seg], ref.permute(1, 0, 2).numpy(), atol=1e-12, rtol=0)
        start += L


@pytest.mark.parametrize("seed", range(4))
def test_backward_matches_torch_autograd(seed):
    S, hq, hkv, d = 60 + 7 * seed, 4, 2 if seed % 2 else 4, 8
    t = tensors(S, hq, hkv, d, 11 + seed)
    sl = W.random_slices(5 + seed, S, S)
    if seed == 3:   # a row range without any slice: rows with no keys
        sl = [s for s in O.slice_tuples(sl) if s[1] <= S // 2 or s[0] >= S // 2 + 5]
    sc = 0.25
    m = torch.from_numpy(O.dense_mask(sl, S, S))
    q = torch.from_numpy(O.to_f64(t["q"])).requires_grad_()
    k = torch.from_numpy(O.to_f64(t["k"])).requires_grad_()
    v = torch.from_numpy(O.to_f64(t["v"])).requires_grad_()
    dout = torch.from_numpy(O.to_f64(t["dout"]))
    kr, vr = k.repeat_interleave(hq // hkv, 1), v.repeat_interleave(hq // hkv, 1)
    s = sc * torch.einsum("ihd,jhd->hij", q, kr)
    s = torch.where(m[None], s, torch.tensor(-math.inf, dtype=torch.float64))
    live = m.any(dim=1)
    p = torch.softmax(torch.where(live[None, :, None], s, torch.zeros_like(s)), dim=-1)
    p = torch.where(live[None, :, None] & m[None], p, torch.zeros_like(p))
    out = torch.einsum("hij,jhd->ihd", p, vr)
    (out * dout).sum().backward()
    _, _, dq = R.attention_rows(t["q"], t["k"], t["v"], sl, sc, range(S), dout=t["dout"])
    dk, dv = R.attention_keys(t["q"], t["k"], t["v"], t["dout"], sl, sc, range(S))
    for a, b in ((dq, q.grad), (dk, k.grad), (dv, v.grad)):
        np.testing.assert_allclose(a, b.numpy(), atol=1e-11, rtol=0)


@pytest.mark.parametrize("seed", range(6))
def test_equals_numpy_oracle(seed):
    """Both oracle implementations agree on ragged, non-square slice lists of every type."""
    sq, sk = 300 + 37 * seed, 260 + 51 * seed
    hq, hkv, d = (4, 2, 64) if seed % 2 else (3, 3, 32)
    t = tensors(sq, hq, hkv, d, seed, sk=sk)
    sl = W.random_slices(seed, sq, sk)
    rows = W.sample_rows(sq, 60, seed, slices=sl, edge=3)
    keys = sorted(set(range(0, sk, 7)) | {sk - 1})
    out, lse, dq = R.attention_rows(t["q"], t["k"], t["v"], sl, 0.1, rows, dout=t["dout"])
    dk, dv = R.attention_keys(t["q"], t["k"], t["v"], t["dout"], sl, 0.1, keys)
    r_out, r_lse = O.attention_forward(t["q"], t["k"], t["v"], sl, 0.1, rows=rows)
    r_dq, r_dk, r_dv = O.attention_backward(t["q"], t["k"], t["v"], t["dout"], sl, 0.1, rows=rows, keys=keys)
    assert np.array_equal(np.isneginf(lse), np.isneginf(r_lse))
    fin = np.isfinite(r_lse)
    np.testing.assert_allclose(lse[fin], r_lse[fin], atol=1e-12, rtol=0)
    for a, b in ((out, r_out), (dq, r_dq), (dk, r_dk), (dv, r_dv)):
        np.testing.assert_allclose(a, b, atol=1e-12, rtol=0)


def test_rejects_bad_rows_and_keys():
    t = tensors(32, 2, 1, 8, 0)
    sl = [(0, 32, 0, 32, O.CAUSAL)]
    with pytest.raises(RuntimeError):
        R.attention_rows(t["q"], t["k"], t["v"], sl, 0.1, [0, 32])
    with pytest.raises(RuntimeError):
        R.attention_keys(t["q"], t["k"], t["v"], t["dout"], sl, 0.1, [-1, 3])
