"""Pins for the fp64 oracle against facts the pages and mathematics fix.

Nothing here checks the oracle against itself: masks against hand-written
fixtures and the pages' area formulas, the forward against torch's SDPA (an
independent library routine) and per-document attention, the backward against
finite differences and torch autograd, the block classifier against brute
force and closed-form block counts.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from conftest import golden_lines

TYPES = {"FULL": O.FULL, "CAUSAL": O.CAUSAL, "INV_CAUSAL": O.INV_CAUSAL, "BI_CAUSAL": O.BI_CAUSAL}


# ----------------------------------------------------------------------------
# masks and areas
# ----------------------------------------------------------------------------

def local_mask(t, lq, lk):
    return O.dense_mask([(0, lq, 0, lk, t)], lq, lk)


def test_golden_slice_masks():
    n = 0
    for tname, lq, lk, *rows in golden_lines("slice_masks.txt"):
        lq, lk = int(lq), int(lk)
        want = np.array([[ch == "1" for ch in r] for r in rows], dtype=bool)
        assert want.shape == (lq, lk)
        assert np.array_equal(local_mask(TYPES[tname], lq, lk), want), (tname, lq, lk)
        n += 1
    assert n >= 10


def test_page_area_formulas():
    for _, n, full, causal in (l for l in golden_lines("areas.txt") if l[0] == "page_formula"):
        n, full, causal = int(n), int(full), int(causal)
        assert O.mask_area_closed_form(n, n, O.FULL) == full
        assert O.mask_area_closed_form(n, n, O.CAUSAL) == causal
        if n <= 128:
            assert int(local_mask(O.FULL, n, n).sum()) == full
            assert int(local_mask(O.CAUSAL, n, n).sum()) == causal
            assert int(local_mask(O.INV_CAUSAL, n, n).sum()) == causal


def test_closed_form_areas_match_brute_force():
    for lq, lk in itertools.product(range(0, 33), repeat=2):
        for t in TYPES.values():
            assert O.mask_area_closed_form(lq, lk, t) == int(local_mask(t, lq, lk).sum()), (t, lq, lk)


def test_reversal_and_intersection_identities():
    for lq, lk in itertools.product(range(1, 20), repeat=2):
        c = local_mask(O.CAUSAL, lq, lk)
        inv = local_mask(O.INV_CAUSAL, lq, lk)
        bi = local_mask(O.BI_CAUSAL, lq, lk)
        assert np.array_equal(inv, c[::-1, ::-1])        # reversing both axes swaps the corners
        assert np.array_equal(bi, c & inv)


def test_bi_causal_is_sliding_window():
    # A BI-CAUSAL slice with Lk = Lq + W - 1 whose keys start W - 1 before its
    # queries is the textbook window: query i sees keys i-W+1 .. i.  The first
    # W rows take a square CAUSAL slice (the sink-and-window workload's layout).
    S, W = 40, 7
    sl = [(0, W, 0, W, O.CAUSAL), (W, S, 1, S, O.BI_CAUSAL)]
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    assert np.array_equal(O.dense_mask(sl, S, S), (j <= i) & (j > i - W))


def test_workload_areas_golden():
    rows = {l[1]: l[2:] for l in golden_lines("areas.txt") if l[0] == "workload"}
    for name, (area, hq, d, flops) in rows.items():
        w = W.workload(name)
        assert O.slices_area(w.slices) == int(area)
        assert O.fwd_flops(int(area), int(hq), int(d)) == int(flops)
        assert w.hq == int(hq) and w.d == int(d)
    w = W.workload("tiny_mixed")
    assert O.mask_area(w.slices, w.seqlen, w.seqlen) == int(rows["tiny_mixed"][0])
    for name in ("video_block_causal_128k", "sink_window_256k"):
        w = W.workload(name)
        _, _, cnt = O.block_counts_from_intervals(w.slices, w.seqlen, w.seqlen, 128, 128)
        assert int(cnt.sum()) == int(rows[name][0])


def test_workload_slice_coverage_is_disjoint():
    w = W.workload("tiny_mixed")
    assert O.coverage_is_disjoint(w.slices, w.seqlen, w.seqlen)
    small = W.sink_window_slices(2, 64, 8, 16)
    assert O.coverage_is_disjoint(small, 128, 128)
    assert O.mask_area(small, 128, 128) == O.slices_area(small)
    for seed in range(20):
        sl = W.random_slices(seed, 70, 90)
        assert O.coverage_is_disjoint(sl, 70, 90)
    # and a genuinely doubly covered pair is seen
    assert not O.coverage_is_disjoint([(0, 4, 0, 4, O.FULL), (2, 3, 3, 5, O.FULL)], 4, 5)


def test_row_intervals_match_dense_mask():
    for seed in range(30):
        sq, sk = 37 + seed, 53 - seed // 2
        sl = W.random_slices(seed, sq, sk)
        row, lo, hi = O.row_intervals(sl, sq)
        m = np.zeros((sq, sk), dtype=bool)
        for r, a, b in zip(row, lo, hi):
            assert not m[r, a:b].any()
            m[r, a:b] = True
        assert np.array_equal(m, O.dense_mask(sl, sq, sk))


def test_flop_formulas():
    assert O.fwd_flops(10, 3, 8) == 2 * 2 * 10 * 3 * 8
    assert O.bwd_flops(10, 3, 8) == 2.5 * 2 * 2 * 10 * 3 * 8


# ----------------------------------------------------------------------------
# forward
# ----------------------------------------------------------------------------

def tensors(S, hq, hkv, d, seed, sk=None):
    t = W.make_tensors(S, hq, hkv, d, seed)
    if sk is not None and sk != S:
        t2 = W.make_tensors(sk, hq, hkv, d, seed + 1000)
        t["k"], t["v"] = t2["k"], t2["v"]
    return t


def sdpa_heads(q, k, v, scale, attn_mask=None, is_causal=False):
    """fp64 torch SDPA per head with GQA by repeating kv heads; -> [S, H, d]."""
    qf = torch.from_numpy(O.to_f64(q)).permute(1, 0, 2)
    kf = torch.from_numpy(O.to_f64(k)).permute(1, 0, 2)
    vf = torch.from_numpy(O.to_f64(v)).permute(1, 0, 2)
    rep = qf.shape[0] // kf.shape[0]
    kf, vf = kf.repeat_interleave(rep, 0), vf.repeat_interleave(rep, 0)
    m = None if attn_mask is None else torch.from_numpy(attn_mask)
    o = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, attn_mask=m, is_causal=is_causal,
                                                         scale=scale)
    return o.permute(1, 0, 2).numpy()


def test_forward_full_equals_sdpa():
    t = tensors(96, 4, 2, 16, 0)
    sc = 0.3
    out, lse = O.attention_forward(t["q"], t["k"], t["v"], [(0, 96, 0, 96, O.FULL)], sc)
    np.testing.assert_allclose(out, sdpa_heads(t["q"], t["k"], t["v"], sc), atol=1e-12, rtol=0)
    q, k = O.to_f64(t["q"]), O.to_f64(t["k"])
    for h in range(4):
        s = sc * q[:, h, :] @ k[:, h // 2, :].T
        want = np.log(np.exp(s).sum(axis=1))
        np.testing.assert_allclose(lse[h], want, atol=1e-12, rtol=0)


def test_forward_square_causal_equals_sdpa_causal():
    t = tensors(80, 2, 2, 8, 1)
    out, _ = O.attention_forward(t["q"], t["k"], t["v"], [(0, 80, 0, 80, O.CAUSAL)], 0.5)
    np.testing.assert_allclose(out, sdpa_heads(t["q"], t["k"], t["v"], 0.5, is_causal=True),
                               atol=1e-12, rtol=0)


def test_forward_random_slices_equals_sdpa_masked():
    for seed in range(8):
        sq, sk = 45 + 3 * seed, 61 - seed
        t = tensors(sq, 4, 1, 8, seed, sk=sk)
        sl = W.random_slices(seed + 100, sq, sk)
        m = O.dense_mask(sl, sq, sk)
        out, lse = O.attention_forward(t["q"], t["k"], t["v"], sl, 0.35)
        ref = sdpa_heads(t["q"], t["k"], t["v"], 0.35, attn_mask=m)
        live = m.any(axis=1)
        np.testing.assert_allclose(out[live], ref[live], atol=1e-12, rtol=0)
        assert np.all(out[~live] == 0) and np.all(np.isneginf(lse[:, ~live]))


def test_varlen_causal_equals_per_document_attention():
    lengths = W.doc_lengths(300, 20, 90, "uniform", 7)
    S = sum(lengths)
    t = tensors(S, 2, 2, 8, 3)
    out, lse = O.attention_forward(t["q"], t["k"], t["v"], W.varlen_slices(lengths), 0.4)
    start = 0
    for L in lengths:
        seg = slice(start, start + L)
        ref = sdpa_heads(t["q"][seg], t["k"][seg], t["v"][seg], 0.4, is_causal=True)
        np.testing.assert_allclose(out[seg], ref, atol=1e-12, rtol=0)
        start += L


def test_lse_merge_of_slice_groups_equals_union():
    for seed in range(6):
        S = 64
        t = tensors(S, 2, 2, 8, seed)
        sl = W.random_slices(seed + 7, S, S, max_segments=2, max_pieces=5)
        if len(sl) < 2:
            continue
        full = O.attention_forward(t["q"], t["k"], t["v"], sl, 0.3)
        parts = [O.attention_forward(t["q"], t["k"], t["v"], sl[i::2], 0.3) for i in range(2)]
        out, lse = O.lse_merge(parts)
        np.testing.assert_allclose(out, full[0], atol=1e-12, rtol=0)
        assert np.array_equal(np.isneginf(lse), np.isneginf(full[1]))
        np.testing.assert_allclose(np.where(np.isfinite(lse), lse, 0), np.where(np.isfinite(full[1]), full[1], 0),
                                   atol=1e-12, rtol=0)


def test_lse_merge_closed_forms():
    # lse_a = 0, lse_b = ln 3: weights 1/4 and 3/4, merged lse = ln 4
    oa = np.full((1, 1, 2), 1.0)
    ob = np.array([[[5.0, -3.0]]])
    out, lse = O.lse_merge([(oa, np.array([[0.0]])), (ob, np.array([[np.log(3.0)]]))])
    np.testing.assert_allclose(out, [[[4.0, -2.0]]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, [[np.log(4.0)]], rtol=0, atol=1e-15)
    # equal lse: the plain average, lse + ln 2
    out, lse = O.lse_merge([(oa, np.array([[1.5]])), (ob, np.array([[1.5]]))])
    np.testing.assert_allclose(out, [[[3.0, -1.0]]], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, [[1.5 + np.log(2.0)]], rtol=0, atol=1e-15)


def test_lse_merge_empty_parts_and_symmetry():
    rng = np.random.default_rng(5)
    R, H, d = 7, 3, 4
    parts = []
    for _ in range(3):
        o = rng.standard_normal((R, H, d))
        l = rng.standard_normal((H, R)) * 3
        l[rng.random((H, R)) < 0.3] = -np.inf
        o[np.isneginf(l).T] = np.nan   # an empty part's out must never be read
        parts.append((o, l))
    empty = (np.full((R, H, d), np.nan), np.full((H, R), -np.inf))
    for o, l in parts:
        out, lse = O.lse_merge([(o, l), empty])
        fin = np.isfinite(l).T
        np.testing.assert_array_equal(out[fin], o[fin])
        assert np.all(out[~fin] == 0) and np.array_equal(np.isneginf(lse), np.isneginf(l))
    ab, _ = O.lse_merge(parts[:2])
    ba, _ = O.lse_merge(parts[1::-1])
    np.testing.assert_allclose(ab, ba, rtol=0, atol=1e-12)
    # associativity: ((a, b), c) == (a, (b, c)) == (a, b, c)
    x = O.lse_merge([O.lse_merge(parts[:2]), parts[2]])
    y = O.lse_merge([parts[0], O.lse_merge(parts[1:])])
    z = O.lse_merge(parts)
    for u in (x, y):
        np.testing.assert_allclose(np.nan_to_num(u[0]), np.nan_to_num(z[0]), rtol=0, atol=1e-12)
        np.testing.assert_array_equal(np.isneginf(u[1]), np.isneginf(z[1]))
    # the weights sum to one wherever some part is non-empty
    w = sum(np.where(np.isfinite(l), np.exp(l - np.where(np.isfinite(z[1]), z[1], 0)), 0) for _, l in parts)
    np.testing.assert_allclose(w[np.isfinite(z[1])], 1.0, rtol=0, atol=1e-12)


def dispatch_fixtures():
    greedy, areas = [], []
    for toks in golden_lines("dispatch.txt"):
        kind, rest = toks[0], " ".join(toks[1:])
        lhs, rhs = rest.split(" -> ")
        if kind == "greedy":
            a, cp = lhs.split(" cp ")
            b, l = rhs.replace("buckets ", "").split(" loads ")
            greedy.append(([int(x) for x in a.split(",")], int(cp), [int(x) for x in b.split(",")],
                           [int(x) for x in l.split(",")]))
        else:
            sl_txt, _, sq, _, sk, _, chunk = lhs.split(" ")
            sl = [tuple(int(x) for x in t.split(",")) for t in sl_txt.split(";")]
            areas.append((sl, int(sq), int(sk), int(chunk), [int(x) for x in rhs.replace("areas ", "").split(",")]))
    return greedy, areas


def test_dispatch_golden():
    greedy, areas = dispatch_fixtures()
    assert len(greedy) >= 5 and len(areas) >= 8
    for a, cp, buckets, loads in greedy:
        b, l = O.dispatch_greedy(a, cp)
        assert b.tolist() == buckets and l.tolist() == loads, (a, cp)
    for sl, sq, sk, chunk, want in areas:
        assert O.chunk_areas(sl, sq, chunk).tolist() == want, sl


def test_chunk_areas_match_dense_mask():
    for seed in range(10):
        rng = np.random.default_rng(700 + seed)
        chunk = int(rng.integers(1, 9))
        sq = chunk * int(rng.integers(1, 12))
        sk = int(rng.integers(1, 90))
        sl = W.random_slices(seed + 800, sq, sk, max_segments=4, max_pieces=4)
        got = O.chunk_areas(sl, sq, chunk)
        dense = O.dense_mask(sl, sq, sk).sum(axis=1).reshape(-1, chunk).sum(axis=1)
        assert got.tolist() == dense.tolist()
        assert got.sum() == O.mask_area(sl, sq, sk)


def test_dispatch_greedy_invariants_and_optimum():
    import itertools
    rng = np.random.default_rng(9)
    for _ in range(30):
        cp = int(rng.integers(1, 4))
        n = cp * int(rng.integers(1, 4))
        areas = rng.integers(0, 50, n).tolist()
        b, loads = O.dispatch_greedy(areas, cp)
        assert np.bincount(b, minlength=cp).tolist() == [n // cp] * cp
        assert [sum(a for a, x in zip(areas, b) if x == j) for j in range(cp)] == loads.tolist()
        # exhaustive optimum over equal-size partitions: the greedy is never below it
        best = min(max(sum(a for a, x in zip(areas, asg) if x == j) for j in range(cp))
                   for asg in itertools.product(range(cp), repeat=n)
                   if all(asg.count(j) == n // cp for j in range(cp)))
        assert loads.max() >= best


def test_range_gather_and_scatter_reduce():
    src = np.arange(10 * 3).reshape(10, 3)
    # hand-worked: rows 7..8, then 0..1, then 4
    g = O.range_gather(src, [(7, 9), (0, 2), (4, 5)])
    assert g.tolist() == [[21, 22, 23], [24, 25, 26], [0, 1, 2], [3, 4, 5], [12, 13, 14]]
    assert O.range_gather(src, []).shape == (0, 3)
    # overlapping destination ranges add: row 1 gets two contributions
    buf = np.ones((4, 2))
    out = O.range_scatter_reduce(buf, [(0, 2), (1, 3)], np.zeros((5, 2)))
    assert out.tolist() == [[1, 1], [2, 2], [1, 1], [0, 0], [0, 0]]
    # gather then scatter over ranges that tile the rows once gives the rows back
    rng = np.random.default_rng(4)
    x = rng.standard_normal((50, 4))
    cuts = [0, 7, 8, 30, 50]
    rs = [(cuts[i], cuts[i + 1]) for i in rng.permutation(4)]
    np.testing.assert_array_equal(O.range_scatter_reduce(O.range_gather(x, rs), rs, np.zeros_like(x)), x)
    # every destination row receives the sum of the buffer rows whose range covers it
    rs = [(3, 9), (0, 5), (4, 6)]
    buf = rng.standard_normal((6 + 5 + 2, 4))
    got = O.range_scatter_reduce(buf, rs, np.zeros((10, 4)))
    want = np.zeros((10, 4))
    pos = 0
    for s_, e_ in rs:
        for r in range(s_, e_):
            want[r] += buf[pos + r - s_]
        pos += e_ - s_
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


def test_forward_sampled_rows_equal_full_rows():
    S = 200
    t = tensors(S, 4, 2, 8, 9)
    sl = W.sink_window_slices(2, 100, 10, 24)
    out, lse = O.attention_forward(t["q"], t["k"], t["v"], sl, 0.3)
    rows = [0, 5, 9, 10, 33, 99, 100, 150, 199]
    o2, l2 = O.attention_forward(t["q"], t["k"], t["v"], sl, 0.3, rows=rows)
    np.testing.assert_array_equal(o2, out[rows])
    np.testing.assert_array_equal(l2, lse[:, rows])


# ----------------------------------------------------------------------------
# backward
# ----------------------------------------------------------------------------

def loss_fn(q, k, v, dout, sl, sc):
    out, _ = O.attention_forward(q, k, v, sl, sc)
    return float(np.sum(out * dout))


@pytest.mark.parametrize("mtype", [O.FULL, O.CAUSAL, O.INV_CAUSAL, O.BI_CAUSAL])
def test_backward_matches_finite_differences(mtype):
    rng = np.random.default_rng(mtype)
    sq, sk, hq, hkv, d = 7, 9, 2, 1, 4
    q, k, v = rng.standard_normal((sq, hq, d)), rng.standard_normal((sk, hkv, d)), rng.standard_normal((sk, hkv, d))
    dout = rng.standard_normal((sq, hq, d))
    # rows 0..5 under the slice under test, row 6 is empty
    sl = [(0, 6, 1, 9, mtype)]
    sc, eps = 0.7, 1e-6
    dq, dk, dv = O.attention_backward(q, k, v, dout, sl, sc)
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            fp = loss_fn(args["q"], args["k"], args["v"], dout, sl, sc)
            args[name] = xm
            fm = loss_fn(args["q"], args["k"], args["v"], dout, sl, sc)
            num[idx] = (fp - fm) / (2 * eps)
        err = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-30)
        assert err < 1e-6, (name, err)
    assert np.all(dq[6] == 0)


def dense_sink_reference(q, k, v, slices, scale, sink):
    """The sink by its plain definition: each row's softmax over [allowed logits, sink_h], with the
    sink's value vector zero (dense mask, small sizes only)."""
    sq, hq, d = q.shape
    sk, hkv, _ = k.shape
    m = O.dense_mask(slices, sq, sk)
    out = np.zeros((sq, hq, d))
    lse = np.zeros((hq, sq))
    for h in range(hq):
        g = h // (hq // hkv)
        logits = np.concatenate([np.where(m, scale * q[:, h] @ k[:, g].T, -np.inf),
                                 np.full((sq, 1), sink[h])], axis=1)
        mx = logits.max(axis=1, keepdims=True)
        e = np.exp(logits - mx)
        den = e.sum(axis=1, keepdims=True)
        lse[h] = (mx + np.log(den))[:, 0]
        out[:, h] = (e[:, :-1] / den) @ np.concatenate([v[:, g]], axis=0)
    return out, lse


def test_sink_forward_equals_the_extra_logit_definition():
    rng = np.random.default_rng(8)
    sq, sk, hq, hkv, d = 9, 11, 4, 2, 5
    q, k, v = rng.standard_normal((sq, hq, d)), rng.standard_normal((sk, hkv, d)), rng.standard_normal((sk, hkv, d))
    sink = np.array([0.3, -2.0, 4.0, -50.0])
    sl = [(0, 6, 1, 9, O.CAUSAL), (6, 8, 0, 11, O.FULL)]       # row 8 has no key
    out, lse = O.attention_forward(q, k, v, sl, 0.7, sink=sink)
    r_out, r_lse = dense_sink_reference(q, k, v, sl, 0.7, sink)
    np.testing.assert_allclose(out, r_out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, r_lse, rtol=0, atol=1e-13)
    assert np.all(out[8] == 0) and np.allclose(lse[:, 8], sink)   # an empty row: out 0, lse = sink
    # a sink at -inf changes nothing; the sink equals an LSE merge with the part (0, sink)
    o0, l0 = O.attention_forward(q, k, v, sl, 0.7)
    o1, l1 = O.attention_forward(q, k, v, sl, 0.7, sink=np.full(hq, -np.inf))
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)
    om, lm = O.lse_merge([(o0, l0), (np.zeros_like(o0), np.repeat(sink[:, None], sq, axis=1))])
    np.testing.assert_allclose(om, out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lm, lse, rtol=0, atol=1e-13)


def test_sink_backward_matches_finite_differences():
    rng = np.random.default_rng(9)
    sq, sk, hq, hkv, d = 6, 7, 2, 1, 3
    q, k, v = rng.standard_normal((sq, hq, d)), rng.standard_normal((sk, hkv, d)), rng.standard_normal((sk, hkv, d))
    dout = rng.standard_normal((sq, hq, d))
    sink = np.array([0.5, -1.0])
    sl = [(0, 5, 0, 7, O.BI_CAUSAL), (0, 5, 0, 2, O.FULL)]        # row 5 has no key
    sc, eps = 0.8, 1e-6

    def loss(q_, k_, v_, s_):
        return float(np.sum(O.attention_forward(q_, k_, v_, sl, sc, sink=s_)[0] * dout))

    dq, dk, dv = O.attention_backward(q, k, v, dout, sl, sc, sink=sink)
    ds = O.sink_gradient(q, k, v, dout, sl, sc, sink)
    for name, g in (("q", dq), ("k", dk), ("v", dv), ("sink", ds)):
        args = {"q": q, "k": k, "v": v, "sink": sink}
        x = args[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            a = dict(args)
            a[name] = xp
            fp = loss(a["q"], a["k"], a["v"], a["sink"])
            a[name] = xm
            fm = loss(a["q"], a["k"], a["v"], a["sink"])
            num[idx] = (fp - fm) / (2 * eps)
        err = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-30)
        assert err < 1e-6, (name, err)


def test_sink_backward_matches_torch_autograd():
    torch.manual_seed(3)
    sq, hq, hkv, d = 24, 4, 2, 8
    sl = W.random_slices(4, sq, sq, max_segments=3, max_pieces=3)
    q = torch.randn(sq, hq, d, dtype=torch.float64, requires_grad=True)
    k = torch.randn(sq, hkv, d, dtype=torch.float64, requires_grad=True)
    v = torch.randn(sq, hkv, d, dtype=torch.float64, requires_grad=True)
    sink = torch.randn(hq, dtype=torch.float64, requires_grad=True)
    dout = torch.randn(sq, hq, d, dtype=torch.float64)
    m = torch.from_numpy(O.dense_mask(sl, sq, sq))
    g = hq // hkv
    logits = torch.einsum("qhd,khd->hqk", q, k.repeat_interleave(g, dim=1)) * 0.5
    logits = torch.where(m[None], logits, torch.tensor(-float("inf"), dtype=torch.float64))
    full = torch.cat([logits, sink[:, None, None].expand(hq, sq, 1)], dim=2)
    p = torch.softmax(full, dim=2)[:, :, :-1]
    out = torch.einsum("hqk,khd->qhd", p, v.repeat_interleave(g, dim=1))
    (out * dout).sum().backward()
    args = [x.detach().numpy() for x in (q, k, v)]
    dq, dk, dv = O.attention_backward(*args, dout.numpy(), sl, 0.5, sink=sink.detach().numpy())
    ds = O.sink_gradient(*args, dout.numpy(), sl, 0.5, sink.detach().numpy())
    for a, b in ((dq, q.grad), (dk, k.grad), (dv, v.grad), (ds, sink.grad)):
        np.testing.assert_allclose(a, b.numpy(), rtol=0, atol=1e-10)


def test_backward_matches_torch_autograd_gqa():
    S, hq, hkv, d = 60, 4, 2, 8
    t = tensors(S, hq, hkv, d, 11)
    sl = W.random_slices(5, S, S)
    sc = 0.25
    m = torch.from_numpy(O.dense_mask(sl, S, S))
    q = torch.from_numpy(O.to_f64(t["q"])).requires_grad_()
    k = torch.from_numpy(O.to_f64(t["k"])).requires_grad_()
    v = torch.from_numpy(O.to_f64(t["v"])).requires_grad_()
    dout = torch.from_numpy(O.to_f64(t["dout"]))
    kr = k.repeat_interleave(hq // hkv, 1)
    vr = v.repeat_interleave(hq // hkv, 1)
    s = sc * torch.einsum("ihd,jhd->hij", q, kr)
    s = torch.where(m[None], s, torch.tensor(-math.inf, dtype=torch.float64))
    live = m.any(dim=1)
    p = torch.softmax(torch.where(live[None, :, None], s, torch.zeros_like(s)), dim=-1)
    p = torch.where(live[None, :, None] & m[None], p, torch.zeros_like(p))
    out = torch.einsum("hij,jhd->ihd", p, vr)
    (out * dout).sum().backward()
    dq, dk, dv = O.attention_backward(t["q"], t["k"], t["v"], t["dout"], sl, sc)
    for a, b in ((dq, q.grad), (dk, k.grad), (dv, v.grad)):
        np.testing.assert_allclose(a, b.numpy(), atol=1e-11, rtol=0)


def test_backward_sampled_equals_full():
    S = 150
    t = tensors(S, 4, 2, 8, 13)
    sl = W.varlen_slices([40, 70, 40])
    dq, dk, dv = O.attention_backward(t["q"], t["k"], t["v"], t["dout"], sl, 0.3)
    rows, keys = [0, 39, 40, 77, 149], [3, 41, 109, 110, 149]
    dq2, dk2, dv2 = O.attention_backward(t["q"], t["k"], t["v"], t["dout"], sl, 0.3, rows=rows, keys=keys)
    np.testing.assert_allclose(dq2, dq[rows], atol=1e-13, rtol=0)
    np.testing.assert_allclose(dk2, dk[keys], atol=1e-13, rtol=0)
    np.testing.assert_allclose(dv2, dv[keys], atol=1e-13, rtol=0)


# ----------------------------------------------------------------------------
# block classes, CSR, LPT order
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("direction", ["q2k", "k2q"])
def test_interval_classifier_equals_brute_force(direction):
    for seed in range(40):
        sq, sk = 50 + 7 * seed, 260 - 3 * seed
        bm, bn = [(16, 16), (8, 32), (32, 8), (16, 64), (64, 16)][seed % 5]
        sl = W.random_slices(seed + 200, sq, sk, max_segments=5, max_pieces=5)
        cls = O.classify_blocks_dense(sl, sq, sk, bm, bn, direction)
        want = O.csr_from_classes(cls, direction)
        got = O.block_csr_from_intervals(sl, sq, sk, bm, bn, direction)
        for a, b in zip(want, got):
            np.testing.assert_array_equal(a, b)


def test_square_causal_block_counts_closed_form():
    # L = m t, tile t: the diagonal blocks are Partial, the m(m-1)/2 below it Full.
    for m, t in ((1, 16), (5, 16), (8, 8), (3, 32)):
        L = m * t
        for direction in ("q2k", "k2q"):
            fo, fi, mo, mi = O.block_csr_from_intervals([(0, L, 0, L, O.CAUSAL)], L, L, t, t, direction)
            assert fo[-1] == (m * m - m) // 2 and mo[-1] == m
            np.testing.assert_array_equal(mi, np.arange(m))


def test_q_only_out_of_bounds_rule():
    # S = 20, tiles of 16: the second q-tile has 12 out-of-bounds rows.
    sl = [(0, 20, 0, 16, O.FULL)]
    fo, fi, mo, mi = O.block_csr_from_intervals(sl, 20, 32, 16, 16, "q2k")
    assert fo.tolist() == [0, 1, 2] and fi.tolist() == [0, 0] and mo[-1] == 0
    fo, fi, mo, mi = O.block_csr_from_intervals(sl, 20, 32, 16, 16, "k2q")
    assert fo.tolist() == [0, 1, 1] and fi.tolist() == [0]
    assert mo.tolist() == [0, 1, 1] and mi.tolist() == [1]
    # columns out of bounds are never Full, in either order
    fo, fi, mo, mi = O.block_csr_from_intervals([(0, 16, 0, 20, O.FULL)], 16, 20, 16, 16, "q2k")
    assert fi.tolist() == [0] and mi.tolist() == [1]


def test_lpt_order():
    full_off = np.array([0, 2, 2, 5, 6])     # tiles: 2F, 0F, 3F, 1F
    mask_off = np.array([0, 1, 2, 2, 3])     # tiles: 1P, 1P, 0P, 1P
    # costs with (4, 5): 13, 5, 12, 9
    assert O.lpt_order(full_off, mask_off, 4, 5).tolist() == [0, 2, 3, 1]
    assert O.lpt_order([0, 1, 2], [0, 0, 0], 1, 1).tolist() == [0, 1]
