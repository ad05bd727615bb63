"""fp64 CPU oracle for Flex-Flash-Attention over AttnSlice masks.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the library.

Sources (MagiAttention pages):
  * blog "MagiAttention: ultra-long-context distributed attention", section
    "Flex-Flash-Attention and AttnSlice": AttnSlice = (QRange, KRange,
    MaskType), mask types FULL / CAUSAL / INV-CAUSAL / BI-CAUSAL, the global
    mask as the union of slices, partial results of slices merged by
    reduction (Figure 5 caption), backward required for training;
  * same blog, "Training and Benchmark settings": FLOPs(fwd) = 2*2*MaskArea
    *batch*Hq*d, FLOPs(bwd) = 2.5*FLOPs(fwd), full area = seqlen^2, causal
    area = seqlen*(seqlen+1)/2;
  * MagiAttention documentation, "FFA_FA4 backend" items 1-2: blocks are
    Full / Partial / Empty, in q2k (forward) and k2q (backward) order; the
    forward treats blocks out of bounds only along q as Full; only non-empty
    blocks are stored, in CSR form (full_block_offset / mask_block_offset).

Readings where the pages are silent (each one is listed with its reason in
the design notes of the repository):
  * slice-local coordinates r = i - q_start, c = j - k_start, Lq, Lk the range
    lengths; CAUSAL is bottom-right aligned (c <= r + Lk - Lq), INV-CAUSAL
    top-left aligned (c >= r), BI-CAUSAL is both;
  * (q, k) coverage by the slices is disjoint, so the union mask and the LSE
    merge of per-slice partials agree;
  * lse is the natural log of sum_j exp(scale * q.k_j); a row with no allowed
    key has out = 0 and lse = -inf and contributes no gradient;
  * GQA maps q head h to kv head h // (Hq / Hkv);
  * the backward (k2q) classification calls any block with out-of-bounds rows
    or columns Partial.

All arithmetic is float64 (bf16 inputs widen exactly); matrix products use
numpy's matmul as a library step.  No blocking or reordering beyond the
definitions: a row's softmax is taken over all of its allowed keys at once.
"""
from __future__ import annotations

from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

FULL, CAUSAL, INV_CAUSAL, BI_CAUSAL = 0, 1, 2, 3
EMPTY_BLOCK, PARTIAL_BLOCK, FULL_BLOCK = 0, 1, 2

__all__ = [
    "FULL", "CAUSAL", "INV_CAUSAL", "BI_CAUSAL", "EMPTY_BLOCK", "PARTIAL_BLOCK", "FULL_BLOCK",
    "slice_tuples", "slice_predicate", "coverage_block", "mask_block", "dense_mask",
    "coverage_is_disjoint", "mask_area", "mask_area_closed_form", "slices_area",
    "fwd_flops", "bwd_flops", "row_intervals", "attention_forward", "attention_backward", "sink_gradient",
    "lse_merge", "chunk_areas", "dispatch_greedy", "range_gather", "range_scatter_reduce", "classify_blocks_dense", "csr_from_classes", "block_counts_from_intervals",
    "block_csr_from_intervals", "lpt_order", "to_f64",
]


# ----------------------------------------------------------------------------
# AttnSlice masks
# ----------------------------------------------------------------------------

def slice_tuples(slices: Iterable) -> List[Tuple[int, int, int, int, int]]:
    """Accept AttnSlice objects or 5-tuples (q_start, q_end, k_start, k_end, type)."""
    out = []
    for s in slices:
        t = s.as_tuple() if hasattr(s, "as_tuple") else tuple(s)
        out.append(tuple(int(x) for x in t))
    return out


def slice_predicate(mask_type: int, r: np.ndarray, c: np.ndarray, lq: int, lk: int) -> np.ndarray:
    """Allowed-ness of slice-local (r, c) for one mask type (broadcasting).

    CAUSAL keeps c <= r + (Lk - Lq) (diagonal through the bottom-right corner);
    INV-CAUSAL keeps c >= r (diagonal through the top-left corner);
    BI-CAUSAL keeps both.
    """
    if mask_type == FULL:
        return np.ones(np.broadcast_shapes(np.shape(r), np.shape(c)), dtype=bool)
    if mask_type == CAUSAL:
        return c <= r + (lk - lq)
    if mask_type == INV_CAUSAL:
        return c >= r
    if mask_type == BI_CAUSAL:
        return (c >= r) & (c <= r + (lk - lq))
    raise ValueError(f"unknown mask type {mask_type}")


def coverage_block(slices, rows: np.ndarray, cols: np.ndarray) -> np.ndarray:
    """Number of slices allowing each (rows[x], cols[y]); rows and cols sorted."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    cov = np.zeros((rows.size, cols.size), dtype=np.int32)
    for qs, qe, ks, ke, t in slice_tuples(slices):
        r0, r1 = np.searchsorted(rows, [qs, qe])
        c0, c1 = np.searchsorted(cols, [ks, ke])
        if r1 <= r0 or c1 <= c0:
            continue
        r = (rows[r0:r1] - qs)[:, None]
        c = (cols[c0:c1] - ks)[None, :]
        cov[r0:r1, c0:c1] += slice_predicate(t, r, c, qe - qs, ke - ks)
    return cov


def mask_block(slices, rows: np.ndarray, cols: np.ndarray) -> np.ndarray:
    """Union mask M[i][j] restricted to the given sorted rows and columns."""
    return coverage_block(slices, rows, cols) > 0


def dense_mask(slices, seqlen_q: int, seqlen_k: int) -> np.ndarray:
    """The whole union mask as a [seqlen_q, seqlen_k] boolean array."""
    return mask_block(slices, np.arange(seqlen_q), np.arange(seqlen_k))


def coverage_is_disjoint(slices, seqlen_q: int, seqlen_k: int) -> bool:
    """True when no (q, k) pair is allowed by two slices (brute force)."""
    return int(coverage_block(slices, np.arange(seqlen_q), np.arange(seqlen_k)).max(initial=0)) <= 1


def mask_area(slices, seqlen_q: int, seqlen_k: int) -> int:
    """Brute-force count of allowed pairs of the union mask."""
    return int(dense_mask(slices, seqlen_q, seqlen_k).sum())


def mask_area_closed_form(lq: int, lk: int, mask_type: int) -> int:
    """Allowed pairs of one slice, summed row by row in closed form.

    FULL: Lq*Lk.  CAUSAL: Lq*(Lk-Lq) + Lq*(Lq+1)/2 if Lq <= Lk else Lk*(Lk+1)/2.
    INV-CAUSAL: Lq*Lk - Lq*(Lq-1)/2 if Lq <= Lk else Lk*(Lk+1)/2.
    BI-CAUSAL: Lq*(Lk-Lq+1) if Lk >= Lq else 0.  Square CAUSAL gives the
    pages' n(n+1)/2 and FULL their n^2.
    """
    lq, lk = max(lq, 0), max(lk, 0)
    if lq == 0 or lk == 0:
        return 0
    if mask_type == FULL:
        return lq * lk
    if mask_type == CAUSAL:
        return lq * (lk - lq) + lq * (lq + 1) // 2 if lq <= lk else lk * (lk + 1) // 2
    if mask_type == INV_CAUSAL:
        return lq * lk - lq * (lq - 1) // 2 if lq <= lk else lk * (lk + 1) // 2
    if mask_type == BI_CAUSAL:
        return lq * (lk - lq + 1) if lk >= lq else 0
    raise ValueError(f"unknown mask type {mask_type}")


def slices_area(slices) -> int:
    """Sum of per-slice closed-form areas (the union area when coverage is disjoint)."""
    return sum(mask_area_closed_form(qe - qs, ke - ks, t) for qs, qe, ks, ke, t in slice_tuples(slices))


def fwd_flops(area: int, hq: int, d: int, batch: int = 1) -> int:
    """FLOPs(fwd) = 2 * 2 * MaskArea * batch * Hq * d (benchmark settings)."""
    return 2 * 2 * area * batch * hq * d


def bwd_flops(area: int, hq: int, d: int, batch: int = 1) -> float:
    """FLOPs(bwd) = 2.5 * FLOPs(fwd)."""
    return 2.5 * fwd_flops(area, hq, d, batch)


def row_intervals(slices, seqlen_q: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Allowed key intervals of every row: arrays (row, lo, hi), sorted by (row, lo).

    Each slice predicate bounds c from below and/or above only, so the keys a
    slice allows in one of its rows form one interval [lo, hi):
    FULL [ks, ke); CAUSAL [ks, ks + r + Lk - Lq + 1); INV-CAUSAL [ks + r, ke);
    BI-CAUSAL [ks + r, ks + r + Lk - Lq + 1), each clipped to [ks, ke); rows
    whose interval is empty are dropped.
    """
    rs, los, his = [], [], []
    for qs, qe, ks, ke, t in slice_tuples(slices):
        qe = min(qe, seqlen_q)
        if qe <= qs or ke <= ks:
            continue
        r = np.arange(qe - qs, dtype=np.int64)
        lq, lk = qe - qs, ke - ks
        lo = np.full_like(r, ks) if t in (FULL, CAUSAL) else ks + r
        hi = np.full_like(r, ke) if t in (FULL, INV_CAUSAL) else ks + r + (lk - lq) + 1
        lo, hi = np.maximum(lo, ks), np.minimum(hi, ke)
        keep = lo < hi
        rs.append(r[keep] + qs), los.append(lo[keep]), his.append(hi[keep])
    if not rs:
        z = np.zeros(0, dtype=np.int64)
        return z, z.copy(), z.copy()
    row, lo, hi = np.concatenate(rs), np.concatenate(los), np.concatenate(his)
    order = np.lexsort((lo, row))
    return row[order], lo[order], hi[order]


# ----------------------------------------------------------------------------
# attention (forward / backward), full or on sampled rows / keys
# ----------------------------------------------------------------------------

def to_f64(x) -> np.ndarray:
    """torch tensor (any float dtype, any device) or array -> float64 numpy."""
    if hasattr(x, "detach"):
        import torch
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _take(x, rows) -> np.ndarray:
    """float64 copy of x[rows] (rows: a slice or an index array), converting only those rows."""
    if hasattr(x, "detach"):
        import torch
        if not isinstance(rows, slice):
            rows = torch.as_tensor(np.asarray(rows), dtype=torch.long, device=x.device)
        return x[rows].detach().to("cpu", torch.float64).numpy()
    return np.asarray(x[rows], dtype=np.float64)


def _row_groups(slices, rows: np.ndarray, seqlen_k: int, budget: int = 1 << 24):
    """Split sorted ``rows`` into runs sharing a key span, with the span.

    A row's span is [min k_start, max k_end) over the slices whose q-range holds
    it; consecutive rows with the same span start are grouped (bounded by
    ``budget`` elements of the rows x span block).
    """
    st = slice_tuples(slices)
    lo = np.full(rows.size, seqlen_k, dtype=np.int64)
    hi = np.zeros(rows.size, dtype=np.int64)
    for qs, qe, ks, ke, _ in st:
        inside = (rows >= qs) & (rows < qe)
        lo = np.where(inside, np.minimum(lo, ks), lo)
        hi = np.where(inside, np.maximum(hi, ke), hi)
    i = 0
    while i < rows.size:
        j = i + 1
        span_hi = hi[i]
        while j < rows.size and lo[j] == lo[i]:
            new_hi = max(span_hi, hi[j])
            if (j + 1 - i) * max(new_hi - lo[i], 1) > budget:
                break
            span_hi = new_hi
            j += 1
        yield rows[i:j], int(lo[i]), int(max(span_hi, lo[i]))
        i = j


def attention_forward(q, k, v, slices, scale: float, rows: Optional[Sequence[int]] = None, sink=None):
    """Softmax attention over the union mask, in fp64.

    q [Sq, Hq, d], k/v [Sk, Hkv, d].  Returns ``out`` [R, Hq, d] and
    ``lse`` [Hq, R] for the rows ``rows`` (all rows when None), where
    s_ij = scale * <q_i, k_j> over allowed j, lse_i = ln sum_j exp(s_ij)
    and out_i = sum_j exp(s_ij - lse_i) v_j; a row with no allowed key gets
    out 0 and lse -inf.

    ``sink`` (optional, [Hq]): the attention sink, one more logit sink_h in
    every row's softmax with a zero value vector (MagiAttention pages name a
    learnable attention sink; this reading is the plain one).  Then
    lse_i = ln(sum_j exp(s_ij) + exp(sink_h)) and out_i = sum_j exp(s_ij -
    lse_i) v_j, i.e. the sink-free result scaled by exp(lse_i' - lse_i).
    """
    sq, hq, d = q.shape
    sk, hkv, dv_ = v.shape
    group = hq // hkv
    rows = np.arange(sq, dtype=np.int64) if rows is None else np.asarray(sorted(rows), dtype=np.int64)
    out = np.zeros((rows.size, hq, dv_))
    lse = np.full((hq, rows.size), -np.inf)
    pos = 0
    for grp, k0, k1 in _row_groups(slices, rows, sk):
        sl = slice(pos, pos + grp.size)
        pos += grp.size
        if k1 <= k0:
            continue
        qg, kg, vg = _take(q, grp), _take(k, slice(k0, k1)), _take(v, slice(k0, k1))
        cols = np.arange(k0, k1, dtype=np.int64)
        m = mask_block(slices, grp, cols)
        empty = ~m.any(axis=1)
        for h in range(hq):
            g = h // group
            s = scale * (qg[:, h, :] @ kg[:, g, :].T)
            s = np.where(m, s, -np.inf)
            mx = np.where(empty, 0.0, s.max(axis=1, initial=-np.inf))
            e = np.where(m, np.exp(s - mx[:, None]), 0.0)
            den = e.sum(axis=1)
            lse[h, sl] = np.where(empty, -np.inf, mx + np.log(np.where(empty, 1.0, den)))
            p = e / np.where(empty, 1.0, den)[:, None]
            out[sl, h, :] = p @ vg[:, g, :]
    if sink is not None:
        sk_ = np.asarray(sink, dtype=np.float64).reshape(hq, 1)
        lse_s = np.logaddexp(lse, sk_)
        w = np.where(np.isfinite(lse), np.exp(lse - np.where(np.isfinite(lse_s), lse_s, 0.0)), 0.0)   # [Hq, R]
        out = out * w.T[:, :, None]
        lse = lse_s
    return out, lse


def _rows_attending(slices, keys: np.ndarray, seqlen_q: int) -> np.ndarray:
    """Sorted rows that are allowed at least one of ``keys``."""
    st = slice_tuples(slices)
    cand = set()
    for qs, qe, ks, ke, _ in st:
        if np.any((keys >= ks) & (keys < ke)):
            cand.update(range(qs, min(qe, seqlen_q)))
    if not cand:
        return np.zeros(0, dtype=np.int64)
    cand = np.array(sorted(cand), dtype=np.int64)
    keep = np.zeros(cand.size, dtype=bool)
    step = max(1, (1 << 24) // max(keys.size, 1))
    for i in range(0, cand.size, step):
        keep[i:i + step] = mask_block(slices, cand[i:i + step], keys).any(axis=1)
    return cand[keep]


def attention_backward(q, k, v, dout, slices, scale: float,
                       rows: Optional[Sequence[int]] = None,
                       keys: Optional[Sequence[int]] = None, sink=None):
    """Analytic gradients of the fp64 attention above (with the sink when
    ``sink`` is given: P and D below then use the sink-inclusive lse and out).

    With P_ij = exp(s_ij - lse_i) (0 off the mask), D_i = <dO_i, O_i>:
    dV_j = sum_{h in group} sum_i P_ij dO_i;  dP_ij = <dO_i, v_j>;
    dS_ij = P_ij (dP_ij - D_i);  dQ_i = scale sum_j dS_ij k_j;
    dK_j = scale sum_{h in group} sum_i dS_ij q_i.

    Returns (dq [R, Hq, d] for ``rows``, dk [K, Hkv, d], dv [K, Hkv, d] for
    ``keys``); None selects all rows / all keys.
    """
    sq, hq, d = q.shape
    sk, hkv, dv_ = v.shape
    group = hq // hkv
    rows = np.arange(sq, dtype=np.int64) if rows is None else np.asarray(sorted(rows), dtype=np.int64)
    keys = np.arange(sk, dtype=np.int64) if keys is None else np.asarray(sorted(keys), dtype=np.int64)

    # dq on the requested rows
    dq = np.zeros((rows.size, hq, d))
    out_r, lse_r = attention_forward(q, k, v, slices, scale, rows, sink=sink)
    pos = 0
    for grp, k0, k1 in _row_groups(slices, rows, sk):
        sl = slice(pos, pos + grp.size)
        pos += grp.size
        if k1 <= k0:
            continue
        qg, dog = _take(q, grp), _take(dout, grp)
        kg, vg = _take(k, slice(k0, k1)), _take(v, slice(k0, k1))
        m = mask_block(slices, grp, np.arange(k0, k1, dtype=np.int64))
        for h in range(hq):
            g = h // group
            lse_h = lse_r[h, sl]
            finite = np.isfinite(lse_h)
            s = scale * (qg[:, h, :] @ kg[:, g, :].T)
            p = np.where(m & finite[:, None], np.exp(s - np.where(finite, lse_h, 0.0)[:, None]), 0.0)
            dp = dog[:, h, :] @ vg[:, g, :].T
            dd = np.sum(dog[:, h, :] * out_r[sl, h, :], axis=1)
            ds = p * (dp - dd[:, None])
            dq[sl, h, :] = scale * (ds @ kg[:, g, :])

    # dk / dv on the requested keys
    dk = np.zeros((keys.size, hkv, d))
    dv = np.zeros((keys.size, hkv, dv_))
    qrows = _rows_attending(slices, keys, sq)
    if qrows.size:
        out_q, lse_q = attention_forward(q, k, v, slices, scale, qrows, sink=sink)
        kk, vk = _take(k, keys), _take(v, keys)
        step = max(1, (1 << 24) // max(keys.size, 1))
        for i in range(0, qrows.size, step):
            grp = qrows[i:i + step]
            qg, dog = _take(q, grp), _take(dout, grp)
            m = mask_block(slices, grp, keys)
            for h in range(hq):
                g = h // group
                lse_h = lse_q[h, i:i + step]
                finite = np.isfinite(lse_h)
                s = scale * (qg[:, h, :] @ kk[:, g, :].T)
                p = np.where(m & finite[:, None], np.exp(s - np.where(finite, lse_h, 0.0)[:, None]), 0.0)
                dp = dog[:, h, :] @ vk[:, g, :].T
                dd = np.sum(dog[:, h, :] * out_q[i:i + step, h, :], axis=1)
                ds = p * (dp - dd[:, None])
                dv[:, g, :] += p.T @ dog[:, h, :]
                dk[:, g, :] += scale * (ds.T @ qg[:, h, :])
    return dq, dk, dv


def sink_gradient(q, k, v, dout, slices, scale: float, sink):
    """d(sum out * dout) / d sink_h = -sum_i exp(sink_h - lse_i) <dO_i, O_i>,
    with the sink-inclusive (out, lse): the sink's softmax weight times the
    row's D_i, as for any logit whose value vector is zero."""
    out, lse = attention_forward(q, k, v, slices, scale, sink=sink)
    dd = np.sum(to_f64(dout) * out, axis=2)                                     # [R, Hq]
    sk_ = np.asarray(sink, dtype=np.float64).reshape(-1, 1)
    p_sink = np.where(np.isfinite(lse), np.exp(sk_ - np.where(np.isfinite(lse), lse, 0.0)), 0.0)
    return -(p_sink * dd.T).sum(axis=1)


def lse_merge(parts):
    """Merge partial (out [R,H,d], lse [H,R]) results over disjoint key sets.

    lse = ln sum_s exp(lse_s); out = sum_s exp(lse_s - lse) out_s; a part
    whose lse is -inf for a row contributes nothing there (its out is not
    read); rows that are empty in every part stay (0, -inf).
    """
    lses = np.stack([p[1] for p in parts])            # [P, H, R]
    lse = np.logaddexp.reduce(lses, axis=0)
    finite = np.isfinite(lse)
    out = np.zeros_like(parts[0][0])
    for o, l in parts:
        w = np.where(finite & np.isfinite(l), np.exp(l - np.where(finite, lse, 0.0)), 0.0)  # [H, R]
        # a part empty for a row (lse = -inf) contributes nothing: its out is not read
        out += np.where(w.T[:, :, None] != 0.0, w.T[:, :, None] * np.where(np.isfinite(l).T[:, :, None], o, 0.0), 0.0)
    return out, lse


# ----------------------------------------------------------------------------
# Dispatch solver (MagiAttention blog, "Dispatch Solver", Figure 10)
# ----------------------------------------------------------------------------

def chunk_areas(slices, seqlen_q: int, chunk_size: int) -> np.ndarray:
    """Area(C_i) of every query chunk C_i = rows [i*chunk_size, (i+1)*chunk_size):
    the allowed (query, key) pairs of the union mask in the chunk's rows."""
    row, lo, hi = row_intervals(slices, seqlen_q)
    per_row = np.zeros(seqlen_q, dtype=np.int64)
    np.add.at(per_row, row, (hi - lo).astype(np.int64))
    return per_row.reshape(seqlen_q // chunk_size, chunk_size).sum(axis=1)


def dispatch_greedy(areas, cp_size: int) -> Tuple[np.ndarray, np.ndarray]:
    """The pages' min-heap greedy: chunks in order of area, heaviest first
    (ties: lower chunk index), each to the bucket with the least area so far
    among those holding fewer than n / cp_size chunks (ties: lower bucket
    index).  Returns (bucket of each chunk, area of each bucket)."""
    import heapq
    areas = [int(a) for a in areas]
    n = len(areas)
    assert n % cp_size == 0
    cap = n // cp_size
    order = sorted(range(n), key=lambda i: (-areas[i], i))
    heap = [(0, j) for j in range(cp_size)]
    heapq.heapify(heap)
    bucket = np.zeros(n, dtype=np.int64)
    load = [0] * cp_size
    count = [0] * cp_size
    for c in order:
        _, j = heapq.heappop(heap)
        bucket[c] = j
        load[j] += areas[c]
        count[j] += 1
        if count[j] < cap:
            heapq.heappush(heap, (load[j], j))
    return bucket, np.array(load, dtype=np.int64)


# ----------------------------------------------------------------------------
# Range-Gather / Range-Scatter-Reduce (MagiAttention blog, group-collective
# section: the pre / post kernels of the AlltoAll-v exchange)
# ----------------------------------------------------------------------------

def range_gather(src, ranges) -> np.ndarray:
    """The rows of ``src`` (token-major [S, ...]) in the ranges [s, e), back to
    back in list order."""
    src = np.asarray(src)
    parts = [src[s:e] for s, e in ranges]
    return np.concatenate(parts, axis=0) if parts else src[:0]


def range_scatter_reduce(src, ranges, dst) -> np.ndarray:
    """``dst`` plus the rows of ``src`` (back to back, in list order) added into
    the ranges [s, e) of ``dst``; overlapping ranges add all their rows.
    Returns a new array in float64."""
    out = np.array(dst, dtype=np.float64, copy=True)
    pos = 0
    for s, e in ranges:
        n = e - s
        out[s:e] += np.asarray(src[pos:pos + n], dtype=np.float64)
        pos += n
    return out


# ----------------------------------------------------------------------------
# Full / Partial / Empty blocks and their CSR lists
# ----------------------------------------------------------------------------

def _full_allowed(direction: str, a: int, b: int, bm: int, bn: int, sq: int, sk: int) -> bool:
    """Out-of-bounds rule: q2k may be Full with rows past seqlen_q (they are
    never stored) but not with columns past seqlen_k; k2q with neither."""
    k_oob = (b + 1) * bn > sk
    q_oob = (a + 1) * bm > sq
    if direction == "q2k":
        return not k_oob
    if direction == "k2q":
        return not (k_oob or q_oob)
    raise ValueError(direction)


def classify_blocks_dense(slices, seqlen_q: int, seqlen_k: int, bm: int, bn: int,
                          direction: str) -> np.ndarray:
    """Brute-force block classes [m_a, n_b] from the dense union mask."""
    m_a, n_b = -(-seqlen_q // bm), -(-seqlen_k // bn)
    mask = np.zeros((m_a * bm, n_b * bn), dtype=bool)
    mask[:seqlen_q, :seqlen_k] = dense_mask(slices, seqlen_q, seqlen_k)
    cnt = mask.reshape(m_a, bm, n_b, bn).sum(axis=(1, 3))
    out = np.zeros((m_a, n_b), dtype=np.int8)
    for a in range(m_a):
        nr = min(bm, seqlen_q - a * bm)
        for b in range(n_b):
            nc = min(bn, seqlen_k - b * bn)
            if cnt[a, b] == 0:
                out[a, b] = EMPTY_BLOCK
            elif cnt[a, b] == nr * nc and _full_allowed(direction, a, b, bm, bn, seqlen_q, seqlen_k):
                out[a, b] = FULL_BLOCK
            else:
                out[a, b] = PARTIAL_BLOCK
    return out


def csr_from_classes(classes: np.ndarray, direction: str):
    """CSR lists (full_off, full_idx, mask_off, mask_idx), ascending indices.

    q2k: one list per q-tile over k-tiles; k2q: one list per k-tile over q-tiles.
    """
    c = classes if direction == "q2k" else classes.T
    full_off, mask_off, full_idx, mask_idx = [0], [0], [], []
    for row in c:
        f = np.nonzero(row == FULL_BLOCK)[0]
        p = np.nonzero(row == PARTIAL_BLOCK)[0]
        full_idx.extend(f.tolist())
        mask_idx.extend(p.tolist())
        full_off.append(len(full_idx))
        mask_off.append(len(mask_idx))
    as32 = lambda x: np.asarray(x, dtype=np.int32)
    return as32(full_off), as32(full_idx), as32(mask_off), as32(mask_idx)


def block_counts_from_intervals(slices, seqlen_q: int, seqlen_k: int, bm: int, bn: int):
    """Allowed-element counts of every non-empty block, from row intervals.

    For the rows of q-tile a, F(x) = sum over their intervals of
    |[lo, hi) intersect [0, x)|; block (a, b) holds F((b+1)bn) - F(b bn)
    allowed elements.  Returns arrays (a, b, count) with count > 0, sorted by
    (a, b).  A different algorithm from the dense brute force.
    """
    row, lo, hi = row_intervals(slices, seqlen_q)
    m_a = -(-seqlen_q // bm)
    starts = np.searchsorted(row, np.arange(m_a + 1, dtype=np.int64) * bm)
    aa, bb, cc = [], [], []
    for a in range(m_a):
        i0, i1 = starts[a], starts[a + 1]
        if i1 <= i0:
            continue
        l, h = lo[i0:i1], hi[i0:i1]
        b0, b1 = int(l.min()) // bn, (int(h.max()) - 1) // bn
        x = np.minimum(np.arange(b0, b1 + 2, dtype=np.int64) * bn, seqlen_k)
        f = np.clip(x[None, :] - l[:, None], 0, (h - l)[:, None]).sum(axis=0)
        cnt = np.diff(f)
        nz = np.nonzero(cnt)[0]
        aa.append(np.full(nz.size, a, dtype=np.int64))
        bb.append(nz + b0)
        cc.append(cnt[nz])
    if not aa:
        z = np.zeros(0, dtype=np.int64)
        return z, z.copy(), z.copy()
    return np.concatenate(aa), np.concatenate(bb), np.concatenate(cc)


def block_csr_from_intervals(slices, seqlen_q: int, seqlen_k: int, bm: int, bn: int,
                             direction: str, counts=None):
    """CSR lists as in ``csr_from_classes``, without a dense mask or class grid."""
    a, b, cnt = counts if counts is not None else block_counts_from_intervals(
        slices, seqlen_q, seqlen_k, bm, bn)
    m_a, n_b = -(-seqlen_q // bm), -(-seqlen_k // bn)
    nr = np.minimum(bm, seqlen_q - a * bm)
    nc = np.minimum(bn, seqlen_k - b * bn)
    k_oob = (b + 1) * bn > seqlen_k
    q_oob = (a + 1) * bm > seqlen_q
    ok = ~k_oob if direction == "q2k" else ~(k_oob | q_oob)
    is_full = (cnt == nr * nc) & ok
    if direction == "q2k":
        major, minor, n_major = a, b, m_a
    else:
        order = np.lexsort((a, b))
        major, minor, is_full, n_major = b[order], a[order], is_full[order], n_b
    full_off = np.zeros(n_major + 1, dtype=np.int64)
    mask_off = np.zeros(n_major + 1, dtype=np.int64)
    np.add.at(full_off, major[is_full] + 1, 1)
    np.add.at(mask_off, major[~is_full] + 1, 1)
    return (np.cumsum(full_off).astype(np.int32), minor[is_full].astype(np.int32),
            np.cumsum(mask_off).astype(np.int32), minor[~is_full].astype(np.int32))


def lpt_order(full_off: np.ndarray, mask_off: np.ndarray, cost_full: int, cost_mask: int) -> np.ndarray:
    """Longest-processing-time-first order of the tiles of one CSR direction.

    Cost of tile t = cost_full * #Full(t) + cost_mask * #Partial(t); tiles are
    listed by decreasing cost, ties by increasing index.  Handing the next
    tile of this list to whichever worker frees up first is the greedy of the
    pages' dispatch solver (heaviest item to the least-loaded bucket).
    """
    nf = np.diff(np.asarray(full_off, dtype=np.int64))
    nm = np.diff(np.asarray(mask_off, dtype=np.int64))
    cost = cost_full * nf + cost_mask * nm
    return np.lexsort((np.arange(cost.size), -cost)).astype(np.int32)
