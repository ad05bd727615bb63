"""Seeded synthetic inputs for the Flex-Flash-Attention (FFA) hot path.

This module is shared by the CUDA path's tests and bench and by the CPU
oracle.  It only *describes inputs*: document lengths, the AttnSlice lists
built from them, and random q/k/v/dout tensors.  It holds none of the
method's arithmetic (no mask predicates, no areas, no attention).

An AttnSlice is ``(QRange, KRange, MaskType)`` with half-open, contiguous
ranges (MagiAttention blog, section "Flex-Flash-Attention and AttnSlice").
The four mask types are named there: FULL, CAUSAL, INV-CAUSAL, BI-CAUSAL.

Workloads follow the benchmark settings on the same page ("Training and
Benchmark settings": batch 1, self-attention with seqlen_q = seqlen_k,
bf16, head dim 128, GQA head ratios) and its varlen recipe (documents
packed back to back, each at most a quarter of the total length).  The real
length distribution of the pages is not available; seeded uniform and
log-uniform draws stand in for it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Callable, Dict, List, Optional, Sequence, Tuple

import torch

MASK_FULL = 0
MASK_CAUSAL = 1
MASK_INV_CAUSAL = 2
MASK_BI_CAUSAL = 3
MASK_NAMES = {MASK_FULL: "FULL", MASK_CAUSAL: "CAUSAL",
              MASK_INV_CAUSAL: "INV_CAUSAL", MASK_BI_CAUSAL: "BI_CAUSAL"}


@dataclass(frozen=True)
class AttnSlice:
    """One AttnSlice: rows [q_start, q_end) x keys [k_start, k_end), mask_type."""
    q_start: int
    q_end: int
    k_start: int
    k_end: int
    mask_type: int

    def as_tuple(self) -> Tuple[int, int, int, int, int]:
        return (self.q_start, self.q_end, self.k_start, self.k_end, self.mask_type)


# ----------------------------------------------------------------------------
# document lengths
# ----------------------------------------------------------------------------

def doc_lengths(total: int, lo: int, hi: int, dist: str, seed: int) -> List[int]:
    """Draw document lengths until ``total`` tokens are filled (last one truncated).

    ``dist`` is ``"uniform"`` (integers uniform in [lo, hi]) or
    ``"loguniform"`` (floor(exp(U(ln lo, ln hi))), clamped to [lo, hi]).
    Draws come from a CPU ``torch.Generator`` seeded with ``seed``.
    """
    g = torch.Generator().manual_seed(seed)
    out: List[int] = []
    remaining = total
    while remaining > 0:
        if dist == "uniform":
            length = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        elif dist == "loguniform":
            u = float(torch.rand(1, generator=g, dtype=torch.float64).item())
            length = int(math.floor(math.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))))
            length = max(lo, min(hi, length))
        else:
            raise ValueError(f"unknown length distribution {dist!r}")
        length = min(length, remaining)
        out.append(length)
        remaining -= length
    return out


# ----------------------------------------------------------------------------
# slice-list builders for the workloads
# ----------------------------------------------------------------------------

def varlen_slices(lengths: Sequence[int], mask_type: int = MASK_CAUSAL) -> List[AttnSlice]:
    """One slice per packed document, q range == k range == the document."""
    out, start = [], 0
    for length in lengths:
        out.append(AttnSlice(start, start + length, start, start + length, mask_type))
        start += length
    return out


def tiny_mixed_slices() -> List[AttnSlice]:
    """512 tokens, one slice of each mask type (the tiny mixed-mask case)."""
    return [AttnSlice(0, 128, 0, 128, MASK_CAUSAL),
            AttnSlice(128, 256, 0, 256, MASK_FULL),
            AttnSlice(256, 384, 256, 384, MASK_INV_CAUSAL),
            AttnSlice(384, 512, 256, 512, MASK_BI_CAUSAL)]


def video_block_causal_slices(n_docs: int, doc_len: int, block: int) -> List[AttnSlice]:
    """Per document, frame block i attends FULL to [doc start, end of block i)."""
    out = []
    for d in range(n_docs):
        ds = d * doc_len
        for i in range(doc_len // block):
            out.append(AttnSlice(ds + i * block, ds + (i + 1) * block, ds, ds + (i + 1) * block,
                                 MASK_FULL))
    return out


def sink_window_slices(n_docs: int, doc_len: int, sink: int, window: int) -> List[AttnSlice]:
    """Per document: every query sees the first ``sink`` keys (FULL), and keys at or
    after ``ds + sink`` through a causal window of ``window`` keys.

    The window is one CAUSAL slice over the first ``window`` rows after the sink
    and one BI-CAUSAL slice for the rest, whose key range starts one key later so
    that each query q sees keys [q - window + 1, q].  The q-ranges overlap the
    sink slice's, the key ranges do not.
    """
    out = []
    for d in range(n_docs):
        ds, de = d * doc_len, (d + 1) * doc_len
        out.append(AttnSlice(ds, de, ds, ds + sink, MASK_FULL))
        out.append(AttnSlice(ds + sink, ds + sink + window, ds + sink, ds + sink + window,
                             MASK_CAUSAL))
        out.append(AttnSlice(ds + sink + window, de, ds + sink + 1, de, MASK_BI_CAUSAL))
    return out


def random_slices(seed: int, seqlen_q: int, seqlen_k: int, max_segments: int = 4,
                  max_pieces: int = 4, allow_empty: bool = True) -> List[AttnSlice]:
    """Random slice list whose (q, k) coverage is disjoint by construction.

    The q axis is cut into segments; inside a segment the k axis is cut into
    disjoint pieces, and each chosen piece gets its own random sub-range of the
    segment's rows and a random mask type.  Slices of one segment share no key,
    slices of different segments share no query, so no pair (q, k) is covered
    twice, while q-ranges inside a segment overlap freely.
    """
    g = torch.Generator().manual_seed(seed)

    def rint(lo: int, hi: int) -> int:  # inclusive
        return int(torch.randint(lo, hi + 1, (1,), generator=g).item())

    def cuts(n: int, parts: int) -> List[int]:
        pts = sorted({rint(0, n) for _ in range(parts - 1)})
        return [0] + pts + [n]

    out: List[AttnSlice] = []
    qcuts = cuts(seqlen_q, rint(1, max_segments))
    for a, b in zip(qcuts[:-1], qcuts[1:]):
        if b <= a:
            continue
        kcuts = cuts(seqlen_k, rint(1, max_pieces))
        for ks, ke in zip(kcuts[:-1], kcuts[1:]):
            if ke <= ks or rint(0, 3) == 0:
                continue
            qs = rint(a, b - 1)
            qe = rint(qs + 1, b)
            if not allow_empty and qe <= qs:
                continue
            out.append(AttnSlice(qs, qe, ks, ke, rint(0, 3)))
    return out


# ----------------------------------------------------------------------------
# named workloads
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    seqlen: int
    hq: int
    hkv: int
    d: int
    seed: int
    slices: Tuple[AttnSlice, ...]
    backward: bool
    description: str

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


def _w(name, seqlen, hq, hkv, d, seed, slices, backward, description) -> Workload:
    return Workload(name, seqlen, hq, hkv, d, seed, tuple(slices), backward, description)


WORKLOAD_BUILDERS: Dict[str, Callable[[], Workload]] = {
    "tiny_mixed": lambda: _w(
        "tiny_mixed", 512, 2, 2, 64, 0, tiny_mixed_slices(), False,
        "S=512, Hq=Hkv=2, d=64: one slice of each mask type"),
    "varlen_causal_64k": lambda: _w(
        "varlen_causal_64k", 65536, 16, 16, 128, 1,
        varlen_slices(doc_lengths(65536, 1024, 16384, "uniform", 1)), True,
        "S=64K varlen causal, docs U[1024,16384], Hq=Hkv=16, d=128"),
    "video_block_causal_128k": lambda: _w(
        "video_block_causal_128k", 131072, 64, 8, 128, 2,
        video_block_causal_slices(4, 32768, 4096), True,
        "S=128K, 4 docs x 8 FULL frame blocks of 4096, Hq=64, Hkv=8, d=128"),
    "sink_window_256k": lambda: _w(
        "sink_window_256k", 262144, 32, 32, 128, 3,
        sink_window_slices(8, 32768, 1024, 4096), True,
        "S=256K, 8 docs x (1024-key sink + 4096-key window), Hq=Hkv=32, d=128"),
    "varlen_causal_1m": lambda: _w(
        "varlen_causal_1m", 1048576, 16, 4, 128, 4,
        varlen_slices(doc_lengths(1048576, 2048, 262144, "loguniform", 4)), True,
        "S=1M varlen causal, docs log-U[2048,262144], Hq=16, Hkv=4, d=128"),
    # profiling case: the 1M workload's shape family at 128K tokens, small enough
    # for ncu captures (a few GB on the device) while its tensors exceed L2
    "varlen_causal_128k": lambda: _w(
        "varlen_causal_128k", 131072, 16, 4, 128, 4,
        varlen_slices(doc_lengths(131072, 2048, 32768, "loguniform", 4)), True,
        "S=128K varlen causal, docs log-U[2048,32768], Hq=16, Hkv=4, d=128 (profiling size)"),
}

WORKLOAD_ORDER = ["tiny_mixed", "varlen_causal_64k", "video_block_causal_128k",
                  "sink_window_256k", "varlen_causal_1m"]


def workload(name: str) -> Workload:
    return WORKLOAD_BUILDERS[name]()


# ----------------------------------------------------------------------------
# tensors
# ----------------------------------------------------------------------------

def make_tensors(seqlen: int, hq: int, hkv: int, d: int, seed: int,
                 device: str = "cpu", with_dout: bool = True,
                 dtype: torch.dtype = torch.bfloat16) -> Dict[str, torch.Tensor]:
    """q [S,Hq,d], k/v [S,Hkv,d] (and dout [S,Hq,d]) ~ N(0,1) rounded to ``dtype``.

    Drawn in the order q, k, v, dout from a ``torch.Generator`` on ``device``
    seeded with ``seed`` (fp32 ``randn`` then a round-to-nearest-even cast).
    """
    g = torch.Generator(device=device).manual_seed(seed)

    def draw(shape):
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)

    out = {"q": draw((seqlen, hq, d)), "k": draw((seqlen, hkv, d)), "v": draw((seqlen, hkv, d))}
    if with_dout:
        out["dout"] = draw((seqlen, hq, d))
    return out


def sample_rows(seqlen: int, n: int, seed: int, slices: Optional[Sequence[AttnSlice]] = None,
                edge: int = 0) -> List[int]:
    """Sorted distinct row indices: ``n`` uniform draws plus, when ``slices`` is
    given, the first and last ``edge`` rows of every slice's q-range."""
    g = torch.Generator().manual_seed(seed)
    rows = set(torch.randint(0, seqlen, (n,), generator=g).tolist()) if n > 0 else set()
    if slices is not None and edge > 0:
        for s in slices:
            rows.update(range(s.q_start, min(s.q_end, s.q_start + edge)))
            rows.update(range(max(s.q_start, s.q_end - edge), s.q_end))
    return sorted(r for r in rows if 0 <= r < seqlen)


def make_partials(seqlen: int, hq: int, d: int, seed: int, empty_frac: float = 0.2, lse_scale: float = 4.0,
                  device: str = "cpu") -> Dict[str, torch.Tensor]:
    """A random partial attention result: out [S,Hq,d] ~ N(0,1) rounded to bf16 and
    lse [Hq,S] ~ lse_scale * N(0,1) in fp32, with a fraction ``empty_frac`` of the
    (head, row) entries set to -inf (rows with no keys in this part)."""
    g = torch.Generator(device=device).manual_seed(seed)
    out = torch.randn((seqlen, hq, d), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    lse = torch.randn((hq, seqlen), generator=g, device=device, dtype=torch.float32) * lse_scale
    empty = torch.rand((hq, seqlen), generator=g, device=device) < empty_frac
    lse = torch.where(empty, torch.full_like(lse, -math.inf), lse)
    return {"out": out, "lse": lse}
