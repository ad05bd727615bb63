"""ctypes binding of ``ffa_rows.c``: the oracle's row-by-row fp64 attention in C.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``.  It computes the same
definitions as ``ffa_oracle.attention_forward`` / ``attention_backward``
(MagiAttention blog, "Flex-Flash-Attention and AttnSlice": the AttnSlice mask
types, the union mask, softmax attention and its analytic gradients) for
listed rows or keys, visiting only each row's allowed keys, with OpenMP over
rows.  That makes sampled checks of 1M-token problems over every head
affordable.  The tests pin it against torch's fp64 SDPA and autograd and
against ``ffa_oracle``.

The C source is compiled with the host C compiler into
``oracle/libffa_oracle_rows.so`` by :func:`build` (``__graft_entry__.build()``
calls it beside the CUDA library build).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
from typing import Optional, Sequence, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ffa_rows.c")
LIB = os.path.join(HERE, "libffa_oracle_rows.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``ffa_rows.c`` (gcc or cc, -O3, OpenMP) unless the library is newer."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler (gcc / cc) to build the row oracle")
    tmp = f"{LIB}.{os.getpid()}.tmp"
    cmd = [cc, "-O3", "-std=gnu11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, SRC, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the row oracle failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p
        for name in ("ffa_oracle_rows", "ffa_oracle_keys"):
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, i32, vp, i64, dbl, vp, i64, vp, vp, vp][
                : 17 if name == "ffa_oracle_rows" else 16]
        _lib = lib
    return _lib


def _bits(x) -> np.ndarray:
    """A bf16 torch tensor (any device) as a contiguous host uint16 array of its bit patterns."""
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError(f"the row oracle takes bf16 tensors, got {x.dtype}")
    return np.ascontiguousarray(x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16))


def _slices(slices) -> np.ndarray:
    from .ffa_oracle import slice_tuples
    st = slice_tuples(slices)
    return np.ascontiguousarray(np.array(st, dtype=np.int64).reshape(len(st), 5))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def attention_rows(q, k, v, slices, scale: float, rows: Sequence[int], dout=None
                   ) -> Tuple[np.ndarray, np.ndarray, Optional[np.ndarray]]:
    """(out [R, Hq, d], lse [Hq, R], dq [R, Hq, d] or None) for the sorted ``rows``.

    q [Sq, Hq, d], k / v [Sk, Hkv, d], dout like q: bf16 torch tensors.  dq is
    computed when ``dout`` is given."""
    sq, hq, d = q.shape
    sk, hkv, _ = k.shape
    rows = np.ascontiguousarray(np.asarray(sorted(rows), dtype=np.int64))
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    db = _bits(dout) if dout is not None else None
    sl = _slices(slices)
    out = np.zeros((rows.size, hq, d))
    lse = np.zeros((hq, rows.size))
    dq = np.zeros((rows.size, hq, d)) if dout is not None else None
    rc = _load().ffa_oracle_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(db), sq, sk, hq, hkv, d, _ptr(sl), sl.shape[0],
                                 float(scale), _ptr(rows), rows.size, _ptr(out), _ptr(lse), _ptr(dq))
    if rc != 0:
        raise RuntimeError(f"ffa_oracle_rows failed ({'bad arguments' if rc == 1 else 'out of memory'})")
    return out, lse, dq


def attention_keys(q, k, v, dout, slices, scale: float, keys: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    """(dk [K, Hkv, d], dv [K, Hkv, d]) for the sorted, distinct ``keys``."""
    sq, hq, d = q.shape
    sk, hkv, _ = k.shape
    keys = np.ascontiguousarray(np.asarray(sorted(set(int(x) for x in keys)), dtype=np.int64))
    qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
    sl = _slices(slices)
    dk = np.zeros((keys.size, hkv, d))
    dv = np.zeros((keys.size, hkv, d))
    rc = _load().ffa_oracle_keys(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(db), sq, sk, hq, hkv, d, _ptr(sl), sl.shape[0],
                                 float(scale), _ptr(keys), keys.size, _ptr(dk), _ptr(dv))
    if rc != 0:
        raise RuntimeError(f"ffa_oracle_keys failed ({'bad arguments' if rc == 1 else 'out of memory'})")
    return dk, dv
