"""ctypes binding of the C ABI declared in ``include/ffa.h``.

Argument marshalling only: every step of the attention path runs in the CUDA
kernels of ``libffa_gb300.so``.  PyTorch provides device memory and streams.
There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np

from .build import LIB_PATH

FFA_OK = 0
STATUS_NAMES = {0: "FFA_OK", 1: "FFA_ERR_INVALID_ARG", 2: "FFA_ERR_INVALID_SLICE",
                3: "FFA_ERR_OVERLAPPING_COVERAGE", 4: "FFA_ERR_UNSUPPORTED", 5: "FFA_ERR_OVERFLOW",
                6: "FFA_ERR_CUDA", 7: "FFA_ERR_DEVICE_CHECK"}

MASK_FULL, MASK_CAUSAL, MASK_INV_CAUSAL, MASK_BI_CAUSAL = 0, 1, 2, 3


class FFAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({_status_string(code)})")


class AttnSliceC(ctypes.Structure):
    _fields_ = [("q_start", ctypes.c_int64), ("q_end", ctypes.c_int64), ("k_start", ctypes.c_int64),
                ("k_end", ctypes.c_int64), ("mask_type", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class TileCfgC(ctypes.Structure):
    _fields_ = [("fwd_bm", ctypes.c_int32), ("fwd_bn", ctypes.c_int32), ("bwd_bm", ctypes.c_int32),
                ("bwd_bn", ctypes.c_int32)]


class PlanInfoC(ctypes.Structure):
    _fields_ = [("seqlen_q", ctypes.c_int64), ("seqlen_k", ctypes.c_int64), ("tiles", TileCfgC),
                ("m_tiles", ctypes.c_int32), ("n_tiles", ctypes.c_int32),
                ("bwd_m_tiles", ctypes.c_int32), ("bwd_n_tiles", ctypes.c_int32),
                ("n_slices", ctypes.c_int64), ("mask_area", ctypes.c_int64), ("q2k_full", ctypes.c_int64),
                ("q2k_mask", ctypes.c_int64), ("k2q_full", ctypes.c_int64), ("k2q_mask", ctypes.c_int64),
                ("row_intervals", ctypes.c_int64), ("key_intervals", ctypes.c_int64),
                ("bwd_items", ctypes.c_int64), ("plan_bytes", ctypes.c_int64),
                ("bwd_chunk_tiles", ctypes.c_int32), ("plan_launches", ctypes.c_int32)]


_lib = None
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_p32 = ctypes.POINTER(ctypes.c_int32)


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load ``libffa_gb300.so`` (built by ``__graft_entry__.build()``) and declare its signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise FFAError(6, f"library {path} not built (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    lib.ffa_status_string.restype = ctypes.c_char_p
    lib.ffa_status_string.argtypes = [ctypes.c_int]
    lib.ffa_plan_create.restype = ctypes.c_int
    lib.ffa_plan_create.argtypes = [ctypes.POINTER(AttnSliceC), _i64, _i64, _i64, ctypes.POINTER(TileCfgC), _vp,
                                    ctypes.POINTER(_vp)]
    lib.ffa_plan_destroy.restype = ctypes.c_int
    lib.ffa_plan_destroy.argtypes = [_vp]
    lib.ffa_plan_info.restype = ctypes.c_int
    lib.ffa_plan_info.argtypes = [_vp, ctypes.POINTER(PlanInfoC)]
    lib.ffa_plan_copy_csr.restype = ctypes.c_int
    lib.ffa_plan_copy_csr.argtypes = [_vp, _i32, _p32, _p32, _p32, _p32, _p32]
    lib.ffa_plan_copy_bwd_items.restype = ctypes.c_int
    lib.ffa_plan_copy_bwd_items.argtypes = [_vp, _p32]
    lib.ffa_plan_copy_row_intervals.restype = ctypes.c_int
    lib.ffa_plan_copy_row_intervals.argtypes = [_vp, _p32, _p32]
    lib.ffa_plan_check_status.restype = ctypes.c_int
    lib.ffa_plan_check_status.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.ffa_fwd.restype = ctypes.c_int
    lib.ffa_fwd.argtypes = [_vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp, ctypes.c_float, _vp, _vp, _vp]
    lib.ffa_fwd_accumulate.restype = ctypes.c_int
    lib.ffa_fwd_accumulate.argtypes = [_vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp, ctypes.c_float, _vp, _vp,
                                       _vp]
    lib.ffa_fwd_sink.restype = ctypes.c_int
    lib.ffa_fwd_sink.argtypes = [_vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp, ctypes.c_float, _vp, _vp, _vp,
                                 _vp]
    lib.ffa_bwd_sink.restype = ctypes.c_int
    lib.ffa_bwd_sink.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp, ctypes.c_float,
                                 _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.ffa_dispatch_solve.restype = ctypes.c_int
    lib.ffa_dispatch_solve.argtypes = [ctypes.POINTER(AttnSliceC), _i64, _i64, _i64, _i64, _i32, _vp, _vp, _vp]
    lib.ffa_range_gather.restype = ctypes.c_int
    lib.ffa_range_gather.argtypes = [_vp, _i64, _i64, _vp, _i64, _vp, _vp]
    lib.ffa_range_scatter_reduce.restype = ctypes.c_int
    lib.ffa_range_scatter_reduce.argtypes = [_vp, _vp, _i64, _i64, _i32, _vp, _i64, _vp]
    lib.ffa_lse_combine.restype = ctypes.c_int
    lib.ffa_lse_combine.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _vp]
    lib.ffa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.ffa_bwd_workspace_size.argtypes = [_i64, _i64, _i32, _i32, _i32]
    lib.ffa_bwd.restype = ctypes.c_int
    lib.ffa_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp, ctypes.c_float,
                            _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.ffa_bwd_noalloc.restype = ctypes.c_int
    lib.ffa_bwd_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp,
                                    ctypes.c_float, _vp, _vp, _vp, _vp]
    lib.ffa_selftest_bounded_wait.restype = ctypes.c_int
    lib.ffa_selftest_bounded_wait.argtypes = [_vp, ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32)]
    lib.ffa_plan_enable_cta_trace.restype = ctypes.c_int
    lib.ffa_plan_enable_cta_trace.argtypes = [_vp, _i32]
    lib.ffa_plan_read_cta_trace.restype = ctypes.c_int
    lib.ffa_plan_read_cta_trace.argtypes = [_vp, _i32, _vp, ctypes.POINTER(ctypes.c_uint64), _i32,
                                            ctypes.POINTER(ctypes.c_int32)]
    lib.ffa_plan_enable_timing.restype = ctypes.c_int
    lib.ffa_plan_enable_timing.argtypes = [_vp, _i32]
    lib.ffa_plan_read_timing.restype = ctypes.c_int
    lib.ffa_plan_read_timing.argtypes = [_vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]
    if path == LIB_PATH:
        _lib = lib
    return lib


def selftest_bounded_wait(stream=None) -> Tuple[int, int]:
    """Run the kernels' bounded wait on barriers nothing arrives at (about 2 s); returns
    (the status word it recorded, the number of threads that gave up)."""
    st, n = ctypes.c_uint32(0), ctypes.c_uint32(0)
    _check(load_library().ffa_selftest_bounded_wait(_stream_handle(stream), ctypes.byref(st), ctypes.byref(n)),
           "ffa_selftest_bounded_wait")
    return st.value, n.value


def _status_string(code: int) -> str:
    try:
        return load_library().ffa_status_string(code).decode()
    except Exception:  # the library itself may be what is missing
        return STATUS_NAMES.get(code, "unknown")


def _check(code: int, where: str) -> None:
    if code != FFA_OK:
        raise FFAError(code, where)


def _slices_array(slices: Sequence) -> Tuple[ctypes.Array, int]:
    tup = [s.as_tuple() if hasattr(s, "as_tuple") else tuple(s) for s in slices]
    arr = (AttnSliceC * max(1, len(tup)))()
    for i, (qs, qe, ks, ke, t) in enumerate(tup):
        arr[i] = AttnSliceC(int(qs), int(qe), int(ks), int(ke), int(t), 0)
    return arr, len(tup)


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_p32)


class Plan:
    """Owns an ``ffa_plan_t``: the mask's per-row intervals, CSR block lists and tile orders."""

    def __init__(self, slices: Sequence, seqlen_q: int, seqlen_k: int, block_m: int = 128, block_n: int = 128,
                 stream=None, bwd_block_m: Optional[int] = None, bwd_block_n: Optional[int] = None):
        """Tiles: block_m x block_n (query rows x key columns) for the forward (q2k) lists, and
        bwd_block_m x bwd_block_n for the backward (k2q) lists (default: the forward's)."""
        lib = load_library()
        arr, n = _slices_array(slices)
        handle = _vp()
        bbm = block_m if bwd_block_m is None else bwd_block_m
        bbn = block_n if bwd_block_n is None else bwd_block_n
        tiles = TileCfgC(int(block_m), int(block_n), int(bbm), int(bbn))
        _check(lib.ffa_plan_create(arr, n, int(seqlen_q), int(seqlen_k), ctypes.byref(tiles),
                                   _stream_handle(stream), ctypes.byref(handle)), "ffa_plan_create")
        self._h = handle
        self.seqlen_q, self.seqlen_k = int(seqlen_q), int(seqlen_k)
        self.block_m, self.block_n = int(block_m), int(block_n)
        self.bwd_block_m, self.bwd_block_n = int(bbm), int(bbn)

    @property
    def handle(self):
        if self._h is None:
            raise FFAError(1, "plan already destroyed")
        return self._h

    def info(self) -> dict:
        inf = PlanInfoC()
        _check(load_library().ffa_plan_info(self.handle, ctypes.byref(inf)), "ffa_plan_info")
        d = {name: getattr(inf, name) for name, _ in PlanInfoC._fields_ if name != "tiles"}
        d.update({name: getattr(inf.tiles, name) for name, _ in TileCfgC._fields_})
        return d

    def csr(self, direction: str):
        """(full_off, full_idx, mask_off, mask_idx, order) as int32 numpy arrays."""
        inf = self.info()
        d = {"q2k": 0, "k2q": 1}[direction]
        rows = inf["m_tiles"] if d == 0 else inf["bwd_n_tiles"]
        nf = inf["q2k_full"] if d == 0 else inf["k2q_full"]
        nm = inf["q2k_mask"] if d == 0 else inf["k2q_mask"]
        fo, mo = np.zeros(rows + 1, np.int32), np.zeros(rows + 1, np.int32)
        fi, mi = np.zeros(max(nf, 1), np.int32), np.zeros(max(nm, 1), np.int32)
        order = np.zeros(max(rows, 1), np.int32)
        _check(load_library().ffa_plan_copy_csr(self.handle, d, _ptr(fo), _ptr(fi), _ptr(mo), _ptr(mi),
                                                _ptr(order)), "ffa_plan_copy_csr")
        return fo, fi[:nf], mo, mi[:nm], order[:rows]

    def bwd_items(self):
        """Backward work items as an int32 array [n, 4]: (k-tile, first Full index,
        first Partial index, #Full | #Partial << 16), in the order ffa_bwd runs them."""
        n = self.info()["bwd_items"]
        items = np.zeros((max(n, 1), 4), np.int32)
        _check(load_library().ffa_plan_copy_bwd_items(self.handle, _ptr(items)), "ffa_plan_copy_bwd_items")
        return items[:n]

    def row_intervals(self):
        """(off [seqlen_q + 1], iv [n, 2]) int32 arrays of the query rows' key intervals."""
        n = self.info()["row_intervals"]
        off = np.zeros(self.seqlen_q + 1, np.int32)
        iv = np.zeros((max(n, 1), 2), np.int32)
        _check(load_library().ffa_plan_copy_row_intervals(self.handle, _ptr(off), _ptr(iv)),
               "ffa_plan_copy_row_intervals")
        return off, iv[:n]

    def check_status(self, stream=None) -> int:
        """Synchronize the stream and return (and clear) the device status word; raise if non-zero."""
        w = ctypes.c_uint32(0)
        code = load_library().ffa_plan_check_status(self.handle, _stream_handle(stream), ctypes.byref(w))
        if code not in (FFA_OK, 7):
            _check(code, "ffa_plan_check_status")
        if w.value:
            raise FFAError(7, f"device status word 0x{w.value:x}")
        return w.value

    KERNELS = ("fwd", "bwd_pre", "bwd_main", "bwd_dq")

    def enable_timing(self, enable: bool = True) -> None:
        _check(load_library().ffa_plan_enable_timing(self.handle, int(bool(enable))), "ffa_plan_enable_timing")

    def read_timing(self) -> dict:
        """{kernel: (total device ms, launches)} over the launches recorded so far."""
        ms = (ctypes.c_double * 4)()
        n = (ctypes.c_int64 * 4)()
        _check(load_library().ffa_plan_read_timing(self.handle, ms, n), "ffa_plan_read_timing")
        return {k: (ms[i], n[i]) for i, k in enumerate(self.KERNELS)}

    def enable_cta_trace(self, enable: bool = True) -> None:
        _check(load_library().ffa_plan_enable_cta_trace(self.handle, int(bool(enable))), "ffa_plan_enable_cta_trace")

    def read_cta_trace(self, kernel: str, stream=None) -> np.ndarray:
        """Per-CTA [start ns, end ns, units, blocks] of the latest traced launch of ``kernel``
        ("fwd" or "bwd_main"), as a uint64 array [n_ctas, 4]."""
        kid = {"fwd": 0, "bwd_main": 2}[kernel]
        cap = 4096
        buf = (ctypes.c_uint64 * (4 * cap))()
        n = ctypes.c_int32(0)
        _check(load_library().ffa_plan_read_cta_trace(self.handle, kid, _stream_handle(stream), buf, cap,
                                                      ctypes.byref(n)), "ffa_plan_read_cta_trace")
        return np.frombuffer(buf, dtype=np.uint64, count=4 * n.value).reshape(n.value, 4).copy()

    def destroy(self) -> None:
        if self._h is not None:
            load_library().ffa_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def _need(t, dtype, name, shape=None):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise FFAError(1, f"{name} must be a contiguous CUDA {dtype} tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise FFAError(1, f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def fwd(q, k, v, plan: Plan, scale: float, out=None, lse=None, stream=None):
    """out [Sq, Hq, d] bf16 and lse [Hq, Sq] fp32 of attention over the plan's mask."""
    import torch
    sq, hq, d = q.shape
    sk, hkv, _ = k.shape
    _need(q, torch.bfloat16, "q")
    _need(k, torch.bfloat16, "k")
    _need(v, torch.bfloat16, "v", k.shape)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((hq, sq), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(out, torch.bfloat16, "out", q.shape)
    _need(lse, torch.float32, "lse", (hq, sq))
    _check(load_library().ffa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), sq, sk, hq, hkv, d, plan.handle,
                                  float(scale), out.data_ptr(), lse.data_ptr(), _stream_handle(stream)), "ffa_fwd")
    return out, lse


def fwd_accumulate(q, k, v, plan: Plan, scale: float, out, lse, stream=None):
    """Merge attention over the plan's mask into the partial result (out, lse), in place, by LSE."""
    import torch
    sq, hq, d = q.shape
    sk, hkv, _ = k.shape
    _need(q, torch.bfloat16, "q")
    _need(k, torch.bfloat16, "k")
    _need(v, torch.bfloat16, "v", k.shape)
    _need(out, torch.bfloat16, "out", q.shape)
    _need(lse, torch.float32, "lse", (hq, sq))
    _check(load_library().ffa_fwd_accumulate(q.data_ptr(), k.data_ptr(), v.data_ptr(), sq, sk, hq, hkv, d,
                                             plan.handle, float(scale), out.data_ptr(), lse.data_ptr(),
                                             _stream_handle(stream)), "ffa_fwd_accumulate")
    return out, lse


def fwd_sink(q, k, v, plan: Plan, scale: float, sink, out=None, lse=None, stream=None):
    """out, lse of attention over the plan's mask whose every row's softmax also holds the
    per-head sink logit sink [Hq] (fp32, CUDA) with a zero value vector."""
    import torch
    sq, hq, d = q.shape
    sk, hkv, _ = k.shape
    _need(q, torch.bfloat16, "q")
    _need(k, torch.bfloat16, "k")
    _need(v, torch.bfloat16, "v", k.shape)
    _need(sink, torch.float32, "sink", (hq,))
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((hq, sq), dtype=torch.float32, device=q.device) if lse is None else lse
    _need(out, torch.bfloat16, "out", q.shape)
    _need(lse, torch.float32, "lse", (hq, sq))
    _check(load_library().ffa_fwd_sink(q.data_ptr(), k.data_ptr(), v.data_ptr(), sq, sk, hq, hkv, d, plan.handle,
                                       float(scale), sink.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                       _stream_handle(stream)), "ffa_fwd_sink")
    return out, lse


def bwd_sink(q, k, v, out, lse, dout, plan: Plan, scale: float, sink, stream=None):
    """dq, dk, dv (bf16) and dsink [Hq] (fp32) for the output of fwd_sink."""
    import torch
    sq, hq, d = q.shape
    sk, hkv, _ = k.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse", (hq, sq))
    _need(sink, torch.float32, "sink", (hq,))
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dsink = torch.empty_like(sink)
    ws_bytes = bwd_workspace_size(sq, sk, hq, hkv, d)
    workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    _check(load_library().ffa_bwd_sink(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                       dout.data_ptr(), sq, sk, hq, hkv, d, plan.handle, float(scale),
                                       sink.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                       dsink.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                       _stream_handle(stream)), "ffa_bwd_sink")
    return dq, dk, dv, dsink


def dispatch_solve(slices, seqlen_q: int, seqlen_k: int, chunk_size: int, cp_size: int):
    """The dispatch solver (host only): (bucket of each query chunk int32 [n], Area of each chunk
    int64 [n], area of each bucket int64 [cp_size]) for n = seqlen_q // chunk_size chunks."""
    arr, n_slices = _slices_array(slices)
    n = int(seqlen_q) // int(chunk_size) if chunk_size > 0 else 0
    bucket = np.zeros(max(n, 1), np.int32)
    carea = np.zeros(max(n, 1), np.int64)
    barea = np.zeros(max(int(cp_size), 1), np.int64)
    _check(load_library().ffa_dispatch_solve(arr, n_slices, int(seqlen_q), int(seqlen_k), int(chunk_size),
                                             int(cp_size), carea.ctypes.data_as(_vp), bucket.ctypes.data_as(_vp),
                                             barea.ctypes.data_as(_vp)), "ffa_dispatch_solve")
    return bucket[:n], carea[:n], barea[:int(cp_size)]


def _ranges_array(ranges):
    arr = np.asarray(list(ranges), dtype=np.int64).reshape(-1, 2)
    return np.ascontiguousarray(arr), arr.shape[0]


def range_gather(src, ranges, out=None, stream=None):
    """The rows of src (token-major CUDA tensor) in the (start, end) ranges, back to back."""
    import torch
    if not isinstance(src, torch.Tensor) or not src.is_cuda or not src.is_contiguous():
        raise FFAError(1, "src must be a contiguous CUDA tensor")
    arr, n = _ranges_array(ranges)
    total = int(sum(max(0, int(e) - int(s)) for s, e in arr)) if n else 0
    out = torch.empty((total,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device) if out is None else out
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] else src.element_size()
    _check(load_library().ffa_range_gather(src.data_ptr(), src.shape[0], row_bytes, arr.ctypes.data_as(_vp), n,
                                           out.data_ptr(), _stream_handle(stream)), "ffa_range_gather")
    return out


def range_scatter_reduce(src, ranges, dst, stream=None):
    """dst[start:end] += the rows of src, back to back in range order (fp32 or bf16), in place."""
    import torch
    for t, n in ((src, "src"), (dst, "dst")):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise FFAError(1, f"{n} must be a contiguous CUDA tensor")
    if src.dtype != dst.dtype or dst.dtype not in (torch.float32, torch.bfloat16):
        raise FFAError(1, "src and dst must both be float32 or both bfloat16")
    arr, n = _ranges_array(ranges)
    row_elems = dst[0].numel() if dst.shape[0] else 1
    _check(load_library().ffa_range_scatter_reduce(src.data_ptr(), arr.ctypes.data_as(_vp), n, row_elems,
                                                   0 if dst.dtype == torch.float32 else 1, dst.data_ptr(),
                                                   dst.shape[0], _stream_handle(stream)), "ffa_range_scatter_reduce")
    return dst


def lse_combine(out_a, lse_a, out_b, lse_b, out=None, lse=None, stream=None):
    """LSE merge of two partial results (out [S, H, d] bf16, lse [H, S] fp32); out / lse may be
    out_a / lse_a or out_b / lse_b."""
    import torch
    s, h, d = out_a.shape
    _need(out_a, torch.bfloat16, "out_a")
    _need(out_b, torch.bfloat16, "out_b", out_a.shape)
    _need(lse_a, torch.float32, "lse_a", (h, s))
    _need(lse_b, torch.float32, "lse_b", (h, s))
    out = torch.empty_like(out_a) if out is None else out
    lse = torch.empty_like(lse_a) if lse is None else lse
    _need(out, torch.bfloat16, "out", out_a.shape)
    _need(lse, torch.float32, "lse", (h, s))
    _check(load_library().ffa_lse_combine(out_a.data_ptr(), lse_a.data_ptr(), out_b.data_ptr(), lse_b.data_ptr(),
                                          out.data_ptr(), lse.data_ptr(), s, h, d, _stream_handle(stream)),
           "ffa_lse_combine")
    return out, lse


def bwd_workspace_size(seqlen_q: int, seqlen_k: int, hq: int, hkv: int, d: int) -> int:
    return int(load_library().ffa_bwd_workspace_size(int(seqlen_q), int(seqlen_k), int(hq), int(hkv), int(d)))


def bwd(q, k, v, out, lse, dout, plan: Plan, scale: float, dq=None, dk=None, dv=None, workspace=None,
        stream=None):
    """dq, dk, dv (bf16) of sum(out * dout) for the forward above."""
    import torch
    sq, hq, d = q.shape
    sk, hkv, _ = k.shape
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse", (hq, sq))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = bwd_workspace_size(sq, sk, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    _check(load_library().ffa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                  dout.data_ptr(), sq, sk, hq, hkv, d, plan.handle, float(scale), dq.data_ptr(),
                                  dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                  _stream_handle(stream)), "ffa_bwd")
    return dq, dk, dv
