"""Helpers shared by the GPU parity tests: run the CUDA path, compare with the oracle.

Tolerances (bf16 inputs, fp32 accumulation):
  out  max-abs <= 1e-2 and mean-abs <= 1e-3
  lse  abs <= 1e-3 on finite rows; -inf must match exactly
  dq / dk / dv  relative Frobenius error <= 1e-2
  block metadata: bit-exact
"""
import numpy as np

OUT_MAX_ABS = 1e-2
OUT_MEAN_ABS = 1e-3
LSE_ABS = 1e-3
GRAD_REL_FRO = 1e-2


def check_out_lse(out_gpu: np.ndarray, lse_gpu: np.ndarray, out_ref: np.ndarray, lse_ref: np.ndarray, what=""):
    err = np.abs(out_gpu.astype(np.float64) - out_ref)
    assert err.max(initial=0.0) <= OUT_MAX_ABS, f"{what} out max-abs {err.max()}"
    assert (err.mean() if err.size else 0.0) <= OUT_MEAN_ABS, f"{what} out mean-abs {err.mean()}"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), np.isneginf(lse_ref)), f"{what} -inf rows differ"
    assert not np.isnan(lse_gpu).any(), f"{what} NaN in lse"
    if fin.any():
        e = np.abs(lse_gpu[fin].astype(np.float64) - lse_ref[fin]).max()
        assert e <= LSE_ABS, f"{what} lse abs {e}"


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    a = a.astype(np.float64)
    nb = np.linalg.norm(b)
    if nb == 0:
        return float(np.linalg.norm(a))
    return float(np.linalg.norm(a - b) / nb)


def check_grad(g: np.ndarray, r: np.ndarray, what=""):
    e = rel_fro(g, r)
    assert e <= GRAD_REL_FRO, f"{what} relative Frobenius error {e}"
    assert not np.isnan(g).any(), f"{what} has NaN"


def to_np(t) -> np.ndarray:
    return t.detach().float().cpu().numpy()
