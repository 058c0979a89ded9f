"""Shared test helpers: the GEMM error metric and small conversions."""
import numpy as np

# GEMM tolerance: max over (m, n) of |y - ref| / max(|ref|, rms(ref[m, :])).
# FP32 accumulation of K/16 exact block terms has a relative rounding error of
# a few 1e-7 times sqrt(K/16) in practice; 1e-3 is the stated bound and still
# flags one dropped 16-block (about 4/sqrt(K) of the row rms, 6e-2 at K=4096).
GEMM_TOL = 1e-3


def gemm_error(y, ref):
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    rms = np.sqrt((ref ** 2).mean(axis=-1, keepdims=True))
    denom = np.maximum(np.abs(ref), rms)
    denom = np.where(denom > 0, denom, 1.0)
    return float(np.max(np.abs(y - ref) / denom))


def sampled_error(y_vals, ref_vals, row_rms):
    denom = np.maximum(np.abs(ref_vals), row_rms)
    denom = np.where(denom > 0, denom, 1.0)
    return float(np.max(np.abs(np.asarray(y_vals, np.float64) - ref_vals) / denom))


def plain_rel_error(y, ref):
    """max |y - ref| / |ref| over the outputs with |ref| >= the rms of their
    row: the plain relative error where it is well conditioned, reported
    beside gemm_error (which floors the denominator at the row rms)."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    rms = np.sqrt((ref ** 2).mean(axis=-1, keepdims=True))
    mask = (np.abs(ref) >= rms) & (np.abs(ref) > 0)
    if not mask.any():
        return 0.0
    return float(np.max(np.abs(y - ref)[mask] / np.abs(ref)[mask]))
