"""Shared helpers for the GPU parity tests (no method arithmetic)."""
import numpy as np

GEMM_TOL = 2e-3      # max relative error of the W4A16 GEMM against the oracle
U32 = 2.0 ** -24     # unit roundoff of fp32


def gemm_rel_err(C, R):
    """max |C - R| / max(|R|, rms(R)): the GEMM error metric (relative error
    with an rms floor, so that near-zero outputs do not dominate)."""
    C = np.asarray(C, np.float64)
    R = np.asarray(R, np.float64)
    rms = float(np.sqrt(np.mean(R * R))) if R.size else 1.0
    den = np.maximum(np.abs(R), rms if rms > 0 else 1.0)
    return float(np.max(np.abs(C - R) / den)) if R.size else 0.0


def logit_bound(X, W, s):
    """Forward-error bound of an fp32 dot product of length K scaled in fp32:
    |L32 - L| <= s * gamma_K * sum_k |x_k w_k| + |L| * u   (Higham, recursive
    summation; any summation order).  Returns [M][V] in double."""
    K = X.shape[1]
    gamma = K * U32 / (1 - K * U32)
    absdot = np.abs(X.astype(np.float64)) @ np.abs(W.astype(np.float64)).T
    sc = s.astype(np.float64)[None, :]
    return sc * absdot * (gamma + 2 * U32) + 1e-30


def to_dev(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
