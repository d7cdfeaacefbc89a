"""Shared test helpers: error metric against the oracle and sampling."""
from __future__ import annotations

import numpy as np
import torch

# fp32 and bf16: the stated bars.  fp16 (no bar stated): psi and the output
# are each rounded to fp16 (<= 2^-11 of sum|terms| each) and the fused paths
# round X or dX once more, so <= 1.5e-3 of sum|terms|; 4e-3 leaves a margin.
TOL = {torch.float32: 1e-5, torch.bfloat16: 1e-2, torch.float16: 4e-3}


def rel_err(gpu: np.ndarray, ref: np.ndarray, S: np.ndarray) -> float:
    """max |gpu - oracle| / sum|terms|; where S == 0 the result must be exactly 0."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    S = np.asarray(S, np.float64)
    zero = S == 0
    if np.any(gpu[zero] != 0):
        return float("inf")
    d = np.abs(gpu - ref)[~zero] / S[~zero]
    return float(d.max()) if d.size else 0.0


def to_np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def ulp_diff_f32(a: np.ndarray, b: np.ndarray) -> int:
    """max distance in fp32 units in the last place (same-sign values)."""
    a = np.ascontiguousarray(a, np.float32).view(np.int32).astype(np.int64)
    b = np.ascontiguousarray(b, np.float32).view(np.int32).astype(np.int64)
    # map to a monotone integer line
    a = np.where(a < 0, -(a & 0x7FFFFFFF), a)
    b = np.where(b < 0, -(b & 0x7FFFFFFF), b)
    return int(np.abs(a - b).max()) if a.size else 0
