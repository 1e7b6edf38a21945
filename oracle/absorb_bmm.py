"""The absorb BMMs either side of the latent decode, written out in plain NumPy.

TEST INFRASTRUCTURE ONLY: nothing in the product path imports this package.

In the absorbed form of MLA the per-head key and value up-projections are moved
onto the query and the output, so the decode itself works in the 512-wide latent
space ("[ROCm] Dspark MLA module", Details: the decode's absorb BMM, run as an
FP8/FP4 BMM when those flags are on, else as torch.bmm):

  before the decode   q_lat[t, h, :] = q_nope[t, h, :] @ W_UK[h]    W_UK [H, 128, 512]
  after the decode    out[t, h, :]   = o_lat[t, h, :]  @ W_UV[h]    W_UV [H, 512, 128]

Both are the same operation, a matrix product per head over the token rows:

  y[t, h, j] = s * sum_k x[t, h, k] * w[h, k, j]

with x in bf16, the weight w in bf16 or fp8 e4m3fn (decoded exactly from its
bits) and s the weight's per-tensor float32 scale (1 for bf16 weights).  The
weight is stored as torch.bmm's right operand, [H, K, N] with N contiguous.
The result here is float64 and unrounded; the kernel rounds it to bf16.  Which
activation precision an "FP8 BMM" uses the pages do not say; this reading keeps
the activations in bf16 and the weight in fp8 with one scale.
"""
from __future__ import annotations

import numpy as np

from .formats import decode_bf16, decode_e4m3fn


def decode_weight(w_bits: np.ndarray, w_dtype: str) -> np.ndarray:
    """Weight bits -> float64 values (bf16: uint16 bits, fp8: uint8 e4m3fn codes)."""
    if w_dtype == "bf16":
        return decode_bf16(w_bits)
    if w_dtype == "fp8":
        return decode_e4m3fn(w_bits)
    raise ValueError(f"unknown weight dtype {w_dtype}")


def head_bmm_f64(x: np.ndarray, w: np.ndarray, scale: float = 1.0) -> np.ndarray:
    """x float64 [n, H, K], w float64 [H, K, N] -> scale * x[t, h] @ w[h], float64 [n, H, N]."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    n, H, K = x.shape
    assert w.shape[0] == H and w.shape[1] == K
    y = np.empty((n, H, w.shape[2]))
    for h in range(H):
        y[:, h, :] = x[:, h, :] @ w[h]
    return float(scale) * y


def absorb_bmm(x_bits: np.ndarray, w_bits: np.ndarray, w_dtype: str, w_scale: float = 1.0) -> np.ndarray:
    """bf16 bits x [n, H, K], weight bits [H, K, N] -> float64 [n, H, N] (before bf16 rounding).

    The scale is taken as the float32 the kernel receives.
    """
    return head_bmm_f64(decode_bf16(x_bits), decode_weight(w_bits, w_dtype), float(np.float32(w_scale)))
