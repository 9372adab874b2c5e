"""CPU oracle of the W8A8 GEMM -- TEST INFRASTRUCTURE ONLY (same import rule as
the rest of ``oracle/``).

What the pages fix: W8A8 is one of the precision formats the engine serves
("LMDeploy Guide: Fast Mixed-Precision LLM Inference Engine", the pillar on
configuration-agnostic generalisation and the comparison table; the PyTorch
engine's "w8a8 quantization"), produced by post-training quantisation such as
SmoothQuant (the guide's introduction): 8-bit integer weights and 8-bit integer
activations.  The pages stop there; our reading, the SmoothQuant scheme in its
plainest form (the smoothing factors are folded into the fp16 weights and the
preceding layer beforehand, so the GEMM never sees them):

  * activations, per token (row m of X [M][K]), symmetric and dynamic:
        a  = max_k |x|;  s_x = a / 127, or 1 when a == 0
        q_x = clamp(rint(x / s_x), -127, 127)        (one division per value)
  * weights, per output channel (column n of W [K][N]), the same rule:
        s_w = max_k |w| / 127 (or 1);  q_w = clamp(rint(w / s_w), -127, 127)
  * every step one IEEE binary32 operation with round-to-nearest-even (the
    decisions are integers, so the oracle states their precision; s is a
    binary32 value here, and x * (1 / s) can differ from x / s by enough to
    move a code, e.g. at a = 0.50146484375, x = a / 2);
  * the product:  Y[m][n] = s_x[m] s_w[n] sum_k q_x[m][k] q_w[k][n]
    -- the integer sum exact (int64 here), the scaling in binary64.

Pinned by ``tests/test_oracle_w8a8.py``.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

QMAX = 127


def _quantize_rows(x: np.ndarray):
    """x binary32 [R][C]: per-row symmetric int8 codes and binary32 scales."""
    a = np.abs(x).max(axis=1)
    s = a / np.float32(QMAX)                         # one binary32 division
    s = np.where(a == np.float32(0), np.float32(1), s).astype(np.float32)
    q = np.clip(np.rint(x / s[:, None]), -QMAX, QMAX).astype(np.int8)  # binary32 division per value
    return q, s


def quantize_act(X: np.ndarray):
    """X fp16 [M][K] (float16, or uint16 bit patterns) -> (q int8 [M][K], s_x float32 [M])."""
    if X.dtype == np.uint16:
        X = X.view(np.float16)
    return _quantize_rows(X.astype(np.float32))


def quantize_weight(W: np.ndarray):
    """W fp16 [K][N] -> (q int8 [K][N], s_w float32 [N]), per output channel."""
    if W.dtype == np.uint16:
        W = W.view(np.float16)
    q, s = _quantize_rows(np.ascontiguousarray(W.astype(np.float32).T))
    return np.ascontiguousarray(q.T), s


def gemm(qx: np.ndarray, sx: np.ndarray, qw: np.ndarray, sw: np.ndarray,
         rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Y [M][N] (or the listed rows) in binary64: s_x[m] s_w[n] (q_x q_w)[m][n],
    the integer products summed exactly in int64."""
    if rows is not None:
        qx, sx = qx[list(rows)], sx[list(rows)]
    acc = qx.astype(np.int64) @ qw.astype(np.int64)          # exact: |sum| < 2^63
    return sx.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :] * acc.astype(np.float64)


def algorithmic_bytes(M: int, K: int, N: int) -> int:
    """Bytes one GEMM must move at least: int8 weights and activations, the
    per-channel and per-token fp32 scales, the fp16 output."""
    return K * N + 4 * N + M * K + 4 * M + 2 * M * N
