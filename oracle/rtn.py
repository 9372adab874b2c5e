"""CPU oracle for round-to-nearest (RTN) INT4 quantisation -- TEST
INFRASTRUCTURE ONLY (same import rule as the rest of ``oracle/``).

What it computes (the pages' "naive round-to-nearest INT4" with a 4-bit zero
point and an fp16 scale per group of g values along K and per column, the
quantisation the W4A16 GEMM consumes: "LMDeploy, in depth", section
"Quantization: AWQ weights and KV cache"; the dequant rule of "LMDeploy
Guide: Fast Mixed-Precision LLM Inference Engine", section 3).  For every
group G (rows G*g .. G*g+g-1) and column n, with w the fp16 weights read as
exact binary32 values:

    lo = min(0, min_k w)      hi = max(0, max_k w)      (0 always representable)
    r  = hi - lo, or 15 when hi == lo (an all-zero group)
    s  = fp16(r / 15), at least the smallest positive fp16 (2^-24)
    z  = clamp(rint(-lo / s), 0, 15)
    q  = clamp(rint(w / s) + z, 0, 15)          (one division per weight)

Every operation is one IEEE binary32 operation with round-to-nearest-even
(rint ties to even), in this order.  The pages leave the precision open and
these values decide integers (codes), so the oracle states the precision in
which each decision is taken.  For the code itself binary32 and exact
arithmetic agree: w and s are fp16 values, and a quotient of two fp16 values
that is not a half-integer lies at least 1/8188 away from every half-integer,
far more than the binary32 rounding of the quotient can move it.  Pinned by
``tests/test_oracle_rtn.py`` (including exact ties at scales whose reciprocal
is inexact, where w * (1/s) would round the wrong way).
"""
from __future__ import annotations

import numpy as np

_TINY = np.float16(2.0 ** -24)


def quantize(W: np.ndarray, g: int):
    """W: fp16 [K][N] (float16 array, or uint16 bit patterns).  Returns
    (q uint8 [K][N], z uint8 [K/g][N], s fp16 [K/g][N])."""
    if W.dtype == np.uint16:
        W = W.view(np.float16)
    K, N = W.shape
    if K % g:
        raise ValueError("K must be a multiple of g")
    G = K // g
    w = W.astype(np.float32).reshape(G, g, N)                 # exact
    lo = np.minimum(w.min(axis=1), np.float32(0))              # [G][N]
    hi = np.maximum(w.max(axis=1), np.float32(0))
    r = hi - lo                                                 # one binary32 subtraction
    r = np.where(r == np.float32(0), np.float32(15), r)
    s16 = (r / np.float32(15)).astype(np.float16)               # binary32 division, then RNE to fp16
    s16 = np.maximum(s16, _TINY)
    sf = s16.astype(np.float32)                                 # exact
    z = np.clip(np.rint(-lo / sf), 0, 15).astype(np.float32)
    q = np.clip(np.rint(w / sf[:, None, :]) + z[:, None, :], 0, 15)  # binary32 division per weight
    return q.reshape(K, N).astype(np.uint8), z.astype(np.uint8), s16


def dequantize(q: np.ndarray, z: np.ndarray, s: np.ndarray, g: int) -> np.ndarray:
    """(q - z) * s in binary64 (exact: a small integer times an fp16 value)."""
    K, N = q.shape
    zz = np.repeat(z.astype(np.float64), g, axis=0)
    ss = np.repeat(s.astype(np.float64), g, axis=0)
    return (q.astype(np.float64) - zz) * ss


def bytes_moved(K: int, N: int, g: int) -> int:
    """Algorithmic bytes of one quantisation: read fp16 W, write one code per
    byte, one zero per byte and one fp16 scale per (group, column)."""
    G = K // g
    return 2 * K * N + K * N + G * N + 2 * G * N
