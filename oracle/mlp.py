"""CPU oracle of the fused gate/up epilogue -- TEST INFRASTRUCTURE ONLY (same
import rule as the rest of ``oracle/``).

The pages mention fused weight-only INT4 GEMMs for the MLP ("LMDeploy, in
depth", section on the TurboMind kernels) without detail; the plainest fusion
for a Llama MLP is the gate/up product followed by SiLU(gate) * up.  Layout
convention (ours): the gate/up weight has N = 2 I columns interleaved in
blocks of 4 -- columns 8b .. 8b+3 are gate columns 4b .. 4b+3 and columns
8b+4 .. 8b+7 the matching up columns -- so that every 8-column-aligned slice
of the output holds whole pairs.  With Y = X . dequant(W) in fp64:

    h[m][j] = silu(Y[m][c(j)]) * Y[m][c(j) + 4],   c(j) = 8 (j div 4) + (j mod 4)
    silu(x) = x / (1 + exp(-x))

evaluated in binary64.  Pinned by ``tests/test_oracle_mlp.py``.
"""
from __future__ import annotations

import numpy as np


def gate_columns(N: int) -> np.ndarray:
    """c(j) for j = 0 .. N/2 - 1."""
    j = np.arange(N // 2)
    return 8 * (j // 4) + (j % 4)


def silu(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def silu_mul(Y: np.ndarray) -> np.ndarray:
    """h [M][N/2] from the gate/up product Y [M][N] (N a multiple of 8)."""
    Y = np.asarray(Y, dtype=np.float64)
    N = Y.shape[1]
    if N % 8:
        raise ValueError("N must be a multiple of 8")
    c = gate_columns(N)
    return silu(Y[:, c]) * Y[:, c + 4]


def error_bound(Y_ref: np.ndarray, gemm_tol: float) -> np.ndarray:
    """Element-wise bound on |h - h_ref| when every element of Y carries an
    error of at most gemm_tol * max|Y_ref| (the GEMM's parity bar) and h is
    rounded once to fp16: |d silu / dx| <= 1.1 (its maximum, 1.0998 at
    x = 2.3994), so |dh| <= e (1.1 |u| + |silu(g)| + 1.1 e) + 2^-11 |h|."""
    Y_ref = np.asarray(Y_ref, dtype=np.float64)
    c = gate_columns(Y_ref.shape[1])
    g, u = Y_ref[:, c], Y_ref[:, c + 4]
    e = gemm_tol * float(np.max(np.abs(Y_ref))) if Y_ref.size else 0.0
    h = silu(g) * u
    return e * (1.1 * np.abs(u) + np.abs(silu(g)) + 1.1 * e) + 2.0 ** -11 * np.abs(h) + 1e-30
