"""CPU oracle for the W4A16 GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or executes anything here.

Contents:
  * ``gemm`` / ``dequant``: ctypes front end of ``oracle.c`` (plain fp64
    definition of Y = X . dequant(W), see that file's header).
  * sizing arithmetic the pages fix (bytes moved by a W4A16 GEMM, KV-cache
    bytes per token, the Llama-3 layer shapes), used as invariants.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
closed forms, library special cases, hand-worked examples and the pages'
printed numbers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (plain -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_gemm.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 4 + [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_dequant.restype = None
        lib.oracle_dequant.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
        lib.oracle_half_to_double.restype = ctypes.c_double
        lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(int(bits) & 0xFFFF)


def gemm(X: np.ndarray, q: np.ndarray, z: np.ndarray, s: np.ndarray, g: int,
         rows: Optional[Sequence[int]] = None, threads: Optional[int] = None) -> np.ndarray:
    """fp64 Y[rows, :] of Y = X . dequant(W).

    X fp16 [M][K], q uint8 [K][N], z uint8 [K/g][N], s fp16 [K/g][N].
    Returns float64 [len(rows)][N] (all M rows when ``rows`` is None).
    """
    X = _c(X, np.float16)
    q = _c(q, np.uint8)
    z = _c(z, np.uint8)
    s = _c(s, np.float16)
    M, K = X.shape
    K2, N = q.shape
    if K2 != K or z.shape != (K // g, N) or s.shape != (K // g, N):
        raise ValueError("shape mismatch")
    if rows is None:
        r = None
        nrows = M
    else:
        r = _c(np.asarray(rows), np.int32)
        nrows = len(r)
    Y = np.empty((nrows, N), dtype=np.float64)
    st = _load().oracle_gemm(X.ctypes.data, q.ctypes.data, z.ctypes.data, s.ctypes.data, M, K, N, g,
                             None if r is None else r.ctypes.data, nrows, Y.ctypes.data,
                             threads or default_threads())
    if st == 3:
        raise ValueError("code above 15")
    if st:
        raise RuntimeError(f"oracle_gemm failed with status {st}")
    return Y


def dequant(q: np.ndarray, z: np.ndarray, s: np.ndarray, g: int) -> np.ndarray:
    q = _c(q, np.uint8)
    z = _c(z, np.uint8)
    s = _c(s, np.float16)
    K, N = q.shape
    W = np.empty((K, N), dtype=np.float64)
    _load().oracle_dequant(q.ctypes.data, z.ctypes.data, s.ctypes.data, K, N, g, W.ctypes.data)
    return W


def rel_max_err(Y: np.ndarray, Y_ref: np.ndarray) -> float:
    """max|Y - Y_ref| / max|Y_ref| -- the parity measure of the W4A16 GEMM."""
    Y = np.asarray(Y, dtype=np.float64)
    den = float(np.max(np.abs(Y_ref))) if Y_ref.size else 0.0
    num = float(np.max(np.abs(Y - Y_ref))) if Y_ref.size else 0.0
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return num / den


# ---------------------------------------------------------------------------
# Sizing arithmetic.

def algorithmic_bytes(M: int, K: int, N: int, g: int) -> int:
    """Bytes a W4A16 GEMM must move: 4-bit codes, fp16 scale and 4-bit zero per
    (group, column), fp16 X in and fp16 Y out."""
    G = K // g
    return K * N // 2 + G * N * 2 + G * N // 2 + 2 * M * K + 2 * M * N


def flops(M: int, K: int, N: int) -> int:
    return 2 * M * N * K


def bits_per_weight(g: int) -> float:
    """Storage bits per weight: 4 for the code plus (16 + 4) per group of g."""
    return 4.0 + 20.0 / g


def compression_vs_fp16(g: int) -> float:
    return 16.0 / bits_per_weight(g)


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    """Keys and values of one token across all layers (the KV sizing example of
    "LMDeploy, in depth", section "KV cache memory: a worked sizing example")."""
    return 2 * layers * kv_heads * head_dim * elem_bytes


def llama_linear_shapes(hidden: int, heads: int, kv_heads: int, head_dim: int,
                        intermediate: int) -> dict:
    """(K, N) of the four linear layers of a Llama-style block, with fused
    qkv and fused gate/up projections."""
    assert heads * head_dim == hidden
    return {
        "qkv": (hidden, hidden + 2 * kv_heads * head_dim),
        "o_proj": (hidden, hidden),
        "gate_up": (hidden, 2 * intermediate),
        "down": (intermediate, hidden),
    }


def linear_weight_count(layers: int, shapes: dict) -> int:
    return layers * sum(K * N for (K, N) in shapes.values())
