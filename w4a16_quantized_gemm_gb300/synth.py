"""Seeded synthetic inputs for the W4A16 GEMM ``Y[M,N] = X[M,K] . dequant(W)``.

This module only draws random numbers; it holds none of the method's
arithmetic (no dequantisation, no product).  Both the CPU oracle and the CUDA
path are fed from it, so the two sides see identical bytes.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style: draw ``i`` of a stream
with 64-bit key ``c`` is ``mix(c + (i + 1) * 0x9E3779B97F4A7C15)``.  A stream
key is ``mix`` of the FNV-1a hash of a text tag naming the tensor and its
shape, so every tensor of every workload has its own stream.

Value recipe (the workloads of the W4A16 pages, shapes of Llama-3-8B/70B
linear layers):
  * q, z   : uniform integers 0..15 (top four bits of a draw).
  * s      : uniform in [1e-3, 2e-2] in fp64 (53-bit uniform), rounded to fp16.
  * X      : N(0, 1) by Box-Muller (cosine branch) in fp64, rounded to fp16.
  * stress : round(0.01*K) salient K-channels, the first ones of a seeded
             permutation, have their X column scaled by 20 before rounding, and
             every group holding at least one of them has its whole scale row
             scaled by 1/20 once before rounding (AWQ-style salient channels).
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, List, Optional, Tuple

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _mix_scalar(v: int) -> int:
    return int(_mix(np.array([v], dtype=np.uint64))[0])


def stream_key(tag: str) -> int:
    """64-bit stream key for a text tag (FNV-1a 64, then one SplitMix64 mix)."""
    h = 0xCBF29CE484222325
    for b in tag.encode():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return _mix_scalar(h)


def draws(key: int, n: int, offset: int = 0) -> np.ndarray:
    """Draws ``offset .. offset+n-1`` of the stream with ``key`` (uint64)."""
    i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(key) + i * _GAMMA)


def _chunks(n: int, work) -> None:
    """Run ``work(a, b)`` over [0, n) in chunks of _CHUNK, on a thread pool when
    there is more than one chunk (NumPy releases the GIL inside its array
    operations; each chunk writes its own slice, so the result does not depend
    on the thread count)."""
    spans = [(a, min(n, a + _CHUNK)) for a in range(0, n, _CHUNK)]
    if len(spans) <= 1:
        for a, b in spans:
            work(a, b)
        return
    with ThreadPoolExecutor(max_workers=min(len(spans), os.cpu_count() or 1)) as ex:
        list(ex.map(lambda ab: work(*ab), spans))


def _fill(key: int, n: int, fn, dtype) -> np.ndarray:
    out = np.empty(n, dtype=dtype)

    def work(a, b):
        out[a:b] = fn(draws(key, b - a, a))

    _chunks(n, work)
    return out


def _nibbles(r: np.ndarray) -> np.ndarray:
    return (r >> np.uint64(60)).astype(np.uint8)


def _unit(r: np.ndarray) -> np.ndarray:
    """[0, 1) with 53 random bits."""
    return (r >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def codes(tag: str, rows: int, cols: int) -> np.ndarray:
    return _fill(stream_key(tag), rows * cols, _nibbles, np.uint8).reshape(rows, cols)


def scales64(tag: str, rows: int, cols: int, lo: float = 1e-3, hi: float = 2e-2) -> np.ndarray:
    return _fill(stream_key(tag), rows * cols, lambda r: lo + (hi - lo) * _unit(r),
                 np.float64).reshape(rows, cols)


def normal64(tag: str, rows: int, cols: int) -> np.ndarray:
    """Standard normal by Box-Muller: draws 2i and 2i+1 give element i."""
    n = rows * cols
    key = stream_key(tag)
    out = np.empty(n, dtype=np.float64)

    def work(a, b):
        r = draws(key, 2 * (b - a), 2 * a)
        u1 = ((r[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)
        u2 = _unit(r[1::2])
        out[a:b] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)

    _chunks(n, work)
    return out.reshape(rows, cols)


def salient_channels(tag: str, K: int) -> np.ndarray:
    """First round(0.01*K) entries of a seeded permutation of 0..K-1 (sorted)."""
    count = int(np.floor(0.01 * K + 0.5))
    perm = np.argsort(draws(stream_key(tag), K), kind="stable")
    return np.sort(perm[:count]).astype(np.int64)


@dataclasses.dataclass
class Problem:
    """One W4A16 GEMM instance: X fp16 [M][K], q u8 [K][N], z u8 [K/g][N], s fp16 [K/g][N]."""
    M: int
    K: int
    N: int
    g: int
    X: np.ndarray
    q: np.ndarray
    z: np.ndarray
    s: np.ndarray
    salient: Optional[np.ndarray] = None

    @property
    def name(self) -> str:
        return f"M{self.M}_K{self.K}_N{self.N}_g{self.g}" + ("_stress" if self.salient is not None else "")


def weights(K: int, N: int, g: int, stress: bool = False, seed: int = 0
            ) -> Tuple[np.ndarray, np.ndarray, np.ndarray, Optional[np.ndarray]]:
    """q, z, s (and the salient channel list under ``stress``) for a K x N layer."""
    if K % g:
        raise ValueError("K must be a multiple of g")
    base = f"seed{seed}/K{K}/N{N}/g{g}" + ("/stress" if stress else "")
    G = K // g
    q = codes(base + "/q", K, N)
    z = codes(base + "/z", G, N)
    s64 = scales64(base + "/s", G, N)
    sal = None
    if stress:
        sal = salient_channels(f"seed{seed}/K{K}/salient", K)
        grp = np.unique(sal // g)
        s64[grp, :] = s64[grp, :] / 20.0
    return q, z, s64.astype(np.float16), sal


def activations(M: int, K: int, salient: Optional[np.ndarray] = None, seed: int = 0,
                tag: str = "") -> np.ndarray:
    x64 = normal64(f"seed{seed}/X/M{M}/K{K}{tag}", M, K)
    if salient is not None:
        x64[:, salient] = x64[:, salient] * 20.0
    return x64.astype(np.float16)


def problem(M: int, K: int, N: int, g: int = 128, stress: bool = False, seed: int = 0) -> Problem:
    q, z, s, sal = weights(K, N, g, stress, seed)
    X = activations(M, K, sal, seed, tag=f"/N{N}/g{g}" + ("/stress" if stress else ""))
    return Problem(M, K, N, g, X, q, z, s, sal)


# ---------------------------------------------------------------------------
# The workloads: Llama-3-8B and Llama-3-70B linear-layer shapes.
# (K, N): qkv = (hidden, hidden + 2*kv_heads*head_dim), o_proj = (hidden, hidden),
# gate_up = (hidden, 2*intermediate), down = (intermediate, hidden).
def fp16_weights(K: int, N: int, g: int = 128, seed: int = 0) -> np.ndarray:
    """Dense fp16 weights [K][N] for the round-to-nearest quantiser: N(0,1)
    times a per-column scale uniform in [0.005, 0.05] (a trained layer's
    spread), rounded to fp16.  The first column's first group is all zeros and
    the second column's first group constant (the quantiser's degenerate
    cases) when the shape has them."""
    tag = f"w16/K{K}/N{N}/g{g}/s{seed}"
    col = scales64(tag + "/col", 1, N, 0.005, 0.05)
    W = (normal64(tag, K, N) * col).astype(np.float16)
    if K >= g and N >= 2:
        W[:g, 0] = 0
        W[:g, 1] = np.float16(0.0123)
    return W


LLAMA3_8B = {"qkv": (4096, 6144), "o_proj": (4096, 4096), "gate_up": (4096, 28672),
             "down": (14336, 4096)}
LLAMA3_70B = {"qkv": (8192, 10240), "o_proj": (8192, 8192), "gate_up": (8192, 57344),
              "down": (28672, 8192)}


@dataclasses.dataclass(frozen=True)
class Case:
    M: int
    K: int
    N: int
    g: int
    stress: bool = False
    layer: str = ""

    @property
    def name(self) -> str:
        return f"{self.layer}_M{self.M}_K{self.K}_N{self.N}_g{self.g}" + ("_stress" if self.stress else "")


def workload(idx: int) -> List[Case]:
    """The five workloads, as lists of GEMM cases.

    0: one 1x4096x4096 GEMM, g=128 (small enough for the full oracle).
    1: Llama-3-8B decode: M in {1,8,16,32} x the four layer shapes, g=128.
    2: Llama-3-8B prefill: M in {128,1024,4096} x the four layer shapes, g=128.
    3: Llama-3-70B: M in {1,16,256,2048} x the four layer shapes, g=128.
    4: stress: 8B gate_up and down, M in {1,64,2048}, g in {64,128}, salient channels.
    """
    if idx == 0:
        return [Case(1, 4096, 4096, 128, False, "square")]
    if idx == 1:
        return [Case(M, K, N, 128, False, l) for M in (1, 8, 16, 32) for l, (K, N) in LLAMA3_8B.items()]
    if idx == 2:
        return [Case(M, K, N, 128, False, l) for M in (128, 1024, 4096) for l, (K, N) in LLAMA3_8B.items()]
    if idx == 3:
        return [Case(M, K, N, 128, False, l) for M in (1, 16, 256, 2048) for l, (K, N) in LLAMA3_70B.items()]
    if idx == 4:
        return [Case(M, K, N, g, True, l) for g in (64, 128) for M in (1, 64, 2048)
                for l in ("gate_up", "down") for (K, N) in [LLAMA3_8B[l]]]
    raise ValueError(idx)


def case_problem(c: Case, seed: int = 0) -> Problem:
    return problem(c.M, c.K, c.N, c.g, c.stress, seed)
