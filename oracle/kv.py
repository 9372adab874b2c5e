"""CPU oracle of the low-bit KV cache -- TEST INFRASTRUCTURE ONLY (same import
rule as the rest of ``oracle/``).

What the pages fix ("LMDeploy, in depth", section "Quantization: AWQ weights
and KV cache"): keys and values are stored as int8 (quant_policy 8) or int4
(quant_policy 4), quantised online, asymmetrically, per head and per token;
the guide's "Adaptive Head Alignment" and "Asynchronous KV Memory Loading
Pipeline" sections describe decode attention that reads the low-bit cache
directly.  Readings (ours, where the pages stop):

  * per (token, head) vector x of D values, B = 2^bits - 1, binary32 with
    round-to-nearest-even at each step (the decisions are integers, so the
    oracle takes the kernel's precision):
        lo = min(0, min x), hi = max(0, max x); r = hi - lo, or B if r == 0
        s = fp16(r / B), at least 2^-24;  z = clamp(rint(-lo / s), 0, B)
        q = clamp(rint(x / s) + z, 0, B)          (one division per value)
    -- the same rule as the weight quantiser, along the head dimension (x and
    s are fp16, so the binary32 quotient rounds to the same integer as the
    exact one);
  * storage: codes [.., D] one byte each (int8) or two per byte, even index in
    the low nibble (int4); s fp16 and z uint8 per (token, head);
  * decode attention for one query token per sequence, grouped-query heads
    (query head h reads KV head h // (Hq / Hkv)):
        k~ = (qk - zk) sk,  v~ = (qv - zv) sv          (exact in binary64)
        p_t = softmax_t( q . k~_t / sqrt(D) ),  t < length
        out = sum_t p_t v~_t
    in binary64 on the dequantised cache.  Pinned by ``tests/test_oracle_kv.py``.
"""
from __future__ import annotations

import numpy as np

_TINY = np.float16(2.0 ** -24)


def quantize(X: np.ndarray, bits: int):
    """X fp16 [..., D] -> (codes uint8 [..., D] or [..., D/2], s fp16 [...], z uint8 [...])."""
    if bits not in (4, 8):
        raise ValueError("bits must be 4 or 8")
    if X.dtype == np.uint16:
        X = X.view(np.float16)
    B = np.float32(2 ** bits - 1)
    x = X.astype(np.float32)
    lo = np.minimum(x.min(axis=-1), np.float32(0))
    hi = np.maximum(x.max(axis=-1), np.float32(0))
    r = hi - lo
    r = np.where(r == np.float32(0), B, r)
    s16 = np.maximum((r / B).astype(np.float16), _TINY)
    sf = s16.astype(np.float32)
    z = np.clip(np.rint(-lo / sf), 0, B).astype(np.float32)
    q = np.clip(np.rint(x / sf[..., None]) + z[..., None], 0, B).astype(np.uint8)  # binary32 division
    if bits == 4:
        q = (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)
    return q, s16, z.astype(np.uint8)


def unpack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    if bits == 8:
        return codes
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = codes & 15
    out[..., 1::2] = codes >> 4
    return out


def dequantize(codes: np.ndarray, s: np.ndarray, z: np.ndarray, bits: int) -> np.ndarray:
    q = unpack_codes(codes, bits).astype(np.float64)
    return (q - z.astype(np.float64)[..., None]) * s.astype(np.float64)[..., None]


def decode_attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray, lengths: np.ndarray) -> np.ndarray:
    """Q [B][Hq][D]; K, V [B][L][Hkv][D] (binary64 values); lengths [B].
    Returns out [B][Hq][D] in binary64 (rows with length 0 are zero)."""
    Q = np.asarray(Q, dtype=np.float64)
    Bsz, Hq, D = Q.shape
    Hkv = K.shape[2]
    grp = Hq // Hkv
    out = np.zeros((Bsz, Hq, D))
    for b in range(Bsz):
        n = int(lengths[b])
        if n == 0:
            continue
        for h in range(Hq):
            kh = K[b, :n, h // grp, :]
            vh = V[b, :n, h // grp, :]
            sc = kh @ Q[b, h] / np.sqrt(D)
            p = np.exp(sc - sc.max())
            out[b, h] = (p / p.sum()) @ vh
    return out


def cache_bytes(Bsz: int, L: int, Hkv: int, D: int, bits: int) -> int:
    """Bytes of K and V for Bsz sequences of L tokens: codes plus an fp16 scale
    and a uint8 zero per (token, head)."""
    return 2 * Bsz * L * Hkv * (D * bits // 8 + 3)
