"""Pins of the low-bit KV-cache oracle (oracle/kv.py): quantiser grid recovery,
bound and packing order; attention closed forms (one token, uniform scores,
the two-token sigmoid that fixes the 1/sqrt(D) scale), the grouped-query head
mapping, the length mask; and planted mistakes the pins must reject."""
import math

import numpy as np
import pytest

import oracle.kv as kv


def _grid(bits, T=6, H=3, D=32, seed=2):
    rng = np.random.default_rng(seed)
    Bq = 2 ** bits - 1
    z = rng.integers(0, Bq + 1, size=(T, H))
    s = np.ldexp(1.0, -rng.integers(4, 10, size=(T, H)))
    q = rng.integers(0, Bq + 1, size=(T, H, D))
    q[..., 0] = 0
    q[..., 1] = Bq
    X = ((q - z[..., None]) * s[..., None]).astype(np.float16)
    return X, q.astype(np.uint8), z.astype(np.uint8), s.astype(np.float16)


def pins(quantize, attention):
    out = {}
    for bits in (8, 4):
        X, q0, z0, s0 = _grid(bits)
        c, s, z = quantize(X, bits)
        q = kv.unpack_codes(c, bits)
        out[f"grid_{bits}"] = bool(np.array_equal(q, q0) and np.array_equal(z, z0)
                                   and np.array_equal(s.view(np.uint16), s0.view(np.uint16)))
        rng = np.random.default_rng(bits)
        Y = (rng.normal(size=(5, 4, 128)) * 0.7).astype(np.float16)
        c, s, z = quantize(Y, bits)
        err = np.abs(Y.astype(np.float64) - kv.dequantize(c, s, z, bits))
        y = Y.astype(np.float64)
        r = np.maximum(y.max(-1), 0) - np.minimum(y.min(-1), 0)
        out[f"bound_{bits}"] = bool(np.all(err <= 0.5 * s.astype(np.float64)[..., None] + r[..., None] * 2.0 ** -10))
    # int4 packing: codes 0..15 in order -> bytes 0x10, 0x32, ..., 0xFE (even index in the low nibble)
    X = (np.arange(16) * 0.25).astype(np.float16).reshape(1, 16)   # lo = 0, hi = 3.75, s = 0.25, z = 0
    c, s, z = quantize(X, 4)
    out["nibbles"] = bool(np.array_equal(c[0], [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE])
                          and float(s[0]) == 0.25 and z[0] == 0)
    # int8 exact ties at a scale whose binary32 reciprocal is inexact: max
    # 1.7431640625 = 255 * 0.0068359375 (= 255 * 7 * 2^-10) gives s = 0.0068359375
    # (fp16 bits 0x1F00) exactly, z = 0; 6.5 s, 12.5 s, 14.5 s are fp16 values whose
    # quotient by s is exactly the half-integer -> the even codes 6, 12, 14
    # (x * fl(1/s) would give 7, 13, 15); 0.5, 1.0, 0.25 divide to 73.14, 146.29, 36.57.
    X = np.array([[0.0, 1.7431640625, 0.04443359375, 0.08544921875, 0.09912109375, 0.5, 1.0, 0.25]],
                 dtype=np.float16)
    c, s, z = quantize(X, 8)
    out["ties_inexact_reciprocal"] = bool(s.view(np.uint16)[0] == 0x1F00 and z[0] == 0
                                          and np.array_equal(c[0], [0, 255, 6, 12, 14, 73, 146, 37]))

    D = 128
    # one token: out = v exactly
    K = np.random.default_rng(0).normal(size=(1, 1, 1, D))
    V = np.random.default_rng(1).normal(size=(1, 1, 1, D))
    Q = np.random.default_rng(2).normal(size=(1, 1, D))
    out["one_token"] = bool(np.allclose(attention(Q, K, V, np.array([1])), V[:, 0], atol=1e-14))
    # uniform scores: out = mean of the V rows
    K = np.zeros((1, 5, 1, D))
    V = np.random.default_rng(3).normal(size=(1, 5, 1, D))
    out["uniform"] = bool(np.allclose(attention(np.ones((1, 1, D)), K, V, np.array([5]))[0, 0],
                                      V[0, :, 0].mean(axis=0), atol=1e-14))
    # two tokens, scores 0 and a / sqrt(D): p1 = 1 / (1 + exp(-a / sqrt(D)))
    a = 5.0
    K = np.zeros((1, 2, 1, D))
    K[0, 1, 0, 0] = a
    V = np.zeros((1, 2, 1, D))
    V[0, 1, 0, :] = 1.0
    Q = np.zeros((1, 1, D))
    Q[0, 0, 0] = 1.0
    p1 = 1.0 / (1.0 + math.exp(-a / math.sqrt(D)))
    out["sigmoid_scale"] = bool(abs(attention(Q, K, V, np.array([2]))[0, 0, 0] - p1) < 1e-14)
    # grouped heads: 8 query heads over 2 KV heads; V of KV head j is the constant j + 1
    K = np.zeros((1, 3, 2, D))
    V = np.zeros((1, 3, 2, D))
    V[:, :, 1, :] = 2.0
    V[:, :, 0, :] = 1.0
    o = attention(np.ones((1, 8, D)), K, V, np.array([3]))
    out["gqa"] = bool(np.allclose(o[0, :, 0], [1, 1, 1, 1, 2, 2, 2, 2]))
    # length mask: tokens at and beyond the length are ignored
    V = np.zeros((1, 4, 1, D))
    V[0, 2:, 0, :] = 1e6
    out["length"] = bool(np.allclose(attention(np.ones((1, 1, D)), np.zeros((1, 4, 1, D)), V, np.array([2])), 0.0))
    return out


def test_oracle_passes_every_pin():
    res = pins(kv.quantize, kv.decode_attention)
    assert all(res.values()), res


def _quant_swapped_nibbles(X, bits):
    c, s, z = kv.quantize(X, bits)
    if bits == 4:
        c = ((c >> 4) | (c << 4)).astype(np.uint8)
    return c, s, z


def _quant_zero_sign(X, bits):
    c, s, z = kv.quantize(X, bits)
    return c, s, ((2 ** bits - 1) - z).astype(np.uint8)


def _quant_reciprocal(X, bits):
    """The rule with x * (1/s) in place of the division x / s."""
    Bq = np.float32(2 ** bits - 1)
    x = X.astype(np.float32)
    lo = np.minimum(x.min(axis=-1), np.float32(0))
    hi = np.maximum(x.max(axis=-1), np.float32(0))
    r = hi - lo
    r = np.where(r == np.float32(0), Bq, r)
    s16 = np.maximum((r / Bq).astype(np.float16), np.float16(2.0 ** -24))
    sf = s16.astype(np.float32)
    z = np.clip(np.rint(-lo / sf), 0, Bq).astype(np.float32)
    q = np.clip(np.rint(x * (np.float32(1) / sf)[..., None]) + z[..., None], 0, Bq).astype(np.uint8)
    if bits == 4:
        q = (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)
    return q, s16, z.astype(np.uint8)


def _attn_no_scale(Q, K, V, lengths):
    return kv.decode_attention(np.asarray(Q) * np.sqrt(Q.shape[-1]), K, V, lengths)


def _attn_head_modulo(Q, K, V, lengths):
    Bsz, Hq, D = Q.shape
    Hkv = K.shape[2]
    out = np.zeros((Bsz, Hq, D))
    for h in range(Hq):
        out[:, h:h + 1] = kv.decode_attention(Q[:, h:h + 1], K[:, :, h % Hkv:h % Hkv + 1], V[:, :, h % Hkv:h % Hkv + 1],
                                              lengths)
    return out


def _attn_length_plus_one(Q, K, V, lengths):
    return kv.decode_attention(Q, K, V, np.minimum(np.asarray(lengths) + 1, K.shape[1]))


@pytest.mark.parametrize("quantize,attention", [
    (_quant_swapped_nibbles, kv.decode_attention), (_quant_zero_sign, kv.decode_attention),
    (_quant_reciprocal, kv.decode_attention),
    (kv.quantize, _attn_no_scale), (kv.quantize, _attn_head_modulo), (kv.quantize, _attn_length_plus_one)],
    ids=["nibble_order", "zero_sign", "reciprocal", "no_sqrt_d", "head_modulo", "length_off_by_one"])
def test_pins_reject_planted_mistakes(quantize, attention):
    res = pins(quantize, attention)
    assert not all(res.values()), res


def test_cache_bytes_against_the_pages_kv_sizing():
    # fp16 KV of Llama-3-8B is 131,072 bytes per token (32 layers x 8 KV heads x 128 x K,V x 2 B)
    fp16 = 32 * 2 * 8 * 128 * 2
    assert fp16 == 131072
    int8 = 32 * kv.cache_bytes(1, 1, 8, 128, 8)
    int4 = 32 * kv.cache_bytes(1, 1, 8, 128, 4)
    assert int8 == 67072 and int4 == 34304        # codes + fp16 scale + uint8 zero per (token, head)
    assert 0.5 < int8 / fp16 < 0.52 and 0.26 < int4 / fp16 < 0.27
