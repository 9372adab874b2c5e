"""Pins of the round-to-nearest INT4 quantisation oracle (oracle/rtn.py),
independent of the oracle's own code: exact recovery of weights that lie on a
quantisation grid, the RTN error bound, the degenerate groups, hand-worked
ties (also at a scale whose binary32 reciprocal is inexact, which tells the
per-weight division from a multiplication by 1/s), and planted mistakes that
each pin set must reject."""
import numpy as np
import pytest

import oracle.rtn as rtn
from w4a16_quantized_gemm_gb300 import synth


def _grid_problem(G=3, g=16, N=24, seed=1):
    """W = (q - z) * s with s a power of two; every (group, column) holds the
    codes 0 and 15, so its range is exactly 15 s and 0 lies inside it."""
    rng = np.random.default_rng(seed)
    z = rng.integers(0, 16, size=(G, N))
    e = rng.integers(3, 11, size=(G, N))
    s = np.ldexp(1.0, -e)                                  # 2^-3 .. 2^-10, exact in fp16
    q = rng.integers(0, 16, size=(G * g, N))
    for gi in range(G):
        q[gi * g, :] = 0
        q[gi * g + 1, :] = 15
    W = (q - np.repeat(z, g, axis=0)) * np.repeat(s, g, axis=0)
    W16 = W.astype(np.float16)
    assert np.array_equal(W16.astype(np.float64), W)     # the grid is exact in fp16
    return W16, q.astype(np.uint8), z.astype(np.uint8), s.astype(np.float16)


def pins(quantize):
    """Every pin as one boolean, so that mutants can be scored."""
    out = {}
    W16, q0, z0, s0 = _grid_problem()
    q, z, s = quantize(W16, 16)
    out["grid_recovery"] = (np.array_equal(q, q0) and np.array_equal(z, z0)
                            and np.array_equal(s.view(np.uint16), s0.view(np.uint16)))

    # RTN bound on dense weights: |w - (q - z) s| <= s/2 plus the fp16 rounding of s
    W = synth.fp16_weights(256, 64, g=64, seed=3)
    q, z, s = quantize(W, 64)
    err = np.abs(W.astype(np.float64) - rtn.dequantize(q, z, s, 64))
    sd = np.repeat(s.astype(np.float64), 64, axis=0)
    w = W.astype(np.float64).reshape(4, 64, 64)
    r = (np.maximum(w.max(axis=1), 0) - np.minimum(w.min(axis=1), 0))
    out["rtn_bound"] = bool(np.all(err <= 0.5 * sd + np.repeat(r, 64, axis=0) * 2.0 ** -10 + 1e-12))
    out["codes_in_range"] = bool(q.max() <= 15 and z.max() <= 15)

    # degenerate groups: all zeros; constant positive; constant negative
    D = np.zeros((8, 3), dtype=np.float16)
    D[:, 1] = 0.75
    D[:, 2] = -0.375
    q, z, s = quantize(D, 8)
    out["zero_group"] = bool(np.all(q[:, 0] == 0) and z[0, 0] == 0 and float(s[0, 0]) == 1.0)
    # 0.75 / 15 = 1.6 * 2^-5: fp16 mantissa 614.4 -> 614, bits 0x2A66 (0.0499878);
    # 0.375 / 15 = 1.6 * 2^-6 -> bits 0x2666 (0.0249939); c / s = +-15.004 -> code 15 or 0
    sb = s.view(np.uint16)
    out["const_pos"] = bool(z[0, 1] == 0 and np.all(q[:, 1] == 15) and sb[0, 1] == 0x2A66)
    out["const_neg"] = bool(z[0, 2] == 15 and np.all(q[:, 2] == 0) and sb[0, 2] == 0x2666)

    # hand-worked ties: range [-7.5, 7.5] -> s = 1, z = rint(7.5) = 8 (half to even);
    # w = 2.5 -> rint 2 -> 10; w = 3.5 -> 4 -> 12; w = -0.5 -> -0 -> 8; w = -6.5 -> -6 -> 2
    T = np.array([-7.5, 7.5, 2.5, 3.5, -0.5, -6.5, 0.0, 1.0], dtype=np.float16).reshape(8, 1)
    q, z, s = quantize(np.repeat(T, 16, axis=1), 8)
    out["ties"] = bool(float(s[0, 0]) == 1.0 and z[0, 0] == 8
                       and np.all(q[:, 0] == np.array([0, 15, 10, 12, 8, 2, 8, 9])))

    # exact ties at a scale whose reciprocal is inexact in binary32: the group
    # max 0.150146484375 = 1230 * 2^-13 gives s = hi / 15 = 1025 * 2^-17 =
    # 0.010009765625 (fp16 bits 0x2120) exactly, z = 0; w = 3.5 s, 7.5 s and
    # 13.5 s are fp16 values, w / s is exactly the half-integer and rounds to
    # the even code 4, 8, 14 (w * fl(1/s) lands just below each and would give
    # 3, 7, 13); 0.01, 0.06 and 0.1 (as fp16) divide to 0.9985, 5.994, 9.988.
    H = np.array([0.0, 0.150146484375, 0.0350341796875, 0.0750732421875, 0.1351318359375, 0.01, 0.06, 0.1],
                 dtype=np.float16).reshape(8, 1)
    q, z, s = quantize(np.repeat(H, 16, axis=1), 8)
    out["ties_inexact_reciprocal"] = bool(s.view(np.uint16)[0, 0] == 0x2120 and z[0, 0] == 0
                                          and np.all(q[:, 0] == np.array([0, 15, 4, 8, 14, 1, 6, 10])))
    return out


def test_oracle_passes_every_pin():
    res = pins(rtn.quantize)
    assert all(res.values()), res


def _mutant(kind):
    def quantize(W, g):
        K, N = W.shape
        G = K // g
        w = W.astype(np.float32).reshape(G, g, N)
        lo, hi = w.min(axis=1), w.max(axis=1)
        if kind != "no_zero_in_range":
            lo, hi = np.minimum(lo, np.float32(0)), np.maximum(hi, np.float32(0))
        r = hi - lo
        r = np.where(r == 0, np.float32(15), r)
        den = np.float32(16 if kind == "divide_by_16" else 15)
        s16 = np.maximum((r / den).astype(np.float16), np.float16(2.0 ** -24))
        sf = s16.astype(np.float32)
        rnd = np.floor if kind == "floor" else np.rint
        zz = rnd((lo if kind == "zero_sign" else -lo) / sf)
        z = np.clip(zz, 0, 15)
        top = 16 if kind == "clamp_16" else 15
        quot = w * (np.float32(1) / sf)[:, None, :] if kind == "reciprocal" else w / sf[:, None, :]
        q = np.clip(rnd(quot) + z[:, None, :], 0, top)
        if kind == "round_half_up":
            q = np.clip(np.floor(quot + 0.5) + z[:, None, :], 0, 15)
            z = np.clip(np.floor(-lo / sf + 0.5), 0, 15)
        return q.reshape(K, N).astype(np.uint8), z.astype(np.uint8), s16
    return quantize


@pytest.mark.parametrize("kind", ["no_zero_in_range", "divide_by_16", "floor", "zero_sign", "clamp_16",
                                  "round_half_up", "reciprocal"])
def test_pins_reject_planted_mistakes(kind):
    res = pins(_mutant(kind))
    assert not all(res.values()), (kind, res)


def test_bytes_moved():
    # fp16 in, one code per byte out, a zero byte and an fp16 scale per (group, column)
    assert rtn.bytes_moved(4096, 4096, 128) == 2 * 4096 * 4096 + 4096 * 4096 + 32 * 4096 * 3
