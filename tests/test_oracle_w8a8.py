"""Pins of the W8A8 oracle (oracle/w8a8.py): grid recovery of the symmetric
quantiser, its error bound and sign symmetry, the all-zero row, the integer
product against brute force on tiny inputs, a hand-worked 2 x 3 x 2 product,
and planted mistakes the pins must reject."""
import numpy as np
import pytest

import oracle.w8a8 as w8


def _grid(R=5, C=64, seed=0):
    """Rows whose values are exactly q * s with max |q| = 127 and s a power of two."""
    rng = np.random.default_rng(seed)
    q = rng.integers(-127, 128, size=(R, C))
    q[:, 0] = 127
    q[1, 0] = -127
    q[1, 1:] = np.clip(q[1, 1:], -126, 126)       # row 1: the maximum magnitude only as -127
    s = np.ldexp(1.0, -rng.integers(6, 12, size=R))
    X = (q * s[:, None]).astype(np.float16)
    assert np.array_equal(X.astype(np.float64), q * s[:, None])   # exactly representable
    return X, q, s


def pins(quantize_act, gemm):
    out = {}
    X, q0, s0 = _grid()
    q, s = quantize_act(X)
    out["grid"] = bool(np.array_equal(q, q0) and np.array_equal(s, s0.astype(np.float32)))
    rng = np.random.default_rng(3)
    Y = (rng.normal(size=(6, 200)) * 0.7).astype(np.float16)
    q, s = quantize_act(Y)
    err = np.abs(Y.astype(np.float64) - q.astype(np.float64) * s.astype(np.float64)[:, None])
    out["bound"] = bool(np.all(err <= 0.5 * s.astype(np.float64)[:, None] * (1 + 2.0 ** -20)))
    out["range"] = bool(q.min() >= -127 and q.max() <= 127 and np.all(np.abs(q).max(axis=1) == 127))
    qn, sn = quantize_act(-Y)
    out["symmetric"] = bool(np.array_equal(qn, -q) and np.array_equal(sn, s))
    Z = np.zeros((2, 16), dtype=np.float16)
    Z[1, 3] = np.float16(-0.5)
    qz, sz = quantize_act(Z)
    out["zero_row"] = bool(sz[0] == 1.0 and not qz[0].any() and qz[1, 3] == -127)
    # division, not multiplication by the reciprocal: a = 0.50146484375 (fp16
    # bits 0x3803) gives s = fl32(a / 127) = 0.0039485423; x = a / 2 divides to
    # fl32(x / s) = 63.499996 -> 63 (and -63), while x * fl32(1/s) rounds to
    # exactly 63.5 and would give the even 64; 0.125 / s = 31.66 -> 32.
    R = np.array([[0.50146484375, 0.250732421875, -0.250732421875, 0.125]], dtype=np.float16)
    qr, sr = quantize_act(R)
    out["division_not_reciprocal"] = bool(np.array_equal(qr[0], [127, 63, -63, 32])
                                          and sr[0] == np.float32(0.50146484375) / np.float32(127))

    # brute force on a tiny product
    qx = rng.integers(-127, 128, size=(3, 7)).astype(np.int8)
    qw = rng.integers(-127, 128, size=(7, 4)).astype(np.int8)
    sx = rng.uniform(0.01, 1, size=3).astype(np.float32)
    sw = rng.uniform(0.01, 1, size=4).astype(np.float32)
    ref = np.zeros((3, 4))
    for m in range(3):
        for n in range(4):
            acc = 0
            for k in range(7):
                acc += int(qx[m, k]) * int(qw[k, n])
            ref[m, n] = float(sx[m]) * float(sw[n]) * acc
    out["brute"] = bool(np.allclose(gemm(qx, sx, qw, sw), ref, rtol=1e-15, atol=0))
    # hand-worked: qx = [[1, -2, 3], [127, 0, -127]], qw = [[1, 0], [2, -1], [0, 127]], sx = [0.5, 2], sw = [1, 0.25]
    hx = np.array([[1, -2, 3], [127, 0, -127]], dtype=np.int8)
    hw = np.array([[1, 0], [2, -1], [0, 127]], dtype=np.int8)
    hy = gemm(hx, np.array([0.5, 2], np.float32), hw, np.array([1, 0.25], np.float32))
    # row 0: [1 - 4 + 0, 0 + 2 + 381] = [-3, 383] -> * 0.5 * [1, 0.25] = [-1.5, 47.875]
    # row 1: [127, -16129] -> * 2 * [1, 0.25] = [254, -8064.5]
    out["hand"] = bool(np.array_equal(hy, np.array([[-1.5, 47.875], [254.0, -8064.5]])))
    # the integer sum stays exact past 2^24: 1040 * 127^2 + 127 * 24 + 3 * 3 = 2^24 + 1,
    # which binary32 cannot hold
    vx = np.array([127] * 1040 + [127, 3], dtype=np.int8)[None, :]
    vw = np.array([127] * 1040 + [24, 3], dtype=np.int8)[:, None]
    one = np.ones(1, np.float32)
    out["exact_sum"] = bool(gemm(vx, one, vw, one)[0, 0] == 2.0 ** 24 + 1)
    return out


def test_oracle_passes_every_pin():
    res = pins(w8.quantize_act, w8.gemm)
    assert all(res.values()), res


def test_weight_quantiser_is_per_output_channel():
    rng = np.random.default_rng(5)
    W = (rng.normal(size=(40, 6)) * np.array([0.01, 0.1, 1, 10, 0.5, 3])).astype(np.float16)
    q, s = w8.quantize_weight(W)
    qt, st = w8.quantize_act(np.ascontiguousarray(W.T))
    assert q.shape == (40, 6) and s.shape == (6,)
    assert np.array_equal(q, qt.T) and np.array_equal(s, st)
    assert np.all(np.abs(q).max(axis=0) == 127)


def _quant_amax_128(X):
    x = X.astype(np.float32)
    a = np.abs(x).max(axis=1)
    s = np.where(a == 0, np.float32(1), a / np.float32(128)).astype(np.float32)
    return np.clip(np.rint(x / s[:, None]), -127, 127).astype(np.int8), s


def _quant_trunc(X):
    x = X.astype(np.float32)
    a = np.abs(x).max(axis=1)
    s = np.where(a == 0, np.float32(1), a / np.float32(127)).astype(np.float32)
    return np.clip(np.trunc(x * (np.float32(1) / s)[:, None]), -127, 127).astype(np.int8), s


def _quant_no_zero_guard(X):
    x = X.astype(np.float32)
    a = np.abs(x).max(axis=1)
    s = (a / np.float32(127)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.nan_to_num(np.rint(x * (np.float32(1) / s)[:, None]))
    return np.clip(q, -127, 127).astype(np.int8), s


def _quant_reciprocal(X):
    x = X.astype(np.float32)
    a = np.abs(x).max(axis=1)
    s = np.where(a == 0, np.float32(1), a / np.float32(127)).astype(np.float32)
    return np.clip(np.rint(x * (np.float32(1) / s)[:, None]), -127, 127).astype(np.int8), s


def _gemm_transposed(qx, sx, qw, sw, rows=None):
    if qw.shape[0] == qw.shape[1]:
        qw = qw.T
    return w8.gemm(qx, sx, qw, sw, rows)


def _gemm_no_sx(qx, sx, qw, sw, rows=None):
    return w8.gemm(qx, np.ones_like(sx), qw, sw, rows)


def _gemm_float_acc(qx, sx, qw, sw, rows=None):
    acc = qx.astype(np.float32) @ qw.astype(np.float32)
    return sx.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :] * acc.astype(np.float64)


@pytest.mark.parametrize("quantize,gemm", [
    (_quant_amax_128, w8.gemm), (_quant_trunc, w8.gemm), (_quant_no_zero_guard, w8.gemm),
    (_quant_reciprocal, w8.gemm), (w8.quantize_act, _gemm_no_sx), (w8.quantize_act, _gemm_float_acc)],
    ids=["scale_128", "truncation", "zero_row", "reciprocal", "missing_sx", "float32_accumulation"])
def test_pins_reject_planted_mistakes(quantize, gemm):
    res = pins(quantize, gemm)
    assert not all(res.values()), res


def test_transposed_weight_is_caught_by_the_hand_case():
    hx = np.array([[1, -2], [3, 4]], dtype=np.int8)
    hw = np.array([[1, 2], [3, 4]], dtype=np.int8)
    one = np.ones(2, np.float32)
    assert not np.array_equal(_gemm_transposed(hx, one, hw, one), w8.gemm(hx, one, hw, one))
    assert np.array_equal(w8.gemm(hx, one, hw, one), np.array([[-5.0, -6.0], [15.0, 22.0]]))


def test_algorithmic_bytes_llama3_8b_gate_up():
    # int8 weights 4096 x 28672, fp32 per-channel scales, one token
    assert w8.algorithmic_bytes(1, 4096, 28672) == 4096 * 28672 + 4 * 28672 + 4096 + 4 + 2 * 28672
