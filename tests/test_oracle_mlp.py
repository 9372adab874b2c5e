"""Pins of the fused gate/up epilogue oracle (oracle/mlp.py): SiLU closed forms
and identities, the column pairing on a hand-worked layout, and planted
mistakes that the pins must reject."""
import math

import numpy as np
import pytest

import oracle.mlp as mlp


def pins(silu, silu_mul):
    out = {}
    x = np.linspace(-30, 30, 601)
    out["silu_zero"] = silu(np.array([0.0]))[0] == 0.0
    out["silu_one"] = abs(silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    # silu(x) - silu(-x) = x for every x (sigmoid(x) + sigmoid(-x) = 1)
    out["odd_identity"] = bool(np.allclose(silu(x) - silu(-x), x, rtol=0, atol=1e-12))
    out["limits"] = bool(abs(silu(np.array([40.0]))[0] - 40.0) < 1e-12 and abs(silu(np.array([-40.0]))[0]) < 1e-15)
    # the derivative's maximum, used by the error bound: about 1.0998 near x = 2.3994
    d = np.gradient(silu(x), x)
    out["derivative_max"] = bool(1.09 < d.max() < 1.1)
    # pairing on N = 16: h[:, j] = silu(Y[:, c]) * Y[:, c + 4], c = 0,1,2,3,8,9,10,11
    Y = np.zeros((1, 16))
    Y[0, :] = np.arange(16)
    h = silu_mul(Y)
    gate = np.array([0, 1, 2, 3, 8, 9, 10, 11], dtype=np.float64)
    up = gate + 4
    out["pairing"] = bool(h.shape == (1, 8) and np.allclose(h[0], [silu(np.array([a]))[0] * b for a, b in zip(gate, up)]))
    return out


def test_oracle_passes_every_pin():
    res = pins(mlp.silu, mlp.silu_mul)
    assert all(res.values()), res


def _silu_sign(x):
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(x))


def _pair_offset2(Y):
    j = np.arange(Y.shape[1] // 2)
    c = 4 * (j // 2) + (j % 2)
    return mlp.silu(Y[:, c]) * Y[:, c + 2]


def _swapped(Y):
    c = mlp.gate_columns(Y.shape[1])
    return mlp.silu(Y[:, c + 4]) * Y[:, c]


@pytest.mark.parametrize("silu,silu_mul", [(_silu_sign, lambda Y: _silu_sign(Y[:, mlp.gate_columns(Y.shape[1])])
                                            * Y[:, mlp.gate_columns(Y.shape[1]) + 4]),
                                           (mlp.silu, _pair_offset2), (mlp.silu, _swapped)],
                         ids=["sigmoid_sign", "pair_offset_2", "gate_up_swapped"])
def test_pins_reject_planted_mistakes(silu, silu_mul):
    res = pins(silu, silu_mul)
    assert not all(res.values()), res


def test_error_bound_is_tight_enough():
    """A 1e-3 relative perturbation of Y stays inside the bound built from 2e-3."""
    rng = np.random.default_rng(0)
    Y = rng.normal(size=(4, 64)) * 3
    Yp = Y + 1e-3 * np.max(np.abs(Y)) * rng.uniform(-1, 1, size=Y.shape)
    dh = np.abs(mlp.silu_mul(Yp) - mlp.silu_mul(Y))
    assert np.all(dh <= mlp.error_bound(Y, 2e-3))
