"""GPU parity of the fused gate/up epilogue (tm_w4a16_gemm_silu_mul) against the
fp64 oracle: every element of H within the bound that the GEMM's own parity bar
(2e-3 of max|Y|) implies through h = silu(gate) * up plus one fp16 rounding
(oracle/mlp.py: error_bound)."""
import numpy as np
import pytest
import torch

import oracle
import oracle.mlp as mlp
from tests.gpu_util import TOL, activations, host_weights, packed, sample_rows
from w4a16_quantized_gemm_gb300 import binding

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _check(M, K, N, g, config=None):
    w = packed(K, N, g)
    X = activations(M, K, N, g)
    Xd = torch.from_numpy(X.view(np.uint16)).cuda().view(torch.float16)
    H = binding.gemm_silu_mul(Xd, w, config=config)
    torch.cuda.synchronize()
    assert binding.device_error(clear=True) == 0
    rows = sample_rows(M)
    q, z, s, _ = host_weights(K, N, g)
    Y_ref = oracle.gemm(X, q, z, s, g, rows=rows)
    h_ref = mlp.silu_mul(Y_ref)
    Hh = H[torch.tensor(rows, device=H.device)].float().cpu().numpy().astype(np.float64)
    assert Hh.shape == h_ref.shape
    bound = mlp.error_bound(Y_ref, TOL)
    excess = np.abs(Hh - h_ref) / bound
    assert np.all(np.isfinite(Hh)) and excess.max() <= 1.0, float(excess.max())


@pytest.mark.parametrize("M", [1, 5, 8, 16, 17, 32, 33, 64, 128, 300])
def test_silu_mul_auto_path(M):
    _check(M, 1024, 2048, 128)


@pytest.mark.parametrize("M", [1, 16])
def test_silu_mul_llama3_8b_gate_up(M):
    _check(M, 4096, 28672, 128)


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("tile_n", [64, 128, 256])
def test_silu_mul_decode_overrides(split, tile_n):
    _check(8, 2048, 512, 128, {"path": 1, "split_k": split, "tile_n": tile_n})


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("tile_m", [16, 64, 256])
def test_silu_mul_tc_overrides(split, tile_m):
    _check(40, 2048, 512, 64, {"path": 3, "split_k": split, "tile_m": tile_m})


def test_silu_mul_ragged_n():
    """N = 272 (17 n-tiles): the last CTA holds a partial tile of pairs."""
    for cfg in ({"path": 1}, {"path": 3}):
        _check(6, 640, 272, 128, cfg)


def test_silu_mul_prefill_path_unsupported():
    w = packed(1024, 2048, 128)
    X = torch.zeros((256, 1024), dtype=torch.float16, device="cuda")
    with pytest.raises(binding.TMError) as e:
        binding.gemm_silu_mul(X, w, config={"path": 2})
    assert e.value.status == 3


def test_silu_mul_tc_multi_wave_tiles():
    # more output tiles than SMs: the later waves carry the fused epilogue too
    # (the sampled rows include the ragged last row tile)
    _check(1500, 256, 8192, 128, {"path": 3, "split_k": 1, "tile_m": 128})
