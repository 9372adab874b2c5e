"""GPU parity of the tensor-memory kernel (path 3: W^T dequantised into tensor
memory, tcgen05 with the A operand in TMEM) against the fp64 oracle, through
the C ABI.  Same bar as the other paths: max|Y - Y_ref| / max|Y_ref| <= 2e-3."""
import numpy as np
import pytest
import torch

from tests.gpu_util import TOL, activations, packed, run_and_compare
from w4a16_quantized_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

TC = {"path": 3}


def _cases(idx):
    return [pytest.param(c, id=c.name) for c in synth.workload(idx)]


@pytest.mark.parametrize("case", _cases(0) + _cases(1) + _cases(2))
def test_tc_llama3_8b_workloads(case):
    err, _ = run_and_compare(case.M, case.K, case.N, case.g, case.stress, config=TC)
    assert err <= TOL, err


@pytest.mark.parametrize("case", _cases(3) + _cases(4))
def test_tc_llama70b_and_stress_workloads(case):
    err, _ = run_and_compare(case.M, case.K, case.N, case.g, case.stress, config=TC)
    assert err <= TOL, err


@pytest.mark.parametrize("M", [1, 7, 15, 16, 17, 31, 33, 63, 64, 65, 127, 129, 200, 255, 257, 300])
def test_tc_ragged_m(M):
    err, _ = run_and_compare(M, 1024, 384, 128, config=TC)
    assert err <= TOL, err


@pytest.mark.parametrize("tile_m", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("M", [5, 40, 130])
def test_tc_tile_m_override(tile_m, M):
    """Every row tile, with M below, inside and above one tile; N = 272 leaves
    a CTA with one of its eight n-tiles."""
    err, _ = run_and_compare(M, 1024, 272, 128, config={"path": 3, "tile_m": tile_m})
    assert err <= TOL, err


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("K,tile_m", [(256, 16), (256, 128), (1024, 32), (2048, 256)])
def test_tc_split_override(split, K, tile_m):
    """Split K over a cluster; with K = 256 (4 k-blocks) and 8 CTAs some get none."""
    err, _ = run_and_compare(48, K, 512, 128, config={"path": 3, "split_k": split, "tile_m": tile_m})
    assert err <= TOL, err


@pytest.mark.parametrize("stages", [2, 3, 7, 12])
def test_tc_stage_override(stages):
    err, _ = run_and_compare(24, 4096, 1024, 64, config={"path": 3, "stages": stages})
    assert err <= TOL, err


@pytest.mark.parametrize("K,N,g", [(128, 16, 128), (64, 16, 64), (192, 48, 64), (640, 272, 128), (896, 4112, 64)])
def test_tc_small_and_ragged_shapes(K, N, g):
    """K = g (one group, odd group count), one n-tile, N not a multiple of 128."""
    for M in (3, 70):
        err, _ = run_and_compare(M, K, N, g, config=TC)
        assert err <= TOL, (M, err)


def test_tc_plan_fields():
    w = packed(4096, 4096, 128)
    # 32 column tiles: row tiles above 64 are halved while fewer than half the SMs get a tile
    for M, bt in ((1, 16), (16, 16), (17, 32), (64, 64), (65, 64), (128, 64), (129, 64), (4096, 256)):
        c = binding.plan(w, M, TC)
        assert c["path"] == 3 and c["tile_m"] == bt and c["tile_n"] == 128
        assert c["split_k"] in (1, 2, 4, 8) and 2 <= c["stages"] <= 16
    with pytest.raises(binding.TMError):
        binding.plan(w, 8, {"path": 3, "tile_m": 48})
    with pytest.raises(binding.TMError):
        binding.plan(w, 8, {"path": 3, "tile_n": 256})


def test_tc_deterministic_bits():
    for cfg in ({"path": 3, "split_k": 4, "tile_m": 32}, {"path": 3, "tile_m": 256}):
        M = 24 if cfg["tile_m"] == 32 else 300
        w = packed(4096, 1024, 128)
        X = torch.from_numpy(activations(M, 4096, 1024, 128).view(np.uint16)).cuda().view(torch.float16)
        Y1 = binding.gemm(X, w, config=cfg).clone()
        Y2 = binding.gemm(X, w, config=cfg).clone()
        torch.cuda.synchronize()
        assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))


def test_tc_one_launch_and_no_device_errors():
    w = packed(1024, 384, 128)
    X = torch.zeros((40, 1024), dtype=torch.float16, device="cuda")
    binding.gemm(X, w, config=TC)
    assert binding.last_launch_count() == 1
    torch.cuda.synchronize()
    assert binding.device_error(clear=False) == 0


# More output tiles (128 columns x tile_m rows) than a GB300 has SMs (152),
# so that later waves of CTAs (one per SM: each holds all of tensor memory)
# reuse the SMs, with a ragged last row tile and a ragged last column tile;
# every row compared.
@pytest.mark.parametrize("M,K,N,g,tile_m", [(2049, 256, 4112, 128, 256), (1100, 128, 2320, 64, 64),
                                             (333, 64, 8208, 64, 16)])
def test_tc_multi_wave_tiles_every_row(M, K, N, g, tile_m):
    cfg = {"path": 3, "split_k": 1, "tile_m": tile_m}
    tiles = -(-N // 128) * -(-M // tile_m)
    assert tiles > 152
    err, _ = run_and_compare(M, K, N, g, config=cfg, rows=list(range(M)))
    assert err <= TOL, err


def test_tc_split_and_unsplit_launches_agree():
    # the same product without a K split (several waves) and with a split of 2
    # (clusters reducing through distributed shared memory) agrees to the
    # parity bar on every element
    M, K, N, g = 700, 512, 6144, 128
    w = packed(K, N, g)
    X = torch.from_numpy(activations(M, K, N, g).view(np.uint16)).cuda().view(torch.float16)
    Y1 = binding.gemm(X, w, config={"path": 3, "split_k": 1, "tile_m": 128}).float()
    Y2 = binding.gemm(X, w, config={"path": 3, "split_k": 2, "tile_m": 128}).float()
    torch.cuda.synchronize()
    assert binding.device_error(clear=True) == 0
    assert ((Y1 - Y2).abs().max() / Y2.abs().max()).item() <= TOL
