"""GPU parity of the grouped decode launch (tm_w4a16_gemm_grouped).

Every product of a grouped launch is checked against the fp64 oracle (all
rows; all columns for the small shapes, three column windows of the Llama-3
shapes -- columns of Y are independent, so a window is an exact check of
those columns) and bit for bit against the same product launched on its own
with the same settings (split, CTA width, warp width), which covers every
remaining column."""
import numpy as np
import pytest
import torch

import oracle
import oracle.mlp as mlp
from tests.gpu_util import TOL, activations, host_weights, packed
from w4a16_quantized_gemm_gb300 import binding

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

LLAMA3_8B = [(4096, 6144), (4096, 4096), (4096, 28672), (14336, 4096)]  # qkv, o_proj, gate_up, down


def _xd(X):
    return torch.from_numpy(X.view(np.uint16)).cuda().view(torch.float16)


def _windows(N, width=256):
    if N <= 3 * width:
        return [(0, N)]
    mid = (N // 2) // 16 * 16
    return [(0, width), (mid, mid + width), (N - width, N)]


def _oracle_check(Y, X, K, N, g, silu, cols=None):
    q, z, s, _ = host_weights(K, N, g)
    for c0, c1 in (cols or [(0, N)]):
        ref = oracle.gemm(X, q[:, c0:c1], z[:, c0:c1], s[:, c0:c1], g)
        if silu:
            # output column 4b + i pairs weight columns 8b + i and 8b + 4 + i
            h_ref = mlp.silu_mul(ref)
            got = Y[:, c0 // 2:c1 // 2].float().cpu().numpy().astype(np.float64)
            excess = np.abs(got - h_ref) / mlp.error_bound(ref, TOL)
            assert np.all(np.isfinite(got)) and excess.max() <= 1.0, float(excess.max())
        else:
            got = Y[:, c0:c1].float().cpu().numpy().astype(np.float64)
            assert np.all(np.isfinite(got))
            err = oracle.rel_max_err(got, ref)
            assert err <= TOL, err


def _single_config(cfg, i):
    return {"path": 1, "split_k": cfg["splits"][i], "tile_n": cfg["tile_n"], "warp_n": cfg["warp_n"],
            "stages": cfg["stages"]}


def _run_group(M, shapes, g, silu=None, config=None, check_oracle=True, windows=False):
    silu = silu or [False] * len(shapes)
    ws = [packed(K, N, g) for K, N in shapes]
    Xs = [activations(M, K, N, g) for K, N in shapes]
    Xd = [_xd(X) for X in Xs]
    outs = binding.gemm_grouped([(x, w, None, f) for x, w, f in zip(Xd, ws, silu)], config=config)
    assert binding.last_launch_count() == 1
    torch.cuda.synchronize()
    assert binding.device_error(clear=True) == 0
    cfg = binding.plan_grouped(ws, M, config=config, silu=silu)
    for i, ((K, N), x, w, f, Y, X) in enumerate(zip(shapes, Xd, ws, silu, outs, Xs)):
        single = (binding.gemm_silu_mul if f else binding.gemm)(x, w, config=_single_config(cfg, i))
        torch.cuda.synchronize()
        assert torch.equal(Y, single), (K, N, f)
        if check_oracle:
            _oracle_check(Y, X, K, N, g, f, _windows(N) if windows else None)
    return outs, cfg


@pytest.mark.parametrize("M", [1, 8, 16, 32])
def test_grouped_llama3_8b_layer(M):
    _, cfg = _run_group(M, LLAMA3_8B, 128, windows=True)
    assert cfg["path"] == 1


@pytest.mark.parametrize("M", [1, 16])
def test_grouped_llama3_8b_layer_fused_gate_up(M):
    _run_group(M, LLAMA3_8B, 128, silu=[False, False, True, False], windows=True)


SMALL = [(1024, 2048), (512, 1024), (2048, 512), (256, 64)]


@pytest.mark.parametrize("M", [1, 3, 7, 8, 13, 16, 29, 32])
def test_grouped_small_shapes_auto(M):
    _run_group(M, SMALL, 128, silu=[False, True, False, False])


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("tile_n", [64, 128])
def test_grouped_settings(split, tile_n):
    _run_group(5, SMALL, 128, config={"path": 1, "split_k": split, "tile_n": tile_n})


def test_grouped_ragged_and_empty_slices():
    # N not a multiple of the CTA width; K not a multiple of 2 g (padded);
    # K = g: fewer super-groups than the split, so some CTAs hold no K.
    _run_group(6, [(192, 144), (64, 48), (320, 80)], 64, config={"path": 1, "split_k": 8, "tile_n": 64})
    _run_group(1, [(192, 144), (64, 48)], 64)


def test_grouped_g64():
    _run_group(9, [(4096, 1024), (1024, 4096)], 64)


def test_grouped_one_problem_equals_single():
    _run_group(4, [(4096, 4096)], 128)


def test_grouped_large_m_runs_one_launch_per_product():
    M = 64
    shapes = [(1024, 2048), (2048, 512)]
    ws = [packed(K, N, 128) for K, N in shapes]
    Xs = [activations(M, K, N, 128) for K, N in shapes]
    outs = binding.gemm_grouped([(_xd(X), w, None, False) for X, w in zip(Xs, ws)])
    assert binding.last_launch_count() == 2
    torch.cuda.synchronize()
    for (K, N), X, w, Y in zip(shapes, Xs, ws, outs):
        assert torch.equal(Y, binding.gemm(_xd(X), w))
        _oracle_check(Y, X, K, N, 128, False)


def test_grouped_rejects_overlap_mixed_g_and_count():
    w1 = packed(1024, 2048, 128)
    w2 = packed(1024, 512, 64)
    X = torch.zeros((2, 1024), dtype=torch.float16, device="cuda")
    Y = torch.empty((2, 2048), dtype=torch.float16, device="cuda")
    X1 = Y.view(-1)[:2048].view(2, 1024)  # the first rows of Y, read as the second product's X
    with pytest.raises(binding.TMError) as e:
        binding.gemm_grouped([(X, w1, Y, False), (X1, w1, None, False)])
    assert e.value.status == 1
    big = torch.empty(2 * 2048 + 1024, dtype=torch.float16, device="cuda")
    lib = binding.load()
    arr = (binding.GemmProblem * 2)()
    for i in range(2):  # two outputs 1024 elements apart: overlapping [2][2048] ranges
        arr[i].X = X.data_ptr()
        arr[i].p = w1.handle
        arr[i].Y = big.data_ptr() + i * 2048
        arr[i].silu = 0
    assert lib.tm_w4a16_gemm_grouped(arr, 2, 2, None, None) == 1
    with pytest.raises(binding.TMError) as e:  # mixed group sizes
        binding.gemm_grouped([(X, w1, None, False), (X, w2, None, False)])
    assert e.value.status == 1
    with pytest.raises(binding.TMError) as e:  # more than TM_GROUP_MAX products
        binding.gemm_grouped([(X, w1, None, False)] * (binding.GROUP_MAX + 1))
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert binding.device_error(clear=True) == 0
