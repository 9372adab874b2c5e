"""tm_w4a16_gemm_host_static through the C ABI: the host-buffer product staged
through the library's fixed device array, for callers that cannot allocate
device memory (a plug-in whose host application already holds the device's
memory in its own pool, or a latency-critical loop where cudaMalloc/cudaFree
may block).  Its results must match the allocating entry point on the same
inputs, on consecutive calls that reuse the one array.

This file is named to be collected last, so that a run stopping at its first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import TOL, activations, packed
from w4a16_quantized_gemm_gb300 import binding

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _host(X):
    return torch.from_numpy(X.view(np.uint16)).view(torch.float16).pin_memory()


def _existing(Xh, w):
    """The allocating host-buffer call (caller-provided staging buffers)."""
    return binding.gemm_host(Xh, w)


def _rel(a, b):
    return oracle.rel_max_err(a.float().numpy().astype(np.float64), b.float().numpy().astype(np.float64))


def test_static_staging_matches_the_allocating_call_on_two_calls_in_a_row():
    # Two different problems back to back: the second call must overwrite the
    # first call's X and Y in the shared array.
    cases = [(8, 4096, 4096, 128), (32, 14336, 4096, 128)]
    for M, K, N, g in cases:
        w = packed(K, N, g)
        Xh = _host(activations(M, K, N, g))
        ref = _existing(Xh, w)
        got = binding.gemm_host_static(Xh, w)
        assert binding.device_error(clear=True) == 0
        assert torch.all(torch.isfinite(got.float()))
        assert _rel(got, ref) <= TOL
    # The same problem again with other activations: no stale result survives.
    M, K, N, g = cases[0]
    w = packed(K, N, g)
    X2 = _host(activations(M, K, N, g, seed=1))
    ref2 = _existing(X2, w)
    got2 = binding.gemm_host_static(X2, w)
    assert _rel(got2, ref2) <= TOL
    assert binding.device_error(clear=True) == 0


def test_static_staging_rejects_requests_beyond_its_size():
    K, N, g = 4096, 4096, 128
    w = packed(K, N, g)
    # 2 M K rounded to 256 plus 2 M N must fit TM_STATIC_STAGING_BYTES (8 MiB).
    M = binding.STATIC_STAGING_BYTES // (2 * (K + N)) + 1
    X = torch.zeros((M, K), dtype=torch.float16)
    Y = torch.full((M, N), 7.0, dtype=torch.float16)
    st = binding.load().tm_w4a16_gemm_host_static(X.data_ptr(), w.handle, Y.data_ptr(), M, None,
                                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 7  # TM_ERR_SCRATCH_LIMIT
    assert binding.status_str(st) == "request exceeds the static staging array"
    assert bool(torch.all(Y == 7.0))  # nothing was copied back
    # the largest M that fits still runs
    M_fit = binding.STATIC_STAGING_BYTES // (2 * (K + N)) - 1
    Xf = _host(activations(M_fit, K, N, g))
    assert _rel(binding.gemm_host_static(Xf, w), _existing(Xf, w)) <= TOL
