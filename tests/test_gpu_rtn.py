"""GPU parity of the round-to-nearest INT4 quantiser (tm_quantize_rtn) against
the binary32 oracle (oracle/rtn.py): codes, zeros and scales bit-exact, then
the whole pipeline quantise -> pack -> GEMM against the fp64 GEMM oracle on the
oracle's own codes."""
import numpy as np
import pytest
import torch

import oracle
import oracle.rtn as rtn
from tests.gpu_util import TOL
from w4a16_quantized_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _gpu_quantize(W16, g):
    Wd = torch.from_numpy(W16.view(np.uint16)).cuda().view(torch.float16)
    q, z, s = binding.quantize_rtn(Wd, g)
    torch.cuda.synchronize()
    return q.cpu().numpy(), z.cpu().numpy(), s.cpu().numpy().view(np.uint16)


def _assert_bit_exact(W16, g):
    q, z, s = _gpu_quantize(W16, g)
    assert binding.device_error(clear=True) == 0
    q0, z0, s0 = rtn.quantize(W16, g)
    assert np.array_equal(s, s0.view(np.uint16))
    assert np.array_equal(z, z0)
    assert np.array_equal(q, q0)


@pytest.mark.parametrize("K,N,g", [(4096, 4096, 128), (4096, 6144, 128), (14336, 4096, 128), (4096, 28672, 128),
                                   (4096, 28672, 64), (192, 48, 64), (128, 16, 128), (256, 272, 32), (512, 64, 256)])
def test_rtn_bit_exact(K, N, g):
    _assert_bit_exact(synth.fp16_weights(K, N, g), g)


def test_rtn_special_values_bit_exact():
    """Ties, degenerate groups, subnormal and largest fp16 magnitudes, signed zeros."""
    T = np.array([-7.5, 7.5, 2.5, 3.5, -0.5, -6.5, 0.0, 1.0], dtype=np.float16)
    cols = [np.repeat(T, 2), np.zeros(16, np.float16), np.full(16, 0.75, np.float16),
            np.full(16, -0.375, np.float16), np.array([6e-8, -6e-8] * 8, np.float16),
            np.array([65504, -65504] + [1.0] * 14, np.float16), np.array([-0.0, 0.0] * 8, np.float16),
            np.linspace(-3, 5, 16).astype(np.float16)]
    W = np.stack(cols + cols, axis=1)  # 16 columns
    _assert_bit_exact(np.ascontiguousarray(W), 16)
    _assert_bit_exact(np.ascontiguousarray(W), 8)
    # the same columns through the tiled kernel of g = 64 and g = 128 (tiles
    # of 128 columns: these 16 are a ragged, zero-filled tile)
    _assert_bit_exact(np.ascontiguousarray(np.tile(W, (4, 1))), 64)
    _assert_bit_exact(np.ascontiguousarray(np.tile(W, (8, 1))), 128)


@pytest.mark.parametrize("K,N,g", [(8192, 4112, 64), (2048, 2064, 128), (128, 144, 128)])
def test_rtn_tiled_ragged_columns_bit_exact(K, N, g):
    # N not a multiple of the 128-column tile; the first shape has more tiles
    # (33 x 128) than two CTAs per SM take at once, so CTAs walk several
    _assert_bit_exact(synth.fp16_weights(K, N, g), g)


def test_rtn_quantize_pack_gemm_pipeline():
    K, N, g, M = 4096, 1024, 128, 8
    W16 = synth.fp16_weights(K, N, g)
    Wd = torch.from_numpy(W16.view(np.uint16)).cuda().view(torch.float16)
    q, z, s = binding.quantize_rtn(Wd, g)
    w = binding.pack(q, z, s, g)
    X = synth.activations(M, K, tag="/rtn")
    Xd = torch.from_numpy(X.view(np.uint16)).cuda().view(torch.float16)
    Y = binding.gemm(Xd, w).float().cpu().numpy().astype(np.float64)
    q0, z0, s0 = rtn.quantize(W16, g)
    Y_ref = oracle.gemm(X, q0, z0, s0, g)
    assert oracle.rel_max_err(Y, Y_ref) <= TOL
    assert binding.device_error() == 0


def test_rtn_rejects_bad_arguments():
    W = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(binding.TMError) as e:
        binding.quantize_rtn(W, 96)          # K % g
    assert e.value.status == 1
    with pytest.raises(binding.TMError) as e:
        binding.quantize_rtn(W[:, :40], 64)  # N % 16 (non-contiguous slice is copied first)
    assert e.value.status == 1


def test_rtn_one_launch():
    W = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    binding.quantize_rtn(W, 64)
    assert binding.last_launch_count() == 1
    torch.cuda.synchronize()


def tie_columns(B, rows, first=0x1C00, count=4096):
    """Columns that each hold, for one fp16 scale s (s = hi / B exactly, hi an
    fp16 value), the group maximum hi and every exact tie (k + 1/2) s that is
    itself an fp16 value; the remaining rows are zeros.  Built on the host from
    fp16 bit patterns: the quotient of every tie by s is exactly a half-integer,
    the case where a multiply by the reciprocal 1/s can round to the wrong
    neighbour."""
    cols = []
    for bits in range(first, first + 8 * count):
        s = np.array([bits], dtype=np.uint16).view(np.float16)[0]
        hi = np.float16(B * float(s))
        if float(hi) != B * float(s) or not np.isfinite(hi):
            continue
        if np.float16(np.float32(hi) / np.float32(B)) != s:
            continue
        ties = [np.float16((k + 0.5) * float(s)) for k in range(B)]
        ties = [t for k, t in enumerate(ties) if float(t) == (k + 0.5) * float(s)]
        col = np.zeros(rows, dtype=np.float16)
        vals = [hi] + ties[: rows - 1]
        col[: len(vals)] = vals
        cols.append(col)
        if len(cols) == count:
            break
    cols = cols[: len(cols) // 16 * 16]  # N % 16 == 0
    return np.ascontiguousarray(np.stack(cols, axis=1))


@pytest.mark.parametrize("g", [16, 64, 128])
def test_rtn_exact_ties_bit_exact(g):
    """Exact ties w = (k + 1/2) s over a few thousand scales, through the
    generic (g = 16) and the tiled (g = 64, 128) kernels: the codes equal the
    division rule's, and the set is one where a plain multiply by fl(1/s)
    would differ (checked on the host with that rule)."""
    W = tie_columns(15, g, count=2048)
    _assert_bit_exact(W, g)
    w = W.astype(np.float32)
    _, _, s0 = rtn.quantize(W, g)
    recip = np.rint(w * (np.float32(1) / s0.astype(np.float32)))
    assert np.count_nonzero(recip != np.rint(w / s0.astype(np.float32))) > 0
