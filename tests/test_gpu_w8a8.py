"""GPU parity of the W8A8 path (tm_w8a8_quantize_act, tm_w8_pack, tm_w8a8_gemm)
against the oracle (oracle/w8a8.py): the quantiser and the packing bit-exact;
the GEMM within max|Y - Y_ref| / max|Y_ref| <= 2e-3 -- and, tighter, each
element within one fp16 rounding of its exact value: the products are exact
fp16 integers, the fp32 sums exact below 2^24, so what is left is the fp32
scaling and the final rounding to fp16 (2^-11 relative)."""
import functools

import numpy as np
import pytest
import torch

import oracle
import oracle.w8a8 as w8
from tests.gpu_util import TOL, sample_rows
from w4a16_quantized_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _fp16(tag, rows, cols, scale=1.0):
    return (synth.normal64(tag, rows, cols) * scale).astype(np.float16)


@functools.lru_cache(maxsize=6)
def _weights(K, N):
    W = _fp16(f"w8/W/{K}/{N}", K, N, 0.05)
    W[:, 0] = 0                       # an all-zero channel (s_w = 1)
    q, s = w8.quantize_weight(W)
    return q, s


@functools.lru_cache(maxsize=6)
def _packed(K, N):
    q, s = _weights(K, N)
    return binding.pack_w8(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda())


def _acts(M, K, tag="x"):
    X = _fp16(f"w8/X/{tag}/{M}/{K}", M, K)
    if M > 2:
        X[1] = 0                       # an all-zero token (s_x = 1)
        X[2, K // 3] = np.float16(300.0)  # an outlier token
    return X


def _check(M, K, N, split=0, rows=None, tile_m=0):
    q, s = _weights(K, N)
    X = _acts(M, K)
    qx, sx = w8.quantize_act(X)
    Y = binding.w8a8_gemm(torch.from_numpy(qx).cuda(), torch.from_numpy(sx).cuda(), _packed(K, N), split=split,
                          tile_m=tile_m)
    torch.cuda.synchronize()
    assert binding.device_error(clear=True) == 0
    rows = sample_rows(M) if rows is None else rows
    ref = w8.gemm(qx, sx, q, s, rows=rows)
    got = Y[torch.tensor(rows, device=Y.device)].float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    err = oracle.rel_max_err(got, ref)
    assert err <= TOL, err
    # one fp16 rounding of the exact value (plus the fp32 scaling and, past 2^24, the fp32 sums)
    bound = np.abs(ref) * (2.0 ** -11 + 2.0 ** -20) + 2.0 ** -24 + 2.0 ** -22 * np.abs(ref).max()
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))


@pytest.mark.parametrize("M", [1, 2, 16, 33, 300])
@pytest.mark.parametrize("K", [16, 1040, 4096])
def test_quantize_act_bit_exact(M, K):
    X = _acts(M, K, tag="q")
    xq, sx = binding.w8a8_quantize_act(torch.from_numpy(X.view(np.uint16)).cuda().view(torch.float16))
    torch.cuda.synchronize()
    q0, s0 = w8.quantize_act(X)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), s0.view(np.uint32))
    assert np.array_equal(xq.cpu().numpy(), q0)


def near_tie_rows(count=1024, first=0x3400):
    """Rows whose maximum a runs over consecutive fp16 values, holding the fp16
    values nearest to +-(k + 1/2) s for s = fl32(a / 127), k = 0..126: quotients
    at or within a few ulps of a half-integer, where a multiply by fl32(1/s)
    rounds some codes differently from the division."""
    rows = []
    for bits in range(first, first + count):
        a = np.array([bits], dtype=np.uint16).view(np.float16)[0]
        s = np.float32(a) / np.float32(127)
        v = [a] + [np.float16((k + 0.5) * float(s)) for k in range(127)]
        rows.append(np.array(v + [-x for x in v[1:]] + [np.float16(0)], dtype=np.float16))
    return np.stack(rows)


def test_quantize_act_near_ties_bit_exact():
    X = near_tie_rows()
    for f16 in (False, True):
        quant = binding.w8a8_quantize_act_f16 if f16 else binding.w8a8_quantize_act
        xq, sx = quant(torch.from_numpy(X.view(np.uint16)).cuda().view(torch.float16))
        torch.cuda.synchronize()
        q0, s0 = w8.quantize_act(X)
        got = xq.cpu().numpy().astype(np.float32).astype(np.int8) if f16 else xq.cpu().numpy()
        assert np.array_equal(sx.cpu().numpy().view(np.uint32), s0.view(np.uint32))
        assert np.array_equal(got, q0)
    x = X.astype(np.float32)
    recip = np.clip(np.rint(x * (np.float32(1) / s0)[:, None]), -127, 127)
    assert np.count_nonzero(recip != q0) > 0  # the set separates the two rules


def test_quantize_weight_near_ties_bit_exact():
    W = np.ascontiguousarray(near_tie_rows(count=512).T)  # [K = 256][N = 512]: one channel per row above
    q, sw = binding.w8_quantize_weight(torch.from_numpy(W.view(np.uint16)).cuda().view(torch.float16))
    torch.cuda.synchronize()
    q0, s0 = w8.quantize_weight(W)
    assert np.array_equal(sw.cpu().numpy().view(np.uint32), s0.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q0)


@pytest.mark.parametrize("K,N", [(1040, 272), (4096, 512), (128, 16)])
def test_pack_roundtrip(K, N):
    q, s = _weights(K, N)
    qd, sd = _packed(K, N).unpack()
    torch.cuda.synchronize()
    assert np.array_equal(qd.cpu().numpy(), q)
    assert np.array_equal(sd.cpu().numpy().view(np.uint32), s.view(np.uint32))


@pytest.mark.parametrize("M", [1, 3, 8, 9, 16, 17, 32, 33, 64, 65, 130, 300])
def test_gemm_auto(M):
    """M <= 32: the mma.sync kernel; above: the tensor-memory kernel (64- or 128-row tiles)."""
    _check(M, 1024, 512)


@pytest.mark.parametrize("tile_m", [64, 128, 256])
@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("M", [40, 129, 300])
def test_gemm_tensor_memory_tiles_split_ragged(tile_m, split, M):
    """Every row tile and cluster split of the tensor-memory kernel on a partial
    last 128-k block (K = 1040), a partial 128-column block (N = 272) and a
    partial row tile."""
    _check(M, 1040, 272, split=split, tile_m=tile_m)


def test_gemm_ragged_k_and_n():
    """K = 1040 (not a multiple of the 128-k block), N = 272 (17 n-tiles)."""
    for M in (1, 12, 40):
        _check(M, 1040, 272)


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("M", [1, 16, 32, 100])
def test_gemm_split_override(split, M):
    _check(M, 2048, 512, split=split)


@pytest.mark.parametrize("shape", ["qkv", "o_proj", "gate_up", "down"])
@pytest.mark.parametrize("M", [1, 32])
def test_gemm_llama3_8b_decode(shape, M):
    K, N = synth.LLAMA3_8B[shape]
    _check(M, K, N, rows=[0] if M == 1 else [0, 7, 16, 31])


def test_gemm_llama3_8b_prefill_sampled_rows():
    K, N = synth.LLAMA3_8B["o_proj"]
    _check(1024, K, N)


def test_quantize_then_gemm_pipeline():
    """GPU quantiser output fed to the GPU GEMM equals the oracle pipeline."""
    K, N, M = 2048, 512, 24
    q, s = _weights(K, N)
    X = _acts(M, K, tag="pipe")
    xq, sx = binding.w8a8_quantize_act(torch.from_numpy(X.view(np.uint16)).cuda().view(torch.float16))
    Y = binding.w8a8_gemm(xq, sx, _packed(K, N))
    torch.cuda.synchronize()
    q0, s0 = w8.quantize_act(X)
    ref = w8.gemm(q0, s0, q, s)
    assert oracle.rel_max_err(Y.float().cpu().numpy().astype(np.float64), ref) <= TOL


def test_rejects_bad_arguments():
    w = _packed(1024, 512)
    xq = torch.zeros((4, 1024), dtype=torch.int8, device="cuda")
    sx = torch.ones(4, dtype=torch.float32, device="cuda")
    with pytest.raises(binding.TMError) as e:
        binding.w8a8_gemm(xq, sx, w, split=3)
    assert e.value.status == 1
    buf = torch.zeros(4 * 1024 + 16, dtype=torch.int8, device="cuda")
    with pytest.raises(binding.TMError) as e:
        binding.w8a8_gemm(buf[8:8 + 4 * 1024].view(4, 1024), sx, w)
    assert e.value.status == 2
    with pytest.raises(binding.TMError) as e:
        binding.pack_w8(torch.zeros((1000, 512), dtype=torch.int8, device="cuda"),
                        torch.ones(512, dtype=torch.float32, device="cuda"))
    assert e.value.status == 1


@pytest.mark.parametrize("K,N", [(1024, 512), (1040, 272), (4096, 16), (600, 4096)])
def test_quantize_weight_bit_exact(K, N):
    """The GPU per-channel weight quantiser equals the binary32 oracle bit for bit
    (K slices of 512 rows combined by the integer atomic max; a zero column)."""
    W = _fp16(f"w8/Wq/{K}/{N}", K, N, 0.05)
    W[:, 1] = 0
    W[3, 2] = np.float16(-7.5)          # a column whose maximum magnitude is negative
    q, sw = binding.w8_quantize_weight(torch.from_numpy(W.view(np.uint16)).cuda().view(torch.float16))
    torch.cuda.synchronize()
    q0, s0 = w8.quantize_weight(W)
    assert np.array_equal(sw.cpu().numpy().view(np.uint32), s0.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q0)


def test_gpu_quantisers_pack_gemm_pipeline():
    """fp16 W and X through the GPU quantisers, the packer and the GEMM equal the
    oracle pipeline."""
    K, N, M = 2048, 1024, 7
    W = _fp16("w8/pipeW", K, N, 0.05)
    X = _acts(M, K, tag="pipeW")
    q, sw = binding.w8_quantize_weight(torch.from_numpy(W.view(np.uint16)).cuda().view(torch.float16))
    xq, sx = binding.w8a8_quantize_act(torch.from_numpy(X.view(np.uint16)).cuda().view(torch.float16))
    Y = binding.w8a8_gemm(xq, sx, binding.pack_w8(q, sw))
    torch.cuda.synchronize()
    q0, s0 = w8.quantize_weight(W)
    qx0, sx0 = w8.quantize_act(X)
    ref = w8.gemm(qx0, sx0, q0, s0)
    assert oracle.rel_max_err(Y.float().cpu().numpy().astype(np.float64), ref) <= TOL


# ---- the codes as fp16 integers (tm_w8a8_quantize_act_f16, tm_w8a8_gemm_f16) ----

@pytest.mark.parametrize("M", [1, 33, 300])
@pytest.mark.parametrize("K", [16, 1040, 4096])
def test_quantize_act_f16_bit_exact(M, K):
    """The fp16 codes are the oracle's integer codes exactly, the scales bit for bit."""
    X = _acts(M, K, tag="q16")
    xq16, sx = binding.w8a8_quantize_act_f16(torch.from_numpy(X.view(np.uint16)).cuda().view(torch.float16))
    torch.cuda.synchronize()
    q0, s0 = w8.quantize_act(X)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), s0.view(np.uint32))
    codes = xq16.float().cpu().numpy()
    assert np.array_equal(codes, q0.astype(np.float32))


def _check_f16(M, K, N, split=0, tile_m=0, rows=None):
    q, s = _weights(K, N)
    X = _acts(M, K)
    qx, sx = w8.quantize_act(X)
    xq16 = torch.from_numpy(qx.astype(np.float16)).cuda()
    sxd = torch.from_numpy(sx).cuda()
    Y = binding.w8a8_gemm_f16(xq16, sxd, _packed(K, N), split=split, tile_m=tile_m)
    torch.cuda.synchronize()
    assert binding.device_error(clear=True) == 0
    rows = sample_rows(M) if rows is None else rows
    ref = w8.gemm(qx, sx, q, s, rows=rows)
    got = Y[torch.tensor(rows, device=Y.device)].float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    bound = np.abs(ref) * (2.0 ** -11 + 2.0 ** -20) + 2.0 ** -24 + 2.0 ** -22 * np.abs(ref).max()
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))
    return Y, torch.from_numpy(qx).cuda(), sxd


@pytest.mark.parametrize("tile_m", [64, 128, 256])
@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("M", [40, 129, 300])
def test_gemm_f16_tiles_split_ragged_equal_to_int8_path(tile_m, split, M):
    """Every row tile and split on a partial last 128-k block, a partial
    128-column block and a partial row tile: within the bound of the oracle,
    and bit for bit the int8 path's result (same products, same order)."""
    Y16, xq, sx = _check_f16(M, 1040, 272, split=split, tile_m=tile_m)
    Y8 = binding.w8a8_gemm(xq, sx, _packed(1040, 272), split=split, tile_m=tile_m)
    torch.cuda.synchronize()
    assert torch.equal(Y16.view(torch.int16), Y8.view(torch.int16))


@pytest.mark.parametrize("M", [1, 7, 32, 33, 1024])
def test_gemm_f16_auto(M):
    """Small M too (the tensor-memory kernel with 64-row tiles)."""
    _check_f16(M, 2048, 1024)


def test_gemm_f16_llama3_8b_prefill_sampled_rows():
    K, N = synth.LLAMA3_8B["gate_up"]
    _check_f16(4096, K, N, rows=[0, 1, 2, 255, 256, 2047, 4095])


def test_f16_pipeline_gpu_quantiser():
    K, N, M = 2048, 512, 200
    q, s = _weights(K, N)
    X = _acts(M, K, tag="pipe16")
    xq16, sx = binding.w8a8_quantize_act_f16(torch.from_numpy(X.view(np.uint16)).cuda().view(torch.float16))
    Y = binding.w8a8_gemm_f16(xq16, sx, _packed(K, N))
    torch.cuda.synchronize()
    q0, s0 = w8.quantize_act(X)
    ref = w8.gemm(q0, s0, q, s)
    assert oracle.rel_max_err(Y.float().cpu().numpy().astype(np.float64), ref) <= TOL


def test_f16_rejects_bad_arguments():
    w = _packed(1024, 512)
    xq = torch.zeros((40, 1024), dtype=torch.float16, device="cuda")
    sx = torch.ones(40, dtype=torch.float32, device="cuda")
    with pytest.raises(binding.TMError) as e:
        binding.w8a8_gemm_f16(xq, sx, w, tile_m=96)
    assert e.value.status == 1
    buf = torch.zeros(40 * 1024 + 16, dtype=torch.float16, device="cuda")
    with pytest.raises(binding.TMError) as e:
        binding.w8a8_gemm_f16(buf[4:4 + 40 * 1024].view(40, 1024), sx, w)
    assert e.value.status == 2
    with pytest.raises(binding.TMError) as e:
        binding.w8a8_quantize_act_f16(torch.zeros((4, 1000), dtype=torch.float16, device="cuda"))
    assert e.value.status == 1
