"""GPU parity: the CUDA path against the fp64 oracle, through the C ABI.

Bar: pack -> unpack bit-exact; GEMM max|Y - Y_ref| / max|Y_ref| <= 2e-3 on
every compared element (all rows for M <= 256, a seeded subset plus the first
and last rows above; rows of Y are independent, so a subset is an exact
check of those rows)."""
import numpy as np
import pytest
import torch

from tests.gpu_util import TOL, activations, host_weights, packed, run_and_compare, sample_rows
from w4a16_quantized_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _dev_f16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.uint16)).cuda().view(torch.float16)


# ---------------------------------------------------------------- packing ----

@pytest.mark.parametrize("K,N,g", [(4096, 4096, 128), (128, 16, 128), (192, 48, 64), (14336, 4096, 128),
                                   (4096, 28672, 64), (384, 144, 128)])
def test_pack_unpack_roundtrip_bit_exact(K, N, g):
    q, z, s, _ = synth.weights(K, N, g)
    w = binding.pack(_dev_u8(q), _dev_u8(z), _dev_f16(s), g)
    q2, z2, s2 = w.unpack()
    assert np.array_equal(q2.cpu().numpy(), q)
    assert np.array_equal(z2.cpu().numpy(), z)
    assert np.array_equal(s2.cpu().numpy().view(np.uint16), s.view(np.uint16))
    assert w.nbytes == binding.packed_bytes(K, N, g)
    w.free()


def test_pack_rejects_bad_codes():
    q, z, s, _ = synth.weights(256, 32, 128)
    q = q.copy()
    q[100, 7] = 16
    with pytest.raises(binding.TMError) as e:
        binding.pack(_dev_u8(q), _dev_u8(z), _dev_f16(s), 128)
    assert e.value.status == 6
    z = z.copy()
    q[100, 7] = 3
    z[1, 31] = 200
    with pytest.raises(binding.TMError) as e:
        binding.pack(_dev_u8(q), _dev_u8(z), _dev_f16(s), 128)
    assert e.value.status == 6
    assert binding.device_error() == 0


# ------------------------------------------------------------ workloads -------

def _cases(idx):
    return [pytest.param(c, id=c.name) for c in synth.workload(idx)]


@pytest.mark.parametrize("case", _cases(0) + _cases(1))
def test_decode_workloads(case):
    err, _ = run_and_compare(case.M, case.K, case.N, case.g, case.stress)
    assert err <= TOL, err


@pytest.mark.parametrize("case", _cases(2))
def test_prefill_workloads(case):
    err, _ = run_and_compare(case.M, case.K, case.N, case.g, case.stress)
    assert err <= TOL, err


@pytest.mark.parametrize("case", _cases(3))
def test_llama70b_workloads(case):
    err, _ = run_and_compare(case.M, case.K, case.N, case.g, case.stress)
    assert err <= TOL, err


@pytest.mark.parametrize("case", _cases(4))
def test_stress_workloads(case):
    err, _ = run_and_compare(case.M, case.K, case.N, case.g, case.stress)
    assert err <= TOL, err


# ------------------------------------------------------------ edge cases ------

@pytest.mark.parametrize("M", [1, 2, 7, 8, 9, 15, 16, 17, 31, 32, 33, 48, 63, 64])
def test_decode_ragged_m(M):
    err, _ = run_and_compare(M, 1024, 384, 128, config={"path": 1})
    assert err <= TOL, err


@pytest.mark.parametrize("M", [1, 33, 64, 65, 127, 128, 129, 200, 257])
def test_prefill_ragged_m(M):
    err, _ = run_and_compare(M, 1024, 384, 128, config={"path": 2})
    assert err <= TOL, err


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("K,N,g", [(128, 16, 128), (64, 16, 64), (192, 48, 64), (640, 272, 128), (896, 4112, 64)])
def test_small_and_ragged_shapes(path, K, N, g):
    """K = g (one group, odd group count), N one n-tile, N not a multiple of the CTA tile."""
    err, _ = run_and_compare(5 if path == 1 else 130, K, N, g, config={"path": path})
    assert err <= TOL, err


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("tile_n", [64, 128, 256])
def test_decode_split_and_tile_overrides(split, tile_n):
    M = 8
    err, _ = run_and_compare(M, 2048, 512, 128, config={"path": 1, "split_k": split, "tile_n": tile_n})
    assert err <= TOL, err


@pytest.mark.parametrize("stages", [2, 3, 5])
def test_decode_stage_override(stages):
    err, _ = run_and_compare(16, 4096, 1024, 64, config={"path": 1, "stages": stages, "split_k": 2})
    assert err <= TOL, err


def test_decode_plan_rejects_bad_settings():
    """Launch settings of the decode kernel outside the served set are refused
    with a status (invalid argument or unsupported), never clamped."""
    w = packed(2048, 512, 128)
    bad = [({"warp_n": 3}, 8, 1), ({"warp_n": 8}, 8, 1), ({"tile_n": 96}, 8, 1), ({"tile_n": 32}, 8, 1),
           ({"stages": 1}, 8, 1), ({"stages": 9}, 8, 1), ({"split_k": 3}, 8, 1), ({"split_k": 16}, 8, 1),
           ({"warp_n": 4}, 32, 3), ({"warp_n": 4, "tile_n": 256}, 32, 3), ({"warp_n": 2, "tile_n": 64}, 64, 3)]
    for cfg, M, status in bad:
        with pytest.raises(binding.TMError) as e:
            binding.plan(w, M, dict(cfg, path=1))
        assert e.value.status == status, (cfg, M, e.value.status)
    # a served combination comes back as asked
    c = binding.plan(w, 8, {"path": 1, "warp_n": 2, "tile_n": 128, "stages": 3, "split_k": 2})
    assert (c["warp_n"], c["tile_n"], c["stages"], c["split_k"]) == (2, 128, 3, 2)


def test_m64_both_paths_agree_with_oracle():
    e1, Y1 = run_and_compare(64, 4096, 1024, 128, config={"path": 1})
    e2, Y2 = run_and_compare(64, 4096, 1024, 128, config={"path": 2})
    assert e1 <= TOL and e2 <= TOL


def test_m_zero_is_noop():
    w = packed(1024, 384, 128)
    X = torch.empty((0, 1024), dtype=torch.float16, device="cuda")
    Y = binding.gemm(X, w)
    assert Y.shape == (0, 384)
    assert binding.last_launch_count() == 0


def test_deterministic_bits():
    for cfg in ({"path": 1, "split_k": 4}, {"path": 2}):
        M = 16 if cfg["path"] == 1 else 256
        w = packed(4096, 1024, 128)
        X = torch.from_numpy(activations(M, 4096, 1024, 128).view(np.uint16)).cuda().view(torch.float16)
        Y1 = binding.gemm(X, w, config=cfg).clone()
        Y2 = binding.gemm(X, w, config=cfg).clone()
        torch.cuda.synchronize()
        assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))


def test_unaligned_pointer_rejected():
    w = packed(1024, 384, 128)
    buf = torch.zeros(2 * 1024 + 8, dtype=torch.float16, device="cuda")
    X = buf[1:1 + 1024].view(1, 1024)  # 2-byte offset
    with pytest.raises(binding.TMError) as e:
        binding.gemm(X, w)
    assert e.value.status == 2


def test_host_buffers_end_to_end():
    """The same call with CPU (pinned) X: copies in, product, copy out."""
    M, K, N, g = 8, 4096, 1024, 128
    X = activations(M, K, N, g)
    Xh = torch.from_numpy(X.view(np.uint16)).view(torch.float16).pin_memory()
    Yh = binding.gemm(Xh, packed(K, N, g))
    assert not Yh.is_cuda
    q, z, s, _ = host_weights(K, N, g)
    import oracle
    err = oracle.rel_max_err(Yh.float().numpy().astype(np.float64), oracle.gemm(X, q, z, s, g))
    assert err <= TOL


def test_gemm_host_entry_point_with_staging_buffers():
    """tm_w4a16_gemm_host with caller-owned device staging buffers, asynchronous
    until the stream is synchronised; every element against the oracle."""
    M, K, N, g = 37, 2048, 1040, 64
    X = activations(M, K, N, g)
    Xh = torch.from_numpy(X.view(np.uint16)).view(torch.float16).pin_memory()
    Yh = torch.full((M, N), float("nan"), dtype=torch.float16).pin_memory()
    Xd = torch.empty(M * K + 64, dtype=torch.float16, device="cuda")
    Yd = torch.empty(M * N + 64, dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    binding.gemm_host(Xh, packed(K, N, g), out=Yh, stream=s, X_dev=Xd, Y_dev=Yd, sync=False)
    assert binding.last_launch_count() == 1
    s.synchronize()
    q, z, s_, _ = host_weights(K, N, g)
    import oracle
    err = oracle.rel_max_err(Yh.float().numpy().astype(np.float64), oracle.gemm(X, q, z, s_, g))
    assert err <= TOL
    # the staged copy of X is X itself, bit for bit
    assert torch.equal(Xd[:M * K].cpu().view(torch.int16), Xh.view(-1).view(torch.int16))


def test_gemm_host_rejects_before_copying():
    w = packed(1024, 384, 128)
    Xh = torch.ones((4, 1024), dtype=torch.float16).pin_memory()
    Yh = torch.zeros((4, 384), dtype=torch.float16).pin_memory()
    Xd = torch.zeros(4 * 1024 + 8, dtype=torch.float16, device="cuda")
    Yd = torch.zeros(4 * 384 + 8, dtype=torch.float16, device="cuda")
    with pytest.raises(binding.TMError) as e:
        binding.gemm_host(Xh, w, out=Yh, X_dev=Xd[1:], Y_dev=Yd)           # misaligned staging buffer
    assert e.value.status == 2
    with pytest.raises(binding.TMError) as e:
        binding.gemm_host(Xh, w, out=Yh, X_dev=Xd, Y_dev=Yd, config={"path": 7})
    assert e.value.status == 1
    torch.cuda.synchronize()
    assert float(Xd.abs().sum()) == 0.0 and float(Yh.abs().sum()) == 0.0


def test_gemm_host_batch_matches_oracle_every_product():
    """tm_w4a16_gemm_host_batch: one copy in, the products in order (decode and
    tensor-memory paths mixed, one M = 0), one copy out."""
    import oracle
    shapes = [(5, 1024, 384, 128), (0, 512, 256, 64), (64, 2048, 1040, 64), (1, 4096, 4096, 128),
              (33, 512, 2048, 128)]
    ws = [packed(K, N, g, seed=i) for i, (M, K, N, g) in enumerate(shapes)]
    batch = binding.HostBatch(ws, [sh[0] for sh in shapes])
    Xs = []
    for i, (M, K, N, g) in enumerate(shapes):
        X = activations(M, K, N, g, seed=i)
        Xs.append(X)
        batch.x(i).copy_(torch.from_numpy(X.view(np.uint16)).view(torch.float16))
    batch.Y_host.fill_(float("nan"))
    batch.run()
    assert binding.last_launch_count() == 4
    for i, (M, K, N, g) in enumerate(shapes):
        if M == 0:
            continue
        q, z, s, _ = host_weights(K, N, g, seed=i)
        err = oracle.rel_max_err(batch.y(i).float().numpy().astype(np.float64), oracle.gemm(Xs[i], q, z, s, g))
        assert err <= TOL, (i, err)
    assert binding.device_error(clear=True) == 0


def test_gemm_host_batch_groups_runs_of_the_same_m():
    """Consecutive products with the same M <= 32 and group size share one
    grouped launch (three g = 128, then, after an M = 0 product, two g = 64);
    M = 40 runs on its own: three launches, every product against the oracle."""
    import oracle
    shapes = [(3, 1024, 384, 128), (3, 512, 256, 128), (3, 2048, 1040, 128), (0, 512, 256, 64),
              (3, 1024, 2048, 64), (3, 4096, 512, 64), (40, 512, 2048, 128)]
    ws = [packed(K, N, g, seed=10 + i) for i, (M, K, N, g) in enumerate(shapes)]
    batch = binding.HostBatch(ws, [sh[0] for sh in shapes])
    Xs = []
    for i, (M, K, N, g) in enumerate(shapes):
        X = activations(M, K, N, g, seed=10 + i)
        Xs.append(X)
        batch.x(i).copy_(torch.from_numpy(X.view(np.uint16)).view(torch.float16))
    batch.Y_host.fill_(float("nan"))
    batch.run()
    assert binding.last_launch_count() == 3
    for i, (M, K, N, g) in enumerate(shapes):
        if M == 0:
            continue
        q, z, s, _ = host_weights(K, N, g, seed=10 + i)
        err = oracle.rel_max_err(batch.y(i).float().numpy().astype(np.float64), oracle.gemm(Xs[i], q, z, s, g))
        assert err <= TOL, (i, err)
    assert binding.device_error(clear=True) == 0


def test_one_launch_per_call():
    w = packed(1024, 384, 128)
    X = torch.zeros((4, 1024), dtype=torch.float16, device="cuda")
    binding.gemm(X, w)
    assert binding.last_launch_count() == 1
    X = torch.zeros((300, 1024), dtype=torch.float16, device="cuda")
    binding.gemm(X, w)
    assert binding.last_launch_count() == 1
    torch.cuda.synchronize()


def test_no_device_errors_left():
    torch.cuda.synchronize()
    assert binding.device_error(clear=False) == 0


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("K", [256, 1024])
def test_prefill_split_override(split, K):
    """Split K over a cluster; with K = 256 and 8 CTAs some CTAs get no K block."""
    err, _ = run_and_compare(200, K, 512, 128, config={"path": 2, "split_k": split})
    assert err <= TOL, err


def test_prefill_auto_split_small_m():
    w = packed(4096, 4096, 128)
    assert binding.plan(w, 128, {"path": 2})["split_k"] > 1
    err, _ = run_and_compare(128, 4096, 4096, 128, config={"path": 2})
    assert err <= TOL, err
