"""The seeded input generator: known answers, determinism and the value recipe."""
import numpy as np

from w4a16_quantized_gemm_gb300 import synth


def test_splitmix64_known_answers():
    """SplitMix64 from seed 0 (Steele, Lea, Flood 2014): the published first outputs."""
    got = [int(v) for v in synth.draws(0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_draws_offsets_are_a_window():
    a = synth.draws(12345, 100)
    b = synth.draws(12345, 40, 60)
    assert np.array_equal(a[60:], b)


def test_deterministic_and_distinct():
    p1 = synth.problem(3, 256, 64, 128)
    p2 = synth.problem(3, 256, 64, 128)
    for a in ("X", "q", "z", "s"):
        assert np.array_equal(getattr(p1, a), getattr(p2, a))
    p3 = synth.problem(3, 256, 64, 128, seed=1)
    assert not np.array_equal(p1.q, p3.q)


def test_value_recipe():
    p = synth.problem(64, 4096, 512, 128)
    assert p.q.dtype == np.uint8 and p.q.max() == 15 and p.q.min() == 0
    counts = np.bincount(p.q.ravel(), minlength=16) / p.q.size
    assert np.all(np.abs(counts - 1 / 16) < 0.005)
    s = p.s.astype(np.float64)
    assert s.min() >= np.float16(1e-3) and s.max() <= np.float16(2e-2)
    x = p.X.astype(np.float64)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02
    assert p.X.dtype == np.float16 and p.s.dtype == np.float16


def test_stress_recipe():
    K, N, g = 4096, 256, 64
    p = synth.problem(8, K, N, g, stress=True)
    assert len(p.salient) == 41  # round(0.01 * 4096)
    assert len(synth.salient_channels("seed0/K14336/salient", 14336)) == 143
    base = f"seed0/K{K}/N{N}/g{g}/stress"
    s64 = synth.scales64(base + "/s", K // g, N)
    grp = np.unique(p.salient // g)
    others = np.setdiff1d(np.arange(K // g), grp)
    assert np.array_equal(p.s[grp], (s64[grp] / 20.0).astype(np.float16))
    assert np.array_equal(p.s[others], s64[others].astype(np.float16))
    # some scales of the salient groups are fp16 subnormal (below 2^-14)
    assert (p.s[grp].astype(np.float64) < 2.0 ** -14).any()
    x64 = synth.normal64(f"seed0/X/M8/K{K}/N{N}/g{g}/stress", 8, K)
    assert np.array_equal(p.X[:, p.salient], (x64[:, p.salient] * 20.0).astype(np.float16))


def test_workloads():
    assert [len(synth.workload(i)) for i in range(5)] == [1, 16, 12, 16, 12]
    c = synth.workload(4)
    assert {x.g for x in c} == {64, 128} and all(x.stress for x in c)
