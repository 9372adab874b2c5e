"""Host-side arithmetic behind the bench line (no GPU): the algorithmic byte
and flop counts each roofline divides, the roofline's choice of bound, the
workload definitions, and the gate that drops a traffic figure once its
kernel's source has changed."""
import os

import pytest

import bench


def test_algorithmic_bytes_counts_each_stream():
    # Llama-3-8B gate_up at M = 1, g = 128, counted stream by stream: 4-bit codes,
    # an fp16 scale and a 4-bit zero per (group, column), fp16 X in, fp16 Y out
    K, N, g, M = 4096, 28672, 128, 1
    codes = K * N // 2            # 58,720,256
    scales = (K // g) * N * 2     # 1,835,008
    zeros = (K // g) * N // 2     # 458,752
    x, y = 2 * M * K, 2 * M * N   # 8,192 and 57,344
    assert codes + scales + zeros + x + y == 61_079_552
    assert bench.algorithmic_bytes(M, K, N, g) == 61_079_552
    # g = 64 doubles the scale and zero streams only
    assert bench.algorithmic_bytes(M, K, N, 64) - bench.algorithmic_bytes(M, K, N, 128) == scales + zeros


def test_flops_and_other_byte_counts():
    assert bench.flops(3, 5, 7) == 2 * 3 * 5 * 7
    # RTN: read fp16 W, write a code byte per weight, a zero byte and an fp16 scale per (group, column)
    assert bench.rtn_bytes(256, 8, 128) == 2 * 256 * 8 + 256 * 8 + 2 * 8 + 2 * 2 * 8
    # KV: K and V, per (token, head) D * bits / 8 code bytes + fp16 scale + uint8 zero
    assert bench.kv_cache_bytes(1, 16, 1, 128, 4) == 2 * 16 * (64 + 3)
    assert bench.kv_cache_bytes(2, 16, 8, 128, 8) == 2 * 2 * 16 * 8 * (128 + 3)
    # W8A8 layer: quantiser (read fp16 X, write int8 X and fp32 s_x) + GEMM
    M, K, N = 2, 128, 64
    assert bench.w8a8_bytes(M, K, N) == (2 * M * K + M * K + 4 * M) + (K * N + 4 * N + M * K + 4 * M + 2 * M * N)


PEAKS = {"hbm_gbs": 1000.0, "bf16_tflops": 100.0, "bf16_tflops_sustained": 80.0, "source": "of test"}


def test_roofline_picks_the_longer_bound():
    # 1e9 bytes (1 ms at 1000 GB/s) against 1e10 flops (0.1 ms at 100 TF/s): HBM-bound
    r = bench.roofline_entry(1e9, 1e10, 2e-3, PEAKS)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(500.0) and r["frac"] == pytest.approx(0.5)
    # 1e9 bytes against 1e12 flops (10 ms): tensor-bound, against the burst peak by default
    r = bench.roofline_entry(1e9, 1e12, 20e-3, PEAKS)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 100.0
    assert r["achieved"] == pytest.approx(50.0) and r["frac"] == pytest.approx(0.5)
    r = bench.roofline_entry(1e9, 1e12, 20e-3, PEAKS, tensor_peak="bf16_tflops_sustained")
    assert r["peak"] == 80.0 and r["frac"] == pytest.approx(0.625) and "sustained" in r["peak_source"]


def test_headline_workload_definition():
    c = bench.workload_config("decode")
    assert c["gemms_per_step"] == 16
    assert c["bytes_per_step"] == 461_185_024
    assert c["flops_per_step"] == 24_863_834_112
    p = bench.workload_config("prefill")
    assert p["gemms_per_step"] == 12 and p["flops_per_step"] == 2_289_217_568_768


def test_traffic_is_dropped_once_the_kernel_changed(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    prof = tmp_path / "profiles" / "decode_kernel_w_traffic.txt"
    prof.write_text("# a summary\ndram_bytes_per_launch=123456\nkernel_source_sha=abcd\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_hash", lambda kind: "abcd")
    assert bench.read_traffic("decode", "w") == 123456.0
    monkeypatch.setattr(bench, "kernel_hash", lambda kind: "ef01")
    assert bench.read_traffic("decode", "w") is None
    assert bench.read_traffic("decode", "missing") is None


def test_kernel_hash_covers_the_listed_sources():
    for kind, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(bench.ROOT, "w4a16_quantized_gemm_gb300", "csrc", f)), (kind, f)
        assert len(bench.kernel_hash(kind)) == 16


def _fake_workload(cases):
    """A bench.Workload holding only the cases (no device tensors): enough for runs()."""
    from types import SimpleNamespace
    wl = object.__new__(bench.Workload)
    wl.items = [{"case": SimpleNamespace(M=M, g=g, name=f"p{i}")} for i, (M, g) in enumerate(cases)]
    return wl


def test_step_runs_group_consecutive_products_of_one_small_m():
    from w4a16_quantized_gemm_gb300 import binding
    sizes = lambda wl: [len(r) for r in wl.runs()]
    # the headline step: four linears at each of M = 1, 8, 16, 32 -> four grouped launches
    wl = _fake_workload([(M, 128) for M in (1, 8, 16, 32) for _ in range(4)])
    assert sizes(wl) == [4, 4, 4, 4]
    assert all(len({it["case"].M for it in r}) == 1 for r in wl.runs())
    # at most GROUP_MAX products a launch; a change of M or g starts a new launch
    assert binding.GROUP_MAX == 4
    assert sizes(_fake_workload([(1, 128)] * 6)) == [4, 2]
    assert sizes(_fake_workload([(8, 128), (8, 64), (8, 64), (16, 64)])) == [1, 2, 1]
    # M above 32 (the tensor-memory path) is never grouped
    assert sizes(_fake_workload([(128, 128)] * 4 + [(33, 128)] * 2)) == [1, 1, 1, 1, 1, 1]
    # the products keep their order
    wl = _fake_workload([(1, 128), (1, 128), (8, 128)])
    assert [it["case"].name for r in wl.runs() for it in r] == ["p0", "p1", "p2"]


def test_step_lanes_pair_large_with_small_m_and_move_small_prefill_products():
    from types import SimpleNamespace
    run = lambda M, K=4096, N=4096: [{"case": SimpleNamespace(M=M, K=K, N=N)}]
    Ms = lambda lane: [r[0]["case"].M for r in lane]
    # decode: M = 32 with 1 on the launching stream, 16 with 8 on the second
    main, side = bench.split_lanes([run(M) for M in (1, 8, 16, 32)], "decode")
    assert (Ms(main), Ms(side)) == ([32, 1], [16, 8])
    main, side = bench.split_lanes([run(M) for M in (1, 8, 16)], "decode")
    assert (Ms(main), Ms(side)) == ([16, 1], [8])
    assert bench.split_lanes([run(4)], "decode") == ([run(4)], [])
    # prefill: the products under 60 GFLOP (2MKN) on the second stream, the rest largest first
    shapes = {"qkv": (4096, 6144), "o_proj": (4096, 4096), "gate_up": (4096, 28672), "down": (14336, 4096)}
    runs = [run(M, K, N) for M in (128, 1024, 4096) for K, N in shapes.values()]
    main, side = bench.split_lanes(runs, "prefill")
    assert Ms(side) == [128, 128, 128, 128, 1024, 1024]
    assert [(r[0]["case"].K, r[0]["case"].N) for r in side[4:]] == [shapes["qkv"], shapes["o_proj"]]
    assert Ms(main) == [4096, 4096, 4096, 4096, 1024, 1024]
    assert all(bench.flops(r[0]["case"].M, r[0]["case"].K, r[0]["case"].N) >= 60e9 for r in main)
    # every run once
    assert len(main) + len(side) == len(runs)
    # other workloads: one stream
    assert bench.split_lanes(runs, "stress") == (runs, [])
