"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- a closed form, a library routine in a special case, a
hand-worked example, or numbers the pages print.  None needs a GPU."""
import numpy as np
import pytest

import oracle
from tests.conftest import parse_matrix, read_golden
from w4a16_quantized_gemm_gb300 import synth


def _rng(seed):
    return np.random.default_rng(seed)


# --- fp16 decoding -----------------------------------------------------------

def test_half_decode_all_patterns_match_numpy():
    """Every binary16 bit pattern decodes like numpy's float16 -> float64."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    lib = oracle._load()
    got = np.array([lib.oracle_half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


@pytest.mark.parametrize("bits,val", [(0x3C00, 1.0), (0xC000, -2.0), (0x7BFF, 65504.0),
                                      (0x0001, 2.0 ** -24), (0x0400, 2.0 ** -14),
                                      (0x03FF, 1023 * 2.0 ** -24), (0x3555, 0.333251953125)])
def test_half_decode_textbook_values(bits, val):
    assert oracle.half_to_double(bits) == val


# --- closed forms of the dequantisation rule ---------------------------------

def _rand_scales(rng, G, N):
    return rng.uniform(1e-3, 2e-2, size=(G, N)).astype(np.float16)


def test_code_equal_zero_gives_zero():
    rng = _rng(1)
    K, N, g = 256, 24, 128
    z = rng.integers(0, 16, size=(K // g, N), dtype=np.uint8)
    q = np.repeat(z, g, axis=0)
    s = _rand_scales(rng, K // g, N)
    X = rng.standard_normal((3, K)).astype(np.float16)
    Y = oracle.gemm(X, q, z, s, g)
    assert np.all(Y == 0.0)


@pytest.mark.parametrize("qv,zv,mult", [(15, 0, 15.0), (0, 15, -15.0), (7, 3, 4.0)])
def test_single_code_closed_form(qv, zv, mult):
    """One-hot X picks one weight: Y = (q - z) * s exactly."""
    rng = _rng(2)
    K, N, g = 128, 16, 64
    q = np.full((K, N), qv, np.uint8)
    z = np.full((K // g, N), zv, np.uint8)
    s = _rand_scales(rng, K // g, N)
    X = np.zeros((K, K), np.float16)
    X[np.arange(K), np.arange(K)] = 1.0
    Y = oracle.gemm(X, q, z, s, g)
    expect = mult * np.repeat(s.astype(np.float64), g, axis=0)
    assert np.array_equal(Y, expect)


# --- special cases that reduce to a library matmul ---------------------------

def test_one_group_constant_zero_and_scale_is_numpy_matmul():
    """g = K, z constant, s = 2^-3: Y = 2^-3 * X @ (Q - z0) (numpy, exact)."""
    rng = _rng(3)
    M, K, N = 5, 64, 40
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    z = np.full((1, N), 9, np.uint8)
    s = np.full((1, N), 0.125, np.float16)
    X = rng.integers(-4, 5, size=(M, K)).astype(np.float16)
    Y = oracle.gemm(X, q, z, s, K)
    ref = 0.125 * (X.astype(np.float64) @ (q.astype(np.float64) - 9.0))
    assert np.array_equal(Y, ref)


def test_grouping_runs_along_k_not_n():
    """Two groups along K with different constant (z, s): the product splits
    into two numpy matmuls over the K halves.  An oracle that grouped along N,
    or indexed the group by k % G, fails this."""
    rng = _rng(4)
    M, K, N, g = 3, 32, 48, 16
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    z = np.stack([np.full(N, 2, np.uint8), np.full(N, 13, np.uint8)])
    s = np.stack([np.full(N, 0.5, np.float16), np.full(N, 4.0, np.float16)])
    X = rng.integers(-4, 5, size=(M, K)).astype(np.float16)
    Y = oracle.gemm(X, q, z, s, g)
    Xd = X.astype(np.float64)
    qd = q.astype(np.float64)
    ref = 0.5 * (Xd[:, :g] @ (qd[:g] - 2.0)) + 4.0 * (Xd[:, g:] @ (qd[g:] - 13.0))
    assert np.array_equal(Y, ref)


def test_column_sums_closed_form():
    """X = ones: Y[n] = sum_groups s * (sum of codes in the group - g * z)."""
    rng = _rng(5)
    K, N, g = 512, 32, 128
    G = K // g
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    z = rng.integers(0, 16, size=(G, N), dtype=np.uint8)
    s = (2.0 ** -rng.integers(2, 9, size=(G, N))).astype(np.float16)
    X = np.ones((1, K), np.float16)
    Y = oracle.gemm(X, q, z, s, g)[0]
    code_sums = q.astype(np.int64).reshape(G, g, N).sum(axis=1)
    ref = (s.astype(np.float64) * (code_sums - g * z.astype(np.int64))).sum(axis=0)
    assert np.array_equal(Y, ref)


def test_linearity_in_x_exact():
    rng = _rng(6)
    M, K, N, g = 4, 256, 24, 64
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    z = rng.integers(0, 16, size=(K // g, N), dtype=np.uint8)
    s = (2.0 ** -rng.integers(3, 10, size=(K // g, N))).astype(np.float16)
    X1 = rng.integers(-3, 4, size=(M, K)).astype(np.float16)
    X2 = rng.integers(-3, 4, size=(M, K)).astype(np.float16)
    a = 3.0
    lhs = oracle.gemm((a * X1.astype(np.float64) + X2).astype(np.float16), q, z, s, g)
    rhs = a * oracle.gemm(X1, q, z, s, g) + oracle.gemm(X2, q, z, s, g)
    assert np.array_equal(lhs, rhs)


def test_transpose_sensitivity_nonsquare():
    """A non-square problem with one-hot rows: row k of Y is row k of the
    dequantised weights, which has N entries; a transposed operand cannot
    reproduce it."""
    rng = _rng(7)
    K, N, g = 128, 40, 64
    q = rng.integers(0, 16, size=(K, N), dtype=np.uint8)
    z = rng.integers(0, 16, size=(K // g, N), dtype=np.uint8)
    s = (2.0 ** -rng.integers(1, 6, size=(K // g, N))).astype(np.float16)
    ks = [0, 1, 63, 64, 127]
    X = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        X[i, k] = 1.0
    Y = oracle.gemm(X, q, z, s, g)
    for i, k in enumerate(ks):
        grp = k // g
        expect = (q[k].astype(np.float64) - z[grp]) * s[grp].astype(np.float64)
        assert np.array_equal(Y[i], expect)


# --- hand-worked example -------------------------------------------------------

def test_handworked_example():
    d = read_golden("w4a16_handworked_2x8x2_g4.txt")
    M, K, N, g = (int(d[k]) for k in ("M", "K", "N", "g"))
    X = np.array(parse_matrix(d["X"]), np.float16)
    q = np.array(parse_matrix(d["q"], int), np.uint8)
    z = np.array(parse_matrix(d["z"], int), np.uint8)
    s = np.array(parse_matrix(d["s"]), np.float16)
    Y = oracle.gemm(X, q, z, s, g)
    assert Y.shape == (M, N)
    assert np.array_equal(Y, np.array(parse_matrix(d["Y"])))


# --- implementation invariants ---------------------------------------------------

def test_row_subset_and_thread_count_bitwise():
    p = synth.problem(7, 256, 48, 64)
    full1 = oracle.gemm(p.X, p.q, p.z, p.s, p.g, threads=1)
    full8 = oracle.gemm(p.X, p.q, p.z, p.s, p.g, threads=8)
    assert np.array_equal(full1, full8)
    rows = [6, 0, 3]
    sub = oracle.gemm(p.X, p.q, p.z, p.s, p.g, rows=rows, threads=3)
    assert np.array_equal(sub, full1[rows])


def test_bad_code_rejected():
    q = np.zeros((64, 16), np.uint8)
    q[5, 3] = 16
    z = np.zeros((1, 16), np.uint8)
    s = np.ones((1, 16), np.float16)
    with pytest.raises(ValueError):
        oracle.gemm(np.ones((1, 64), np.float16), q, z, s, 64)


# --- sizing arithmetic the pages print ------------------------------------------

def test_kv_sizing_worked_example():
    d = read_golden("kv_sizing_llama3_8b.txt")
    per_tok = oracle.kv_bytes_per_token(int(d["layers"]), int(d["kv_heads"]), int(d["head_dim"]),
                                        int(d["elem_bytes"]))
    assert per_tok == int(d["bytes_per_token"])
    assert per_tok * int(d["block_tokens"]) == int(d["bytes_per_block"])


def test_llama3_layer_shapes_match_workloads():
    """The 8B dims of the KV example (8 KV heads of 128) give the fused qkv
    width 4096 + 2*8*128 = 6144 used by the workloads; same for 70B."""
    d = read_golden("kv_sizing_llama3_8b.txt")
    s8 = oracle.llama_linear_shapes(4096, 32, int(d["kv_heads"]), int(d["head_dim"]), 14336)
    assert s8 == synth.LLAMA3_8B
    s70 = oracle.llama_linear_shapes(8192, 64, 8, 128, 28672)
    assert s70 == synth.LLAMA3_70B


def test_compression_ratio_claim():
    d = read_golden("w4a16_footprint_claims.txt")
    g = int(d["group_size"])
    r = oracle.compression_vs_fp16(g)
    assert float(d["compression_low"]) <= r <= float(d["compression_high"])
    assert r == pytest.approx(16.0 / (4.0 + 20.0 / 128.0))
    # bytes of the codes + group metadata of one layer, against the formula's parts
    K, N = 4096, 4096
    assert oracle.algorithmic_bytes(0, K, N, g) * 8 == pytest.approx(K * N * oracle.bits_per_weight(g))


def test_algorithmic_bytes_closed_form():
    # 1 x 4096 x 4096, g=128: codes 8 MiB, scales 256 KiB, zeros 64 KiB, X and Y 8 KiB each
    assert oracle.algorithmic_bytes(1, 4096, 4096, 128) == 8388608 + 262144 + 65536 + 8192 + 8192
    assert oracle.flops(1, 4096, 4096) == 2 * 4096 * 4096


def test_7b_store_claim():
    """A Llama-2-7B-sized model (32 layers, hidden 4096, 32 heads of 128 with no
    grouped KV, intermediate 11008, vocab 32000 -- these dims are an assumption,
    the page names no model) packed at g=128, plus fp16 input and output
    embeddings, lands in the page's rough 4-5 GB."""
    d = read_golden("w4a16_footprint_claims.txt")
    shapes = oracle.llama_linear_shapes(4096, 32, 32, 128, 11008)
    w = oracle.linear_weight_count(32, shapes)
    packed = w * oracle.bits_per_weight(128) / 8
    emb = 2 * 32000 * 4096 * 2
    gb = (packed + emb) / 1e9
    assert float(d["store_7b_low_gb"]) <= gb <= float(d["store_7b_high_gb"])


def test_8b_linear_weight_count():
    w = oracle.linear_weight_count(32, synth.LLAMA3_8B)
    assert w == 6979321856
