"""GPU parity of the low-bit KV cache: the quantiser bit-exact against the
binary32 oracle; decode attention over an oracle-quantised cache within
max|out - out_ref| / max|out_ref| <= 2e-3 of the fp64 oracle.  The bar: scores
are exact products of fp16 queries and integer codes summed in fp32 (~1e-6);
the value weights p s_v are rounded once to fp16 (2^-12 relative per term,
averaging out over tokens); the fp16 output rounding 2^-11 of |out| dominates."""
import numpy as np
import pytest
import torch

import oracle
import oracle.kv as kv
from w4a16_quantized_gemm_gb300 import binding, synth

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

TOL = 2e-3


def _fp16(tag, *shape, scale=1.0):
    n = int(np.prod(shape))
    return (synth.normal64(tag, 1, n).reshape(shape) * scale).astype(np.float16)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_kv_quantize_bit_exact(bits, D):
    X = _fp16(f"kvq/{bits}/{D}", 2, 37, 8, D, scale=0.8)
    X[0, 0, 0] = 0                       # an all-zero vector
    X[0, 0, 1] = np.float16(0.3)         # a constant vector
    c, s, z = binding.kv_quantize(_dev(X.view(np.uint16)).view(torch.float16), bits)
    torch.cuda.synchronize()
    c0, s0, z0 = kv.quantize(X, bits)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), s0.view(np.uint16))
    assert np.array_equal(z.cpu().numpy(), z0)
    assert np.array_equal(c.cpu().numpy(), c0)


@pytest.mark.parametrize("bits", [8, 4])
def test_kv_quantize_exact_ties_bit_exact(bits):
    """Vectors holding, for one fp16 scale each, the maximum B s and every
    exact tie (k + 1/2) s that is an fp16 value: the codes equal the division
    rule's (a multiply by fl(1/s) would round some ties the wrong way)."""
    from tests.test_gpu_rtn import tie_columns
    X = np.ascontiguousarray(tie_columns(2 ** bits - 1, 128, count=1024).T)  # [vectors][D = 128]
    c, s, z = binding.kv_quantize(_dev(X.view(np.uint16)).view(torch.float16), bits)
    torch.cuda.synchronize()
    c0, s0, z0 = kv.quantize(X, bits)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), s0.view(np.uint16))
    assert np.array_equal(z.cpu().numpy(), z0)
    assert np.array_equal(c.cpu().numpy(), c0)


def _hm(a):
    """[B][L][Hkv](...) -> the head-major cache order [B][Hkv][L](...)."""
    return np.ascontiguousarray(np.swapaxes(a, 1, 2))


def _cache(B, L, Hkv, bits, tag):
    K = _fp16(f"{tag}/K", B, L, Hkv, 128)
    V = _fp16(f"{tag}/V", B, L, Hkv, 128)
    return kv.quantize(K, bits), kv.quantize(V, bits)


def _run(B, L, Hq, Hkv, bits, lengths, split=0, tag="attn", poison_tail=False):
    L = (L + 15) // 16 * 16  # the cache capacity is whole 16-token tiles; lengths stay ragged
    (kc, ks, kz), (vc, vs, vz) = _cache(B, L, Hkv, bits, f"{tag}/{B}/{L}/{Hkv}/{bits}")
    Q = _fp16(f"{tag}/Q/{B}/{Hq}", B, Hq, 128)
    lens = np.asarray(lengths, dtype=np.int32)
    ks_d, vs_d = ks.copy(), vs.copy()
    if poison_tail:  # slots past each length hold NaN scales: they must not reach the output
        for b, n in enumerate(lens):
            ks_d[b, max(n, 0):] = np.float16(np.nan)
            vs_d[b, max(n, 0):] = np.float16(np.inf)
    out = binding.kv_decode_attention(
        _dev(Q.view(np.uint16)).view(torch.float16),
        (_dev(_hm(kc)), _dev(_hm(ks_d).view(np.uint16)).view(torch.float16), _dev(_hm(kz))),
        (binding.kv_pack_v(_dev(_hm(vc)), bits), _dev(_hm(vs_d).view(np.uint16)).view(torch.float16), _dev(_hm(vz))),
        _dev(lens), bits, split)
    torch.cuda.synchronize()
    ref = kv.decode_attention(Q.astype(np.float64), kv.dequantize(kc, ks, kz, bits), kv.dequantize(vc, vs, vz, bits),
                              np.minimum(np.maximum(lens, 0), L))
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    return oracle.rel_max_err(got, ref), got, ref


@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (16, 8), (8, 8), (64, 8)])
def test_attention_llama_heads(bits, Hq, Hkv):
    err, _, _ = _run(2, 1024, Hq, Hkv, bits, [1024, 777])
    assert err <= TOL, err


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("bits", [8, 4])
def test_attention_split_override(split, bits):
    err, _, _ = _run(1, 4096, 32, 8, bits, [4096], split=split)
    assert err <= TOL, err


@pytest.mark.parametrize("split", [1, 4, 8])
def test_attention_eight_heads_per_kv_head(split):
    err, _, _ = _run(2, 512, 64, 8, 8, [512, 100], split=split)
    assert err <= TOL, err


@pytest.mark.parametrize("L,lengths", [(1, [1]), (37, [37, 5, 16]), (300, [0, 300, 17]), (129, [129, 128, 1])])
def test_attention_ragged_lengths(L, lengths):
    err, got, _ = _run(len(lengths), L, 32, 8, 8, lengths)
    assert err <= TOL, err
    for b, n in enumerate(lengths):
        if n == 0:
            assert np.all(got[b] == 0)


@pytest.mark.parametrize("bits", [8, 4])
def test_attention_ignores_the_cache_past_each_length(bits):
    err, _, _ = _run(3, 400, 32, 8, bits, [400, 131, 7], poison_tail=True)
    assert err <= TOL, err


def test_attention_long_context_auto_split():
    err, _, _ = _run(1, 32768, 32, 8, 4, [32768])
    assert err <= TOL, err


def test_quantize_then_attention_pipeline():
    """GPU quantiser output fed to GPU attention equals the oracle pipeline."""
    B, L, Hq, Hkv, bits = 2, 528, 32, 8, 8
    K = _fp16("pipe/K", B, L, Hkv, 128)
    V = _fp16("pipe/V", B, L, Hkv, 128)
    Q = _fp16("pipe/Q", B, Hq, 128)
    kq = binding.kv_quantize(_dev(_hm(K).view(np.uint16)).view(torch.float16), bits)
    vq = binding.kv_quantize(_dev(_hm(V).view(np.uint16)).view(torch.float16), bits)
    lens = np.array([513, 300], dtype=np.int32)
    vq = (binding.kv_pack_v(vq[0], bits), vq[1], vq[2])
    out = binding.kv_decode_attention(_dev(Q.view(np.uint16)).view(torch.float16), kq, vq, _dev(lens), bits)
    torch.cuda.synchronize()
    k0, v0 = kv.quantize(K, bits), kv.quantize(V, bits)
    ref = kv.decode_attention(Q.astype(np.float64), kv.dequantize(*k0, bits), kv.dequantize(*v0, bits), lens)
    assert oracle.rel_max_err(out.float().cpu().numpy().astype(np.float64), ref) <= TOL


def test_attention_rejects_unsupported():
    Q = torch.zeros((1, 48, 128), dtype=torch.float16, device="cuda")
    c = torch.zeros((1, 3, 16, 128), dtype=torch.uint8, device="cuda")
    s = torch.zeros((1, 3, 16), dtype=torch.float16, device="cuda")
    z = torch.zeros((1, 3, 16), dtype=torch.uint8, device="cuda")
    lens = torch.tensor([4], dtype=torch.int32, device="cuda")
    with pytest.raises(binding.TMError) as e:       # 16 query heads per KV head
        binding.kv_decode_attention(Q, (c, s, z), (c, s, z), lens, 8)
    assert e.value.status == 3
    c = torch.zeros((1, 3, 12, 128), dtype=torch.uint8, device="cuda")
    s = torch.zeros((1, 3, 12), dtype=torch.float16, device="cuda")
    z = torch.zeros((1, 3, 12), dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.TMError) as e:       # capacity not a multiple of 16 tokens
        binding.kv_decode_attention(Q[:, :6], (c, s, z), (c, s, z), lens, 8)
    assert e.value.status == 1


def test_attention_rejects_misaligned_cache():
    Q = torch.zeros((1, 8, 128), dtype=torch.float16, device="cuda")
    c = torch.zeros((1, 2, 16, 128), dtype=torch.uint8, device="cuda")
    s = torch.zeros((1, 2, 16), dtype=torch.float16, device="cuda")
    z = torch.zeros((1, 2, 16), dtype=torch.uint8, device="cuda")
    z_off = torch.zeros(2 * 16 + 1, dtype=torch.uint8, device="cuda")[1:].view(1, 2, 16)  # one byte off
    lens = torch.tensor([4], dtype=torch.int32, device="cuda")
    with pytest.raises(binding.TMError) as e:
        binding.kv_decode_attention(Q, (c, s, z_off), (c, s, z), lens, 8)
    assert e.value.status == 2


@pytest.mark.parametrize("bits", [8, 4])
def test_append_token_by_token_equals_bulk(bits):
    """Appending the tokens one decode step at a time (tm_kv_append) builds the
    same cache, bit for bit, as quantising them in bulk and packing the value
    tiles; positions outside the cache are ignored."""
    B, Hkv, L, D = 2, 8, 48, 128
    K = _fp16(f"app/K/{bits}", B, Hkv, L, D)   # head-major
    V = _fp16(f"app/V/{bits}", B, Hkv, L, D)
    RB = D * bits // 8
    kc = torch.zeros((B, Hkv, L, RB), dtype=torch.uint8, device="cuda")
    ks = torch.zeros((B, Hkv, L), dtype=torch.float16, device="cuda")
    kz = torch.zeros((B, Hkv, L), dtype=torch.uint8, device="cuda")
    vt = torch.zeros(B * Hkv * L * RB, dtype=torch.uint8, device="cuda")
    vs = torch.zeros((B, Hkv, L), dtype=torch.float16, device="cuda")
    vz = torch.zeros((B, Hkv, L), dtype=torch.uint8, device="cuda")
    Kd = _dev(K.view(np.uint16)).view(torch.float16)
    Vd = _dev(V.view(np.uint16)).view(torch.float16)
    for step in range(L):
        pos = torch.tensor([step, L - 1 - step], dtype=torch.int32, device="cuda")  # sequence 1 fills backwards
        rows = torch.tensor([step, L - 1 - step], device="cuda")
        Kn = torch.stack([Kd[b, :, int(rows[b])] for b in range(B)]).contiguous()
        Vn = torch.stack([Vd[b, :, int(rows[b])] for b in range(B)]).contiguous()
        binding.kv_append(Kn, Vn, pos, (kc, ks, kz), (vt, vs, vz), bits)
    bad = torch.tensor([-1, L], dtype=torch.int32, device="cuda")       # ignored
    binding.kv_append(torch.ones_like(Kn), torch.ones_like(Vn), bad, (kc, ks, kz), (vt, vs, vz), bits)
    torch.cuda.synchronize()
    kq = binding.kv_quantize(Kd, bits)
    vq = binding.kv_quantize(Vd, bits)
    tiles = binding.kv_pack_v(vq[0], bits)
    torch.cuda.synchronize()
    assert torch.equal(kc, kq[0]) and torch.equal(kz, kq[2]) and torch.equal(ks.view(torch.int16), kq[1].view(torch.int16))
    assert torch.equal(vz, vq[2]) and torch.equal(vs.view(torch.int16), vq[1].view(torch.int16))
    assert torch.equal(vt, tiles)
    # and against the oracle's quantiser
    c0, s0, z0 = kv.quantize(K, bits)
    assert np.array_equal(kc.cpu().numpy(), c0) and np.array_equal(kz.cpu().numpy(), z0)
