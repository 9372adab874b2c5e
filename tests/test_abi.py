"""The C ABI: the library builds, loads without a GPU and exports every entry
point that include/tm_w4a16.h declares; host-side argument checks.  No
compute call is made here."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

from tests.conftest import ROOT

HEADERS = glob.glob(os.path.join(ROOT, "include", "*.h"))


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(tm_\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from w4a16_quantized_gemm_gb300 import build, binding
    build.build()
    return binding.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("tm_pack_weights", "tm_unpack_weights", "tm_w4a16_gemm", "tm_packed_bytes", "tm_packed_free",
              "tm_status_str"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from w4a16_quantized_gemm_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (tm_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_binding_names_match_header():
    from w4a16_quantized_gemm_gb300 import binding
    assert sorted(binding.EXPORTS) == declared_functions()


def test_status_strings(lib):
    from w4a16_quantized_gemm_gb300 import binding
    for st in range(8):
        assert binding.status_str(st) == binding._STATUS[st]
    assert binding.status_str(99) == "unknown status"


@pytest.mark.parametrize("K,N,g,ok", [(4096, 4096, 128, True), (128, 16, 128, True), (192, 32, 64, True),
                                      (4096, 4096, 32, False), (100, 4096, 64, False), (4096, 40, 128, False),
                                      (0, 16, 64, False), (128, 0, 64, False)])
def test_packed_bytes_validation(lib, K, N, g, ok):
    out = ctypes.c_size_t()
    st = lib.tm_packed_bytes(K, N, g, ctypes.byref(out))
    assert (st == 0) == ok
    if ok:
        # codes + one fp16 scale and one 4-bit zero per (group, column), K padded to 2g
        Kp = -(-K // (2 * g)) * (2 * g)
        assert out.value >= Kp * N // 2 + (Kp // g) * N * 5 // 2


def test_null_arguments_are_rejected(lib):
    h = ctypes.c_void_p()
    assert lib.tm_pack_weights(None, None, None, 128, 16, 64, ctypes.byref(h)) == 1
    assert lib.tm_pack_weights(None, None, None, 128, 16, 64, None) == 1
    assert lib.tm_unpack_weights(None, None, None, None) == 1
    assert lib.tm_w4a16_gemm(None, None, None, 1, None) == 1
    assert lib.tm_packed_info(None, None, None, None, None) == 1
    lib.tm_packed_free(None)
    assert lib.tm_last_launch_count() == 0


def test_grouped_entry_points_reject_bad_host_arguments(lib):
    """tm_w4a16_gemm_grouped / tm_gemm_plan_grouped check the problem list on
    the host before touching a handle (no device needed)."""
    from w4a16_quantized_gemm_gb300 import binding
    out = binding.GemmConfig()
    arr = (binding.GemmProblem * (binding.GROUP_MAX + 1))()
    assert lib.tm_w4a16_gemm_grouped(None, 1, 1, None, None) == 1
    assert lib.tm_w4a16_gemm_grouped(arr, 0, 1, None, None) == 1
    assert lib.tm_w4a16_gemm_grouped(arr, binding.GROUP_MAX + 1, 1, None, None) == 1
    assert lib.tm_w4a16_gemm_grouped(arr, 1, 1, None, None) == 1          # NULL handle
    assert lib.tm_w4a16_gemm_grouped(arr, 1, -1, None, None) == 1
    assert lib.tm_gemm_plan_grouped(arr, 1, 1, None, None, None) == 1     # NULL out
    assert lib.tm_gemm_plan_grouped(None, 1, 1, None, ctypes.byref(out), None) == 1
    assert lib.tm_last_launch_count() == 0


def test_library_has_sm103a_code():
    """The build targets sm_103a only (checked from the build flags)."""
    from w4a16_quantized_gemm_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_new_entry_points_reject_bad_host_arguments(lib):
    """Argument checks of the quantisers, the KV cache and W8A8 entry points run on
    the host before any launch (fake device addresses: nothing is dereferenced)."""
    a16, odd = ctypes.c_void_p(1 << 20), ctypes.c_void_p((1 << 20) + 1)
    INVALID, ALIGN, UNSUP, OK = 1, 2, 3, 0
    # RTN quantiser
    assert lib.tm_quantize_rtn(None, 128, 16, 128, a16, a16, a16, None) == INVALID
    assert lib.tm_quantize_rtn(a16, 100, 16, 128, a16, a16, a16, None) == INVALID     # K % g
    assert lib.tm_quantize_rtn(odd, 128, 16, 128, a16, a16, a16, None) == ALIGN
    # KV cache
    assert lib.tm_kv_quantize(None, 4, 128, 8, a16, a16, a16, None) == INVALID
    assert lib.tm_kv_quantize(a16, 4, 128, 5, a16, a16, a16, None) == INVALID         # bits
    assert lib.tm_kv_quantize(a16, 4, 96, 8, a16, a16, a16, None) == INVALID          # D
    assert lib.tm_kv_quantize(odd, 4, 128, 8, a16, a16, a16, None) == ALIGN
    assert lib.tm_kv_pack_v(None, 1, 16, 8, 8, a16, None) == INVALID
    assert lib.tm_kv_pack_v(a16, 1, 20, 8, 8, a16, None) == INVALID                   # L % 16
    assert lib.tm_kv_pack_v(a16, 1, 16, 8, 8, odd, None) == ALIGN
    attn = lambda *p, B=1, Hq=32, Hkv=8, L=16, D=128, bits=8, split=0, out=a16: lib.tm_kv_decode_attention(
        *p, B, Hq, Hkv, L, D, bits, split, out, None)
    assert attn(None, a16, a16, a16, a16, a16, a16, a16) == INVALID
    assert attn(a16, a16, a16, a16, a16, a16, a16, a16, L=20) == INVALID              # L % 16
    assert attn(a16, a16, a16, a16, a16, a16, a16, a16, D=64) == INVALID              # D
    assert attn(a16, a16, a16, a16, a16, a16, a16, a16, Hq=48, Hkv=3) == UNSUP        # 16 heads per KV head
    assert attn(a16, a16, a16, a16, a16, a16, a16, a16, split=3) == INVALID
    assert attn(odd, a16, a16, a16, a16, a16, a16, a16) == ALIGN
    assert attn(a16, a16, a16, a16, a16, a16, a16, a16, B=0) == OK                    # nothing to do
    app = lambda *p, B=1, Hkv=8, L=16, D=128, bits=8: lib.tm_kv_append(p[0], p[1], p[2], B, Hkv, L, D, bits,
                                                                        *p[3:], None)
    assert app(None, a16, a16, a16, a16, a16, a16, a16, a16) == INVALID
    assert app(a16, a16, a16, a16, a16, a16, a16, a16, a16, L=20) == INVALID          # L % 16
    assert app(a16, a16, a16, a16, a16, a16, a16, a16, a16, bits=6) == INVALID
    assert app(odd, a16, a16, a16, a16, a16, a16, a16, a16) == ALIGN
    assert app(a16, a16, a16, a16, a16, a16, a16, a16, a16, B=0) == OK
    # W8A8
    assert lib.tm_w8a8_quantize_act(None, 1, 128, a16, a16, None) == INVALID
    assert lib.tm_w8a8_quantize_act(a16, 1, 100, a16, a16, None) == INVALID           # K % 16
    assert lib.tm_w8a8_quantize_act(odd, 1, 128, a16, a16, None) == ALIGN
    assert lib.tm_w8a8_quantize_act(a16, 0, 128, a16, a16, None) == OK                # no rows
    h = ctypes.c_void_p()
    assert lib.tm_w8_pack(None, a16, 128, 16, ctypes.byref(h)) == INVALID
    assert lib.tm_w8_pack(a16, a16, 100, 16, ctypes.byref(h)) == INVALID              # K % 16
    assert lib.tm_w8_pack(a16, a16, 128, 16, None) == INVALID
    assert lib.tm_w8_unpack(None, a16, a16) == INVALID
    assert lib.tm_w8_packed_info(None, None, None, None) == INVALID
    lib.tm_w8_packed_free(None)
    assert lib.tm_w8a8_gemm(None, a16, a16, a16, 1, 0, None) == INVALID
    assert lib.tm_w8a8_gemm(a16, a16, a16, a16, 1, 3, None) == INVALID                 # split
    assert lib.tm_w8a8_gemm_ex(a16, a16, a16, a16, 64, 0, 96, None) == INVALID         # tile_m
    assert lib.tm_w8a8_gemm(odd, a16, a16, a16, 1, 0, None) == ALIGN
    assert lib.tm_w8a8_gemm(a16, a16, a16, a16, 0, 0, None) == OK                      # M = 0
    assert lib.tm_w8_quantize_weight(None, 128, 16, a16, a16, None) == INVALID
    assert lib.tm_w8_quantize_weight(a16, 128, 20, a16, a16, None) == INVALID        # N % 16
    assert lib.tm_w8_quantize_weight(odd, 128, 16, a16, a16, None) == ALIGN


def test_host_buffer_entry_points_reject_bad_arguments(lib):
    """tm_w4a16_gemm_host / tm_w4a16_gemm_host_batch check their arguments on the
    host before any copy (fake device addresses: nothing is dereferenced)."""
    a16, odd = ctypes.c_void_p(1 << 20), ctypes.c_void_p((1 << 20) + 1)
    INVALID, OK = 1, 0
    assert lib.tm_w4a16_gemm_host(a16, None, a16, 1, a16, a16, None, None) == INVALID   # no weights
    assert lib.tm_w4a16_gemm_host(a16, None, a16, -1, a16, a16, None, None) == INVALID
    assert lib.tm_w4a16_gemm_host(None, None, None, 0, None, None, None, None) == INVALID
    assert lib.tm_w4a16_gemm_host_batch(-1, None, None, a16, a16, a16, a16, None) == INVALID
    assert lib.tm_w4a16_gemm_host_batch(0, None, None, None, None, None, None, None) == OK   # nothing to do
    assert lib.tm_w4a16_gemm_host_batch(2, None, None, a16, a16, a16, a16, None) == INVALID
    ps = (ctypes.c_void_p * 2)(None, None)
    ms = (ctypes.c_int * 2)(1, 1)
    assert lib.tm_w4a16_gemm_host_batch(2, ps, ms, a16, a16, a16, odd, None) == INVALID    # null handle
    assert lib.tm_last_launch_count() == 0


def test_w8a8_f16_entry_points_reject_bad_host_arguments(lib):
    a16, odd = ctypes.c_void_p(1 << 20), ctypes.c_void_p((1 << 20) + 2)
    INVALID, ALIGN, OK = 1, 2, 0
    assert lib.tm_w8a8_quantize_act_f16(None, 1, 128, a16, a16, None) == INVALID
    assert lib.tm_w8a8_quantize_act_f16(a16, 1, 100, a16, a16, None) == INVALID       # K % 16
    assert lib.tm_w8a8_quantize_act_f16(a16, 1, 128, odd, a16, None) == ALIGN
    assert lib.tm_w8a8_quantize_act_f16(a16, 0, 128, a16, a16, None) == OK            # no rows
    assert lib.tm_w8a8_gemm_f16(None, a16, a16, a16, 64, 0, 0, None) == INVALID
    assert lib.tm_w8a8_gemm_f16(a16, a16, a16, a16, 64, 3, 0, None) == INVALID         # split
    assert lib.tm_w8a8_gemm_f16(a16, a16, a16, a16, 64, 0, 32, None) == INVALID        # tile_m
    assert lib.tm_w8a8_gemm_f16(odd, a16, a16, a16, 64, 0, 0, None) == ALIGN
    assert lib.tm_w8a8_gemm_f16(a16, a16, a16, a16, 0, 0, 0, None) == OK               # M = 0
