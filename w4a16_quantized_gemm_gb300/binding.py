"""Thin ctypes binding of ``include/tm_w4a16.h`` and ``include/tm_w8a8.h``
(argument marshalling only).

Every step of the computation runs in the CUDA library; PyTorch provides
device memory and streams.  If the library is missing this module raises --
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

TM_OK = 0
_STATUS = {0: "ok", 1: "invalid argument", 2: "pointer not 16-byte aligned", 3: "unsupported configuration",
           4: "CUDA call failed", 5: "device barrier timeout", 6: "code or zero above 15",
           7: "request exceeds the static staging array"}

EXPORTS = ("tm_status_str", "tm_packed_bytes", "tm_pack_weights", "tm_unpack_weights", "tm_packed_info",
           "tm_packed_free", "tm_w4a16_gemm", "tm_w4a16_gemm_ex", "tm_gemm_plan", "tm_device_error",
           "tm_last_launch_count", "tm_quantize_rtn", "tm_w4a16_gemm_silu_mul", "tm_selftest_wait_timeout",
           "tm_kv_quantize", "tm_kv_decode_attention", "tm_kv_pack_v", "tm_w8a8_quantize_act", "tm_w8_pack",
           "tm_w8_unpack", "tm_w8_packed_info", "tm_w8_packed_free", "tm_w8a8_gemm", "tm_w8a8_gemm_ex",
           "tm_w8_quantize_weight", "tm_kv_append", "tm_w4a16_gemm_host", "tm_w4a16_gemm_host_batch",
           "tm_w8a8_quantize_act_f16", "tm_w8a8_gemm_f16", "tm_w4a16_gemm_host_static",
           "tm_w4a16_gemm_grouped", "tm_gemm_plan_grouped")

GROUP_MAX = 4  # TM_GROUP_MAX


class TMError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_STATUS.get(status, status)} (status {status})")
        self.status = status


class GemmConfig(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("split_k", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("stages", ctypes.c_int), ("warp_n", ctypes.c_int), ("tile_m", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class GemmProblem(ctypes.Structure):
    _fields_ = [("X", ctypes.c_void_p), ("p", ctypes.c_void_p), ("Y", ctypes.c_void_p), ("silu", ctypes.c_int)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None):
    """Load the CUDA library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing; run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, ci, csz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.tm_status_str.restype = ctypes.c_char_p
    lib.tm_status_str.argtypes = [ci]
    lib.tm_packed_bytes.restype = ci
    lib.tm_packed_bytes.argtypes = [ci, ci, ci, ctypes.POINTER(csz)]
    lib.tm_pack_weights.restype = ci
    lib.tm_pack_weights.argtypes = [vp, vp, vp, ci, ci, ci, ctypes.POINTER(vp)]
    lib.tm_unpack_weights.restype = ci
    lib.tm_unpack_weights.argtypes = [vp, vp, vp, vp]
    lib.tm_packed_info.restype = ci
    lib.tm_packed_info.argtypes = [vp, ctypes.POINTER(ci), ctypes.POINTER(ci), ctypes.POINTER(ci),
                                   ctypes.POINTER(csz)]
    lib.tm_packed_free.restype = None
    lib.tm_packed_free.argtypes = [vp]
    lib.tm_w4a16_gemm.restype = ci
    lib.tm_w4a16_gemm.argtypes = [vp, vp, vp, ci, vp]
    lib.tm_w4a16_gemm_ex.restype = ci
    lib.tm_w4a16_gemm_ex.argtypes = [vp, vp, vp, ci, ctypes.POINTER(GemmConfig), vp]
    lib.tm_w4a16_gemm_host.restype = ci
    lib.tm_w4a16_gemm_host.argtypes = [vp, vp, vp, ci, vp, vp, ctypes.POINTER(GemmConfig), vp]
    lib.tm_w4a16_gemm_host_static.restype = ci
    lib.tm_w4a16_gemm_host_static.argtypes = [vp, vp, vp, ci, ctypes.POINTER(GemmConfig), vp]
    lib.tm_w4a16_gemm_host_batch.restype = ci
    lib.tm_w4a16_gemm_host_batch.argtypes = [ci, ctypes.POINTER(vp), ctypes.POINTER(ci), vp, vp, vp, vp, vp]
    lib.tm_gemm_plan.restype = ci
    lib.tm_gemm_plan.argtypes = [vp, ci, ctypes.POINTER(GemmConfig), ctypes.POINTER(GemmConfig)]
    lib.tm_device_error.restype = ci
    lib.tm_device_error.argtypes = [ci, ctypes.POINTER(ctypes.c_uint32)]
    lib.tm_last_launch_count.restype = ci
    lib.tm_last_launch_count.argtypes = []
    lib.tm_kv_quantize.restype = ci
    lib.tm_kv_quantize.argtypes = [vp, ctypes.c_longlong, ci, ci, vp, vp, vp, vp]
    lib.tm_kv_pack_v.restype = ci
    lib.tm_kv_pack_v.argtypes = [vp, ci, ci, ci, ci, vp, vp]
    lib.tm_kv_append.restype = ci
    lib.tm_kv_append.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci] + [vp] * 7
    lib.tm_kv_decode_attention.restype = ci
    lib.tm_kv_decode_attention.argtypes = [vp] * 8 + [ci] * 7 + [vp, vp]
    lib.tm_selftest_wait_timeout.restype = ci
    lib.tm_selftest_wait_timeout.argtypes = [vp]
    lib.tm_w4a16_gemm_silu_mul.restype = ci
    lib.tm_w4a16_gemm_silu_mul.argtypes = [vp, vp, vp, ci, ctypes.POINTER(GemmConfig), vp]
    lib.tm_quantize_rtn.restype = ci
    lib.tm_quantize_rtn.argtypes = [vp, ci, ci, ci, vp, vp, vp, vp]
    lib.tm_w8a8_quantize_act.restype = ci
    lib.tm_w8a8_quantize_act.argtypes = [vp, ci, ci, vp, vp, vp]
    lib.tm_w8_pack.restype = ci
    lib.tm_w8_pack.argtypes = [vp, vp, ci, ci, ctypes.POINTER(vp)]
    lib.tm_w8_unpack.restype = ci
    lib.tm_w8_unpack.argtypes = [vp, vp, vp]
    lib.tm_w8_packed_info.restype = ci
    lib.tm_w8_packed_info.argtypes = [vp, ctypes.POINTER(ci), ctypes.POINTER(ci), ctypes.POINTER(csz)]
    lib.tm_w8_packed_free.restype = None
    lib.tm_w8_packed_free.argtypes = [vp]
    lib.tm_w8a8_gemm.restype = ci
    lib.tm_w8a8_gemm.argtypes = [vp, vp, vp, vp, ci, ci, vp]
    lib.tm_w8_quantize_weight.restype = ci
    lib.tm_w8_quantize_weight.argtypes = [vp, ci, ci, vp, vp, vp]
    lib.tm_w8a8_gemm_ex.restype = ci
    lib.tm_w8a8_gemm_ex.argtypes = [vp, vp, vp, vp, ci, ci, ci, vp]
    lib.tm_w8a8_quantize_act_f16.restype = ci
    lib.tm_w8a8_quantize_act_f16.argtypes = [vp, ci, ci, vp, vp, vp]
    lib.tm_w8a8_gemm_f16.restype = ci
    lib.tm_w8a8_gemm_f16.argtypes = [vp, vp, vp, vp, ci, ci, ci, vp]
    lib.tm_w4a16_gemm_grouped.argtypes = [ctypes.POINTER(GemmProblem), ci, ci, ctypes.POINTER(GemmConfig), vp]
    lib.tm_gemm_plan_grouped.argtypes = [ctypes.POINTER(GemmProblem), ci, ci, ctypes.POINTER(GemmConfig),
                                         ctypes.POINTER(GemmConfig), ctypes.POINTER(ci)]
    _lib = lib
    return lib


def _check(st: int, what: str):
    if st != TM_OK:
        raise TMError(st, what)


def status_str(st: int) -> str:
    return load().tm_status_str(st).decode()


def packed_bytes(K: int, N: int, g: int) -> int:
    out = ctypes.c_size_t()
    _check(load().tm_packed_bytes(K, N, g, ctypes.byref(out)), "tm_packed_bytes")
    return out.value


def _dev(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


class PackedWeights:
    """Owns a ``tm_packed`` handle (device memory on the device of ``q``)."""

    def __init__(self, q: torch.Tensor, z: torch.Tensor, s: torch.Tensor, g: int):
        lib = load()
        K, N = q.shape
        handle = ctypes.c_void_p()
        with torch.cuda.device(q.device):
            st = lib.tm_pack_weights(_dev(q, torch.uint8, "q"), _dev(z, torch.uint8, "z"),
                                     _dev(s, torch.float16, "s"), K, N, g, ctypes.byref(handle))
        _check(st, "tm_pack_weights")
        self._h = handle
        self.K, self.N, self.g = K, N, g
        self.device = q.device
        b = ctypes.c_size_t()
        _check(lib.tm_packed_info(handle, None, None, None, ctypes.byref(b)), "tm_packed_info")
        self.nbytes = b.value

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("packed weights were freed")
        return self._h

    def unpack(self):
        q = torch.empty((self.K, self.N), dtype=torch.uint8, device=self.device)
        z = torch.empty((self.K // self.g, self.N), dtype=torch.uint8, device=self.device)
        s = torch.empty((self.K // self.g, self.N), dtype=torch.float16, device=self.device)
        with torch.cuda.device(self.device):
            _check(load().tm_unpack_weights(self.handle, q.data_ptr(), z.data_ptr(), s.data_ptr()),
                   "tm_unpack_weights")
        return q, z, s

    def free(self):
        if self._h is not None:
            load().tm_packed_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def pack(q: torch.Tensor, z: torch.Tensor, s: torch.Tensor, g: int) -> PackedWeights:
    return PackedWeights(q, z, s, g)


def _cfg(config) -> Optional[GemmConfig]:
    if config is None:
        return None
    if isinstance(config, GemmConfig):
        return config
    c = GemmConfig()
    for k, v in dict(config).items():
        setattr(c, k, int(v))
    return c


def plan(w: PackedWeights, M: int, config=None) -> dict:
    out = GemmConfig()
    c = _cfg(config)
    _check(load().tm_gemm_plan(w.handle, M, ctypes.byref(c) if c else None, ctypes.byref(out)), "tm_gemm_plan")
    return out.as_dict()


def gemm(X: torch.Tensor, w: PackedWeights, out: Optional[torch.Tensor] = None, config=None,
         stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Y = X . dequant(W) on the GPU.

    X: fp16 [M][K].  On a CUDA tensor the call is asynchronous on ``stream``
    (default: the current stream).  On a CPU tensor (pinned for speed) X is
    copied to the device, the product runs, and Y comes back to the host --
    the end-to-end form of the same call.
    """
    if X.dim() != 2 or X.shape[1] != w.K or X.dtype != torch.float16:
        raise ValueError("X must be fp16 [M][K]")
    if not X.is_cuda:
        return _gemm_host(X, w, out, config, stream)
    M = X.shape[0]
    if out is None:
        out = torch.empty((M, w.N), dtype=torch.float16, device=X.device)
    elif out.shape != (M, w.N) or out.dtype != torch.float16 or not out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous CUDA fp16 [M][N] tensor")
    X = X.contiguous()
    s = stream if stream is not None else torch.cuda.current_stream(X.device)
    c = _cfg(config)
    lib = load()
    if c is None:
        st = lib.tm_w4a16_gemm(X.data_ptr(), w.handle, out.data_ptr(), M, ctypes.c_void_p(s.cuda_stream))
    else:
        st = lib.tm_w4a16_gemm_ex(X.data_ptr(), w.handle, out.data_ptr(), M, ctypes.byref(c),
                                  ctypes.c_void_p(s.cuda_stream))
    _check(st, "tm_w4a16_gemm")
    return out


def gemm_silu_mul(X: torch.Tensor, w: PackedWeights, out: Optional[torch.Tensor] = None, config=None,
                  stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """H = silu(X . W_gate) * (X . W_up) from one packed gate/up weight whose
    columns interleave gate and up in blocks of 4 (see tm_w4a16_gemm_silu_mul).
    X: CUDA fp16 [M][K]; returns fp16 [M][N/2]; asynchronous on ``stream``."""
    if X.dim() != 2 or X.shape[1] != w.K or X.dtype != torch.float16 or not X.is_cuda:
        raise ValueError("X must be a CUDA fp16 [M][K] tensor")
    M = X.shape[0]
    if out is None:
        out = torch.empty((M, w.N // 2), dtype=torch.float16, device=X.device)
    elif out.shape != (M, w.N // 2) or out.dtype != torch.float16 or not out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous CUDA fp16 [M][N/2] tensor")
    X = X.contiguous()
    s = stream if stream is not None else torch.cuda.current_stream(X.device)
    c = _cfg(config)
    _check(load().tm_w4a16_gemm_silu_mul(X.data_ptr(), w.handle, out.data_ptr(), M,
                                         ctypes.byref(c) if c else None, ctypes.c_void_p(s.cuda_stream)),
           "tm_w4a16_gemm_silu_mul")
    return out


def _problems(items, M, check_out=True):
    arr = (GemmProblem * len(items))()
    for i, (X, w, out, silu) in enumerate(items):
        arr[i].X = X.data_ptr() if X is not None else None
        arr[i].p = w.handle
        arr[i].Y = out.data_ptr() if out is not None else None
        arr[i].silu = 1 if silu else 0
    return arr


def plan_grouped(weights, M: int, config=None, silu=None) -> dict:
    """Settings tm_w4a16_gemm_grouped would use for these packed weights at M
    rows; "splits" lists each product's split along K ("split_k" is the
    launch's cluster size)."""
    silu = list(silu) if silu is not None else [False] * len(weights)
    arr = _problems([(None, w, None, f) for w, f in zip(weights, silu)], M)
    out = GemmConfig()
    splits = (ctypes.c_int * max(1, len(weights)))()
    c = _cfg(config)
    _check(load().tm_gemm_plan_grouped(arr, len(weights), M, ctypes.byref(c) if c else None, ctypes.byref(out),
                                       splits), "tm_gemm_plan_grouped")
    d = out.as_dict()
    d["splits"] = [splits[i] for i in range(len(weights))]
    return d


def gemm_grouped(problems, config=None, stream: Optional[torch.cuda.Stream] = None):
    """Independent products of the same M in one launch (tm_w4a16_gemm_grouped).

    problems: up to GROUP_MAX tuples (X, w, out, silu) -- X CUDA fp16 [M][K],
    w PackedWeights, out a CUDA fp16 [M][N] tensor ([M][N/2] with silu) or
    None to allocate, silu a bool.  No out may overlap any X or another out.
    Returns the list of outputs; asynchronous on ``stream``."""
    items = []
    M = None
    for X, w, out, silu in problems:
        if X.dim() != 2 or X.shape[1] != w.K or X.dtype != torch.float16 or not X.is_cuda:
            raise ValueError("every X must be a CUDA fp16 [M][K] tensor")
        if M is None:
            M = X.shape[0]
        elif X.shape[0] != M:
            raise ValueError("every X must have the same number of rows")
        cols = w.N // 2 if silu else w.N
        if out is None:
            out = torch.empty((M, cols), dtype=torch.float16, device=X.device)
        elif out.shape != (M, cols) or out.dtype != torch.float16 or not out.is_cuda or not out.is_contiguous():
            raise ValueError(f"out must be a contiguous CUDA fp16 [{M}][{cols}] tensor")
        items.append((X.contiguous(), w, out, bool(silu)))
    if not items:
        raise ValueError("at least one problem")
    s = stream if stream is not None else torch.cuda.current_stream(items[0][0].device)
    c = _cfg(config)
    arr = _problems(items, M)
    _check(load().tm_w4a16_gemm_grouped(arr, len(items), M, ctypes.byref(c) if c else None,
                                        ctypes.c_void_p(s.cuda_stream)), "tm_w4a16_gemm_grouped")
    return [it[2] for it in items]


def _gemm_host(X, w, out, config, stream):
    return gemm_host(X, w, out, config, stream)


def _host_fp16(t: torch.Tensor, shape, name: str):
    if t.is_cuda or t.dtype != torch.float16 or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host fp16 tensor of shape {tuple(shape)}")


def _staging(t: Optional[torch.Tensor], numel: int, device, name: str) -> torch.Tensor:
    if t is None:
        return torch.empty(numel, dtype=torch.float16, device=device)
    if not t.is_cuda or t.dtype != torch.float16 or not t.is_contiguous() or t.numel() < numel:
        raise ValueError(f"{name} must be a contiguous CUDA fp16 buffer of at least {numel} elements")
    return t


def gemm_host(X: torch.Tensor, w: PackedWeights, out: Optional[torch.Tensor] = None, config=None,
              stream: Optional[torch.cuda.Stream] = None, X_dev: Optional[torch.Tensor] = None,
              Y_dev: Optional[torch.Tensor] = None, sync: bool = True) -> torch.Tensor:
    """tm_w4a16_gemm_host: X fp16 [M][K] in host memory (pinned for speed) is
    copied to the device buffer ``X_dev``, the product runs into ``Y_dev``, and
    the result comes back into ``out`` (host fp16 [M][N]; pinned, allocated
    when None).  Staging buffers are allocated when None.  With ``sync`` the
    call waits for the stream; otherwise read ``out`` after synchronising it."""
    if X.dim() != 2:
        raise ValueError("X must be fp16 [M][K]")
    M = X.shape[0]
    _host_fp16(X, (M, w.K), "X")
    if out is None:
        out = torch.empty((M, w.N), dtype=torch.float16, pin_memory=True)
    _host_fp16(out, (M, w.N), "out")
    X_dev = _staging(X_dev, M * w.K, w.device, "X_dev")
    Y_dev = _staging(Y_dev, M * w.N, w.device, "Y_dev")
    s = stream if stream is not None else torch.cuda.current_stream(w.device)
    c = _cfg(config)
    _check(load().tm_w4a16_gemm_host(X.data_ptr(), w.handle, out.data_ptr(), M, X_dev.data_ptr(), Y_dev.data_ptr(),
                                     ctypes.byref(c) if c else None, ctypes.c_void_p(s.cuda_stream)),
           "tm_w4a16_gemm_host")
    if sync:
        s.synchronize()
    return out


STATIC_STAGING_BYTES = 8 << 20  # TM_STATIC_STAGING_BYTES


def gemm_host_static(X: torch.Tensor, w: PackedWeights, out: Optional[torch.Tensor] = None, config=None,
                     stream: Optional[torch.cuda.Stream] = None, sync: bool = True) -> torch.Tensor:
    """tm_w4a16_gemm_host_static: as ``gemm_host``, but staged through the
    library's fixed device array, so that the call allocates no device memory
    (``out``, the host result, is allocated here when None).  Calls share the
    array: issue them on one stream."""
    if X.dim() != 2:
        raise ValueError("X must be fp16 [M][K]")
    M = X.shape[0]
    _host_fp16(X, (M, w.K), "X")
    if out is None:
        out = torch.empty((M, w.N), dtype=torch.float16, pin_memory=True)
    _host_fp16(out, (M, w.N), "out")
    s = stream if stream is not None else torch.cuda.current_stream(w.device)
    c = _cfg(config)
    with torch.cuda.device(w.device):
        _check(load().tm_w4a16_gemm_host_static(X.data_ptr(), w.handle, out.data_ptr(), M,
                                                ctypes.byref(c) if c else None, ctypes.c_void_p(s.cuda_stream)),
               "tm_w4a16_gemm_host_static")
    if sync:
        s.synchronize()
    return out


class HostBatch:
    """A fixed list of products with host inputs and outputs for
    tm_w4a16_gemm_host_batch: ``X_host`` / ``Y_host`` are pinned buffers that
    hold every X_i / Y_i back to back (``x(i)`` and ``y(i)`` are views of
    them), staged through one device buffer each way."""

    def __init__(self, weights, Ms, device=None):
        if len(weights) != len(Ms) or any(m < 0 for m in Ms):
            raise ValueError("one non-negative M per weight")
        self.weights, self.Ms = list(weights), [int(m) for m in Ms]
        dev = device if device is not None else (self.weights[0].device if self.weights else 0)
        self.x_off, self.y_off = [0], [0]
        for w, m in zip(self.weights, self.Ms):
            self.x_off.append(self.x_off[-1] + m * w.K)
            self.y_off.append(self.y_off[-1] + m * w.N)
        self.X_host = torch.empty(self.x_off[-1], dtype=torch.float16, pin_memory=True)
        self.Y_host = torch.empty(self.y_off[-1], dtype=torch.float16, pin_memory=True)
        self.X_dev = torch.empty(self.x_off[-1], dtype=torch.float16, device=dev)
        self.Y_dev = torch.empty(self.y_off[-1], dtype=torch.float16, device=dev)
        n = len(self.weights)
        self._p = (ctypes.c_void_p * max(1, n))(*[w.handle for w in self.weights])
        self._m = (ctypes.c_int * max(1, n))(*self.Ms)

    def x(self, i: int) -> torch.Tensor:
        return self.X_host[self.x_off[i]:self.x_off[i + 1]].view(self.Ms[i], self.weights[i].K)

    def y(self, i: int) -> torch.Tensor:
        return self.Y_host[self.y_off[i]:self.y_off[i + 1]].view(self.Ms[i], self.weights[i].N)

    def run(self, stream: Optional[torch.cuda.Stream] = None, sync: bool = True):
        s = stream if stream is not None else torch.cuda.current_stream(self.X_dev.device)
        _check(load().tm_w4a16_gemm_host_batch(len(self.weights), self._p, self._m, self.X_host.data_ptr(),
                                               self.Y_host.data_ptr(), self.X_dev.data_ptr(),
                                               self.Y_dev.data_ptr(), ctypes.c_void_p(s.cuda_stream)),
               "tm_w4a16_gemm_host_batch")
        if sync:
            s.synchronize()


def quantize_rtn(W: torch.Tensor, g: int, stream: Optional[torch.cuda.Stream] = None):
    """Round-to-nearest INT4 quantisation of fp16 W [K][N] on the GPU:
    returns (q uint8 [K][N], z uint8 [K/g][N], s fp16 [K/g][N]), the inputs of
    ``pack``.  Asynchronous on ``stream`` (default: the current stream)."""
    if W.dim() != 2 or W.dtype != torch.float16:
        raise ValueError("W must be fp16 [K][N]")
    K, N = W.shape
    Wd = W.contiguous()
    _dev(Wd, torch.float16, "W")
    q = torch.empty((K, N), dtype=torch.uint8, device=Wd.device)
    z = torch.empty((K // g if g > 0 else 0, N), dtype=torch.uint8, device=Wd.device)
    s = torch.empty((K // g if g > 0 else 0, N), dtype=torch.float16, device=Wd.device)
    st = stream if stream is not None else torch.cuda.current_stream(Wd.device)
    with torch.cuda.device(Wd.device):
        _check(load().tm_quantize_rtn(Wd.data_ptr(), K, N, g, q.data_ptr(), z.data_ptr(), s.data_ptr(),
                                      ctypes.c_void_p(st.cuda_stream)), "tm_quantize_rtn")
    return q, z, s


def kv_quantize(X: torch.Tensor, bits: int, stream: Optional[torch.cuda.Stream] = None):
    """Quantise fp16 vectors X [..., D] (one per (token, head)) to int8 / int4:
    returns (codes uint8 [..., D or D/2], s fp16 [...], z uint8 [...])."""
    if X.dtype != torch.float16 or not X.is_cuda or X.dim() < 1:
        raise ValueError("X must be a CUDA fp16 tensor [..., D]")
    X = X.contiguous()
    D = X.shape[-1]
    lead = tuple(X.shape[:-1])
    rows = X.numel() // D if D else 0
    codes = torch.empty(lead + (D if bits == 8 else D // 2,), dtype=torch.uint8, device=X.device)
    s = torch.empty(lead, dtype=torch.float16, device=X.device)
    z = torch.empty(lead, dtype=torch.uint8, device=X.device)
    st = stream if stream is not None else torch.cuda.current_stream(X.device)
    _check(load().tm_kv_quantize(X.data_ptr(), rows, D, bits, codes.data_ptr(), s.data_ptr(), z.data_ptr(),
                                 ctypes.c_void_p(st.cuda_stream)), "tm_kv_quantize")
    return codes, s, z


def kv_pack_v(codes: torch.Tensor, bits: int, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Value codes [B][Hkv][L][D*bits/8] -> the 16-token tiles in MMA lane
    order the attention kernel reads (see tm_kv_pack_v)."""
    if codes.dim() != 4 or codes.dtype != torch.uint8 or codes.shape[3] != 128 * bits // 8:
        raise ValueError("codes must be uint8 [B][Hkv][L][128*bits/8]")
    B, Hkv, L, _ = codes.shape
    codes = codes.contiguous()
    tiles = torch.empty(B * Hkv * L * 128 * bits // 8, dtype=torch.uint8, device=codes.device)
    st = stream if stream is not None else torch.cuda.current_stream(codes.device)
    _check(load().tm_kv_pack_v(codes.data_ptr(), B, L, Hkv, bits, tiles.data_ptr(), ctypes.c_void_p(st.cuda_stream)),
           "tm_kv_pack_v")
    return tiles


def kv_append(Kn: torch.Tensor, Vn: torch.Tensor, pos: torch.Tensor, k: tuple, v: tuple, bits: int,
              stream: Optional[torch.cuda.Stream] = None) -> None:
    """Quantise the new token's K and V (fp16 [B][Hkv][D]) into the head-major
    cache at positions pos (int32 [B]); k = (codes, s, z), v = (tiles, s, z) as
    for kv_decode_attention (see tm_kv_append)."""
    kc, ks, kz = k
    vc, vs, vz = v
    B, Hkv, D = Kn.shape
    if tuple(Vn.shape) != (B, Hkv, D) or kc.dim() != 4 or kc.shape[0] != B or kc.shape[1] != Hkv:
        raise ValueError("Kn, Vn must be [B][Hkv][D] over a [B][Hkv][L][.] cache")
    if pos.dtype != torch.int32 or tuple(pos.shape) != (B,):
        raise ValueError("pos must be int32 [B]")
    L = kc.shape[2]
    ts = [Kn, Vn, pos, kc, ks, kz, vc, vs, vz]
    if any((not t.is_cuda) or (not t.is_contiguous()) for t in ts):
        raise ValueError("all tensors must be contiguous CUDA tensors")
    st = stream if stream is not None else torch.cuda.current_stream(Kn.device)
    _check(load().tm_kv_append(Kn.data_ptr(), Vn.data_ptr(), pos.data_ptr(), B, Hkv, L, D, bits, kc.data_ptr(),
                               ks.data_ptr(), kz.data_ptr(), vc.data_ptr(), vs.data_ptr(), vz.data_ptr(),
                               ctypes.c_void_p(st.cuda_stream)), "tm_kv_append")


def kv_decode_attention(Q: torch.Tensor, k: tuple, v: tuple, lengths: torch.Tensor, bits: int, split: int = 0,
                        out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """Q fp16 [B][Hq][D]; k = (codes [B][Hkv][L][D*bits/8], s fp16 [B][Hkv][L],
    z uint8 [B][Hkv][L]) -- the head-major cache; v = (tiles from kv_pack_v,
    s, z as for k); lengths int32 [B].  Returns fp16 [B][Hq][D]."""
    B, Hq, D = Q.shape
    kc, ks, kz = k
    vc, vs, vz = v
    if kc.dim() != 4 or kc.shape[0] != B or tuple(lengths.shape) != (B,):
        raise ValueError("key codes must be [B][Hkv][L][D*bits/8] and lengths [B], B as in Q")
    if Q.dtype != torch.float16 or kc.dtype != torch.uint8 or vc.dtype != torch.uint8:
        raise ValueError("Q must be fp16 and the codes uint8")
    Hkv, L = kc.shape[1], kc.shape[2]
    if kc.shape[3] != D * bits // 8 or vc.numel() != B * Hkv * L * D * bits // 8:
        raise ValueError("code sizes do not match D and bits")
    if tuple(ks.shape) != (B, Hkv, L) or tuple(vs.shape) != (B, Hkv, L):
        raise ValueError("scales and zeros must be [B][Hkv][L] like the key codes")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float16, device=Q.device)
    ts = [Q, kc, ks, kz, vc, vs, vz, lengths]
    if any((not t.is_cuda) or (not t.is_contiguous()) for t in ts) or lengths.dtype != torch.int32:
        raise ValueError("all inputs must be contiguous CUDA tensors; lengths int32")
    st = stream if stream is not None else torch.cuda.current_stream(Q.device)
    _check(load().tm_kv_decode_attention(*(t.data_ptr() for t in ts), B, Hq, Hkv, L, D, bits, split,
                                         out.data_ptr(), ctypes.c_void_p(st.cuda_stream)), "tm_kv_decode_attention")
    return out


def selftest_wait_timeout(stream: Optional[torch.cuda.Stream] = None) -> None:
    """Launch the bounded-wait self-test (see tm_selftest_wait_timeout)."""
    s = stream if stream is not None else torch.cuda.current_stream()
    _check(load().tm_selftest_wait_timeout(ctypes.c_void_p(s.cuda_stream)), "tm_selftest_wait_timeout")


def device_error(clear: bool = True) -> int:
    bits = ctypes.c_uint32()
    st = load().tm_device_error(1 if clear else 0, ctypes.byref(bits))
    if st not in (TM_OK, 5):
        raise TMError(st, "tm_device_error")
    return bits.value


def last_launch_count() -> int:
    return load().tm_last_launch_count()


# ------------------------------------------------------------------ W8A8 ---

def w8a8_quantize_act(X: torch.Tensor, out: Optional[tuple] = None, stream: Optional[torch.cuda.Stream] = None):
    """Per-token int8 quantisation of fp16 X [M][K] (see tm_w8a8_quantize_act):
    returns (xq int8 [M][K], sx fp32 [M]), into `out` when given."""
    if X.dim() != 2 or X.dtype != torch.float16:
        raise ValueError("X must be fp16 [M][K]")
    M, K = X.shape
    if out is None:
        xq = torch.empty((M, K), dtype=torch.int8, device=X.device)
        sx = torch.empty((M,), dtype=torch.float32, device=X.device)
    else:
        xq, sx = out
        if tuple(xq.shape) != (M, K) or tuple(sx.shape) != (M,):
            raise ValueError("out must be (int8 [M][K], fp32 [M])")
    st = stream if stream is not None else torch.cuda.current_stream(X.device)
    _check(load().tm_w8a8_quantize_act(_dev(X, torch.float16, "X"), M, K, _dev(xq, torch.int8, "xq"),
                                       _dev(sx, torch.float32, "sx"), ctypes.c_void_p(st.cuda_stream)),
           "tm_w8a8_quantize_act")
    return xq, sx


def w8a8_quantize_act_f16(X: torch.Tensor, out: Optional[tuple] = None, stream: Optional[torch.cuda.Stream] = None):
    """tm_w8a8_quantize_act_f16: the same per-token codes as exact fp16 integers:
    returns (xq16 fp16 [M][K], sx fp32 [M]), into `out` when given."""
    if X.dim() != 2 or X.dtype != torch.float16:
        raise ValueError("X must be fp16 [M][K]")
    M, K = X.shape
    if out is None:
        xq = torch.empty((M, K), dtype=torch.float16, device=X.device)
        sx = torch.empty((M,), dtype=torch.float32, device=X.device)
    else:
        xq, sx = out
        if tuple(xq.shape) != (M, K) or tuple(sx.shape) != (M,):
            raise ValueError("out must be (fp16 [M][K], fp32 [M])")
    st = stream if stream is not None else torch.cuda.current_stream(X.device)
    _check(load().tm_w8a8_quantize_act_f16(_dev(X, torch.float16, "X"), M, K, _dev(xq, torch.float16, "xq16"),
                                           _dev(sx, torch.float32, "sx"), ctypes.c_void_p(st.cuda_stream)),
           "tm_w8a8_quantize_act_f16")
    return xq, sx


def w8_quantize_weight(W: torch.Tensor, stream: Optional[torch.cuda.Stream] = None):
    """Per-output-channel int8 quantisation of fp16 W [K][N] on the GPU (see
    tm_w8_quantize_weight): returns (q int8 [K][N], sw fp32 [N]), the inputs of
    ``pack_w8``."""
    if W.dim() != 2 or W.dtype != torch.float16:
        raise ValueError("W must be fp16 [K][N]")
    K, N = W.shape
    q = torch.empty((K, N), dtype=torch.int8, device=W.device)
    sw = torch.empty((N,), dtype=torch.float32, device=W.device)
    st = stream if stream is not None else torch.cuda.current_stream(W.device)
    _check(load().tm_w8_quantize_weight(_dev(W, torch.float16, "W"), K, N, q.data_ptr(), sw.data_ptr(),
                                        ctypes.c_void_p(st.cuda_stream)), "tm_w8_quantize_weight")
    return q, sw


class W8Packed:
    """Owns a ``tm_w8_packed`` handle (device memory on the device of ``q``)."""

    def __init__(self, q: torch.Tensor, sw: torch.Tensor):
        lib = load()
        K, N = q.shape
        handle = ctypes.c_void_p()
        with torch.cuda.device(q.device):
            st = lib.tm_w8_pack(_dev(q, torch.int8, "q"), _dev(sw, torch.float32, "sw"), K, N, ctypes.byref(handle))
        _check(st, "tm_w8_pack")
        self._h = handle
        self.K, self.N = K, N
        self.device = q.device
        b = ctypes.c_size_t()
        _check(lib.tm_w8_packed_info(handle, None, None, ctypes.byref(b)), "tm_w8_packed_info")
        self.nbytes = b.value

    @property
    def handle(self):
        if self._h is None:
            raise RuntimeError("packed weights were freed")
        return self._h

    def unpack(self):
        q = torch.empty((self.K, self.N), dtype=torch.int8, device=self.device)
        sw = torch.empty((self.N,), dtype=torch.float32, device=self.device)
        with torch.cuda.device(self.device):
            _check(load().tm_w8_unpack(self.handle, q.data_ptr(), sw.data_ptr()), "tm_w8_unpack")
        return q, sw

    def free(self):
        if self._h is not None:
            load().tm_w8_packed_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def pack_w8(q: torch.Tensor, sw: torch.Tensor) -> W8Packed:
    return W8Packed(q, sw)


def w8a8_gemm(xq: torch.Tensor, sx: torch.Tensor, w: W8Packed, out: Optional[torch.Tensor] = None, split: int = 0,
              tile_m: int = 0, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Y = fp16(sx sw^T (xq . q_w)) for int8 xq [M][K] and fp32 sx [M] (tm_w8a8_gemm_ex)."""
    if xq.dim() != 2 or xq.shape[1] != w.K:
        raise ValueError("xq must be int8 [M][K]")
    M = xq.shape[0]
    if tuple(sx.shape) != (M,):
        raise ValueError("sx must be fp32 [M]")
    if out is None:
        out = torch.empty((M, w.N), dtype=torch.float16, device=xq.device)
    if tuple(out.shape) != (M, w.N):
        raise ValueError("out must be fp16 [M][N]")
    st = stream if stream is not None else torch.cuda.current_stream(xq.device)
    _check(load().tm_w8a8_gemm_ex(_dev(xq, torch.int8, "xq"), _dev(sx, torch.float32, "sx"), w.handle,
                                  _dev(out, torch.float16, "out"), M, split, tile_m, ctypes.c_void_p(st.cuda_stream)),
           "tm_w8a8_gemm_ex")
    return out


def w8a8_gemm_f16(xq16: torch.Tensor, sx: torch.Tensor, w: W8Packed, out: Optional[torch.Tensor] = None,
                  split: int = 0, tile_m: int = 0, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """tm_w8a8_gemm_f16: the product with the codes as fp16 integers [M][K]
    (from w8a8_quantize_act_f16), on the tensor-memory kernel for every M."""
    if xq16.dim() != 2 or xq16.shape[1] != w.K:
        raise ValueError("xq16 must be fp16 [M][K]")
    M = xq16.shape[0]
    if tuple(sx.shape) != (M,):
        raise ValueError("sx must be fp32 [M]")
    if out is None:
        out = torch.empty((M, w.N), dtype=torch.float16, device=xq16.device)
    if tuple(out.shape) != (M, w.N):
        raise ValueError("out must be fp16 [M][N]")
    st = stream if stream is not None else torch.cuda.current_stream(xq16.device)
    _check(load().tm_w8a8_gemm_f16(_dev(xq16, torch.float16, "xq16"), _dev(sx, torch.float32, "sx"), w.handle,
                                   _dev(out, torch.float16, "out"), M, split, tile_m, ctypes.c_void_p(st.cuda_stream)),
           "tm_w8a8_gemm_f16")
    return out
