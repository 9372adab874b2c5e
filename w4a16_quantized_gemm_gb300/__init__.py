"""W4A16 mixed-precision GEMM for GB300 (sm_103a).

``Y[M,N] = X[M,K] . dequant(W)`` with 4-bit codes, a 4-bit zero and an fp16
scale per (group of g along K, column).  The computation lives in the CUDA
library ``libtm_w4a16.so`` (C ABI in ``include/tm_w4a16.h``); this package is
its Python binding plus the seeded synthetic-input generator.
"""
from .binding import (GemmConfig, PackedWeights, TMError, device_error, gemm, last_launch_count, load,
                      pack, packed_bytes, plan, status_str)

__all__ = ["GemmConfig", "PackedWeights", "TMError", "device_error", "gemm", "last_launch_count", "load",
           "pack", "packed_bytes", "plan", "status_str"]
