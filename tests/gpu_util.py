"""Helpers shared by the GPU tests: cached synthetic problems on the device and
the oracle comparison."""
import functools

import numpy as np
import torch

import oracle
from w4a16_quantized_gemm_gb300 import binding, synth

TOL = 2e-3  # max|Y - Y_ref| / max|Y_ref|, fp32 accumulation


@functools.lru_cache(maxsize=8)
def host_weights(K, N, g, stress=False, seed=0):
    return synth.weights(K, N, g, stress, seed)


@functools.lru_cache(maxsize=4)
def packed(K, N, g, stress=False, seed=0):
    q, z, s, _ = host_weights(K, N, g, stress, seed)
    qd = torch.from_numpy(q).cuda()
    zd = torch.from_numpy(z).cuda()
    sd = torch.from_numpy(s.view(np.uint16)).cuda().view(torch.float16)
    w = binding.pack(qd, zd, sd, g)
    del qd, zd, sd
    return w


def activations(M, K, N, g, stress=False, seed=0):
    sal = host_weights(K, N, g, stress, seed)[3]
    return synth.activations(M, K, sal, seed, tag=f"/N{N}/g{g}" + ("/stress" if stress else ""))


def sample_rows(M, n=32, seed=0):
    """All rows for M <= 256; else a seeded subset plus the first and last rows."""
    if M <= 256:
        return list(range(M))
    r = np.argsort(synth.draws(synth.stream_key(f"rows/{M}/{seed}"), M), kind="stable")[:n]
    return sorted(set(int(v) for v in r) | {0, M - 1})


def run_and_compare(M, K, N, g, stress=False, config=None, rows=None, seed=0, X=None):
    w = packed(K, N, g, stress, seed)
    if X is None:
        X = activations(M, K, N, g, stress, seed)
    Xd = torch.from_numpy(X.view(np.uint16)).cuda().view(torch.float16)
    Y = binding.gemm(Xd, w, config=config)
    torch.cuda.synchronize()
    assert binding.device_error(clear=True) == 0
    rows = sample_rows(M) if rows is None else rows
    q, z, s, _ = host_weights(K, N, g, stress, seed)
    Y_ref = oracle.gemm(X, q, z, s, g, rows=rows)
    Yh = Y[torch.tensor(rows, device=Y.device)].float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(Yh))
    err = oracle.rel_max_err(Yh, Y_ref)
    return err, Y
