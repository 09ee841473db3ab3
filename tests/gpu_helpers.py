"""Shared pieces of the GPU parity tests: device checks, error bounds, and the
oracle's per-expert work in a spawn-started process pool."""

import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import oracle

# fp32 unit roundoff
U32 = 2.0 ** -24


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def ensure_library():
    from expert_layer_ptpc_gb300 import binding, build
    build.build()
    return binding.load_library()


def gemm_bound(abs_acc, K, extra_ulps=4):
    """Bound on |fp32 result - exact| for a scaled dot product of K exact
    products accumulated in fp32: K roundings of partial sums (each at most
    u * sum|terms|) plus a few roundings of the scaling."""
    return (K * U32 + extra_ulps * U32) * abs_acc


def layer_tolerance_ok(gpu, ref):
    """The layer's accuracy contract: max|gpu - oracle| <= 2e-2 * rms(oracle)
    and sum|gpu - oracle| / sum|oracle| <= 5e-3."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    rms = np.sqrt(np.mean(ref ** 2))
    l1 = err.sum() / max(np.abs(ref).sum(), 1e-300)
    return err.max() <= 2e-2 * rms and l1 <= 5e-3, err.max() / rms, l1


def _quantize_expert(args):
    wgu, wd = args
    return oracle.quantize_expert_ref(wgu, wd)


_POOL = None


def oracle_pool():
    """A process pool for the oracle, started with 'spawn' so it never forks a
    process that holds a CUDA context."""
    global _POOL
    if _POOL is None:
        n = max(1, min(16, (os.cpu_count() or 2) - 1))
        _POOL = mp.get_context("spawn").Pool(n)
    return _POOL


def quantize_experts(raw_pairs):
    """Oracle-quantised weights for a list of (W_gu, W_d) fp32 numpy pairs."""
    if len(raw_pairs) <= 1:
        return [_quantize_expert(p) for p in raw_pairs]
    return oracle_pool().map(_quantize_expert, raw_pairs, chunksize=1)
