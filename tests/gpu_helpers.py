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


def bf16_half_ulp(v):
    """Half the spacing of bfloat16 numbers (8 significant bits) at |v|: the
    most that rounding v to the nearest bf16 can move it (0 at 0)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (np.maximum(e, -126) - 8).astype(np.int64)), 0.0)


def layer_tolerance_ok(gpu, ref):
    """The layer's accuracy contract on its bf16 output against the oracle's
    exact (fp64) output `ref`:

        max_i (|gpu_i - ref_i| - h_i) <= 2e-2 * rms(ref)
        sum_i |gpu_i - ref_i| / sum_i |ref_i| <= 5e-3

    h_i is half a bf16 ulp at the larger of |gpu_i| and |ref_i|: the layer's
    output is one rounding to bf16 of the fp32 sum, and that rounding alone
    moves an element by up to h_i (relative 2^-9 to 2^-8) whatever the
    arithmetic before it. On a large sample a few elements lie beyond 5 rms,
    where h_i by itself exceeds 2e-2 rms, so the max bound is applied to the
    error beyond the output format's own rounding. The L1 bound is applied to
    the whole error. Returns (ok, max excess / rms, L1 ratio, raw max / rms)."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    excess = err - bf16_half_ulp(np.maximum(np.abs(gpu), np.abs(ref)))
    rms = np.sqrt(np.mean(ref ** 2))
    l1 = err.sum() / max(np.abs(ref).sum(), 1e-300)
    return (excess.max() <= 2e-2 * rms and l1 <= 5e-3, excess.max() / rms, l1,
            err.max() / rms)


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


def parity_tokens(ids, E, shared, n_min=256, seed=0):
    """Tokens whose outputs the full-size layer tests compare with the oracle.

    Every output row depends only on its own token once the routing is fixed,
    so a large batch is checked on a sample of tokens. The sample is aimed at
    the rows where the GEMM tiles change, taken from the layer's own
    permutation (counting sort of the routed ids, expert-contiguous rows):

    * the first and the last row of every expert that has rows;
    * both rows on either side of every tile boundary inside an expert's
      slice: every 64 rows (which covers the 64-, 128- and 256-row token
      tiles and the 256-token CTA-pair tiles), or every 16 rows when the
      experts average at most 32 rows (the 16- and 32-row tiles);
    * for the shared expert (one row per token, group E after the routed
      rows): the first and last token, and the tokens on either side of its
      first four and last four tile boundaries;

    then seeded random tokens until there are at least n_min (or all T).
    Returns the sorted token indices."""
    ids = np.asarray(ids)
    T, k = ids.shape
    _, offsets, s2f, _ = oracle.permute_ref(ids, E)
    R = T * k
    step = 16 if R <= 32 * E else 64
    rows = set()
    for g in range(E):
        a, b = int(offsets[g]), int(offsets[g + 1])
        if b <= a:
            continue
        rows.update((a, b - 1))
        for m in range(a + step, b, step):
            rows.update((m - 1, m))
    toks = {int(s2f[s]) // k for s in rows}
    if shared and T > 0:
        toks.update((0, T - 1))
        bounds = list(range(step, T, step))
        for m in bounds[:4] + bounds[-4:]:
            toks.update((m - 1, m))
    want = min(T, n_min)
    if len(toks) < want:
        rng = np.random.default_rng(seed)
        rest = np.setdiff1d(np.arange(T), np.fromiter(toks, np.int64))
        toks.update(int(t) for t in rng.choice(rest, want - len(toks), replace=False))
    return np.array(sorted(toks), dtype=np.int64)
