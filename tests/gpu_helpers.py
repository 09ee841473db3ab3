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
      tiles), or every 16 rows when the experts average at most 32 rows (the
      16- and 32-row tiles), and the boundaries of the CTA-pair kernels'
      balanced tiles (an expert of r rows cut into t = ceil(r / bn) tiles of
      32 * ceil(ceil(r / t) / 32) rows, bn = 192 or 256);
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
        r = b - a
        for bn in (192, 256):
            t = -(-r // bn)
            w = (-(-r // t) + 31) // 32 * 32
            for m in range(a + w, b, w):
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


def swiglu_bound(g, u, abs_g, abs_u, K):
    """Bound on |h_gpu - h| for h = silu(g) u computed by the gate/up GEMM's
    epilogue from fp32 g and u (each within gemm_bound of the exact value):
    first-order propagation of the two GEMM errors, plus the fp32 evaluation
    with the fast exponential and division (CUDA documents at most
    2 + floor(1.173 |x|) ulp for __expf(x) and 2 ulp for __fdividef in this
    range) and the scaling multiplies."""
    eg = gemm_bound(abs_g, K)
    eu = gemm_bound(abs_u, K)
    sig = oracle.sigmoid_ref(g)
    silu = g * sig
    dsilu = np.abs(sig * (1 + g * (1 - sig)))
    ulps = 16 + 2 + np.floor(1.173 * np.abs(g))
    return dsilu * np.abs(u) * eg + np.abs(silu) * eu + ulps * U32 * np.abs(silu * u) + 1e-30


def staged_layer_check(cfg, xv, out_tokens, ids, w, inter, tokens, qmap, w_g):
    """Stage-by-stage parity of one forward on the sampled `tokens`, read
    from the forward's own intermediates (moe_forward_intermediates):

    * x codes and scale at each of the sample's rows: bit-exact against the
      oracle's quantiser on the layer input xv;
    * h of every row of the sample: within the fp32 GEMM + SwiGLU bound of
      the oracle's exact h;
    * the requantisation is an integer decision taken in fp32: the oracle
      takes it on the GPU's own fp32 h, and codes and scales must then match
      bit for bit;
    * y: within the fp32 accumulation bound (plus the fp16 encoding's
      rounding) of the oracle's down GEMM on those codes;
    * out: the accuracy contract (layer_tolerance_ok) against the oracle's
      combine of that y, in fp64 with one bf16 rounding.

    `ids` / `w`: the routing (oracle's, equal to the GPU's on these tokens);
    `qmap[e]`: the oracle-quantised weights of expert e (E: the shared
    expert), `w_g` the shared gate vector or None. Returns the contract's
    (max excess / rms, L1 ratio, raw max / rms)."""
    T, D, E, k, I = cfg.T, cfg.D, cfg.E, cfg.k, cfg.I
    R = T * k
    tokens = np.asarray(tokens, np.int64)
    n = tokens.size
    f2s = inter["flat_to_sorted"].cpu().numpy().astype(np.int64).reshape(T, k)
    rows = f2s[tokens]                                   # [n, k]
    experts = np.asarray(ids)[tokens].astype(np.int64)   # [n, k]
    flat_rows = rows.ravel()
    flat_exp = experts.ravel()
    flat_tok = np.repeat(np.arange(n), k)
    if cfg.shared:
        flat_rows = np.concatenate([flat_rows, R + tokens])
        flat_exp = np.concatenate([flat_exp, np.full(n, E)])
        flat_tok = np.concatenate([flat_tok, np.arange(n)])
    dev_rows = torch.as_tensor(flat_rows, device=inter["h"].device)
    h_g = inter["h"].index_select(0, dev_rows).cpu().numpy()
    hq_g = inter["hq"].index_select(0, dev_rows).cpu().numpy()
    sh_g = inter["sh"].index_select(0, dev_rows).cpu().numpy()
    sx_g = inter["sx"].index_select(0, dev_rows).cpu().numpy()
    xq_g = inter["xq"].index_select(0, dev_rows).cpu().numpy()
    y_g = inter["y"].index_select(0, dev_rows).double()
    if inter["y_fp16"]:
        rs = inter["y_row_scale"].index_select(0, dev_rows).double()
        y_g = y_g * rs[:, None]
        rs = rs.cpu().numpy()
    y_g = y_g.cpu().numpy()

    xq_o, sx_o = oracle.quant_rows_ref(np.asarray(xv, np.float32)[tokens])
    assert np.array_equal(xq_g, xq_o[flat_tok]), "x codes differ"
    assert np.array_equal(sx_g.view(np.uint32), sx_o[flat_tok].view(np.uint32)), \
        "x scales differ"

    y_al = np.zeros((flat_rows.size, D))
    for e in np.unique(flat_exp):
        sel = np.flatnonzero(flat_exp == e)
        wgu, sgu, wd, sd = qmap[int(e)]
        xr, sr = xq_o[flat_tok[sel]], sx_o[flat_tok[sel]]
        gu = oracle.ptpc_matmul_ref(xr, sr, wgu, sgu)
        absgu = (np.abs(oracle.e4m3_decode(xr)) @ np.abs(oracle.e4m3_decode(wgu)).T) * \
            sr[:, None].astype(np.float64) * sgu[None, :].astype(np.float64)
        g, u = gu[:, :I], gu[:, I:]
        h64 = oracle.silu_ref(g) * u
        hb = swiglu_bound(g, u, absgu[:, :I], absgu[:, I:], D)
        err = np.abs(h_g[sel].astype(np.float64) - h64)
        bad = err > hb
        assert not bad.any(), ("h", int(e), np.argwhere(bad)[:3], err[bad][:3], hb[bad][:3])
        hq_o, sh_o, y64 = oracle.down_from_h_ref(h_g[sel], wd, sd)
        assert np.array_equal(hq_o, hq_g[sel]), ("h codes", int(e))
        assert np.array_equal(sh_o.view(np.uint32), sh_g[sel].view(np.uint32)), \
            ("h scales", int(e))
        absy = (np.abs(oracle.e4m3_decode(hq_o)) @ np.abs(oracle.e4m3_decode(wd)).T) * \
            sh_o[:, None].astype(np.float64) * sd[None, :].astype(np.float64)
        yb = gemm_bound(absy, I) + 1e-30
        if inter["y_fp16"]:
            yb = yb * (1 + 1e-3) + np.abs(y64) * (2.0 ** -11 + 4 * U32) + \
                rs[sel, None] * 2.0 ** -25
        err = np.abs(y_g[sel] - y64)
        bad = err > yb
        assert not bad.any(), ("y", int(e), np.argwhere(bad)[:3], err[bad][:3], yb[bad][:3])
        y_al[sel] = y64

    w = np.asarray(w, np.float64)[tokens]                 # [n, k]
    out_al = (w[:, :, None] * y_al[:n * k].reshape(n, k, D)).sum(axis=1)
    if cfg.shared:
        gate = oracle.shared_gate_ref(np.asarray(xv, np.float64)[tokens], w_g)
        out_al = out_al + gate[:, None] * y_al[n * k:]
    ok, max_rel, l1, raw = layer_tolerance_ok(out_tokens, out_al)
    assert ok, (f"{cfg.name}: against the oracle on the GPU's requant decisions: "
                f"max excess/rms {max_rel:.3e} (raw {raw:.3e}), L1 ratio {l1:.3e}")
    return max_rel, l1, raw
