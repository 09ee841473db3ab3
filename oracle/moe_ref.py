"""Slow, plain CPU oracle of the PTPC-FP8 Mixture-of-Experts layer forward.

TEST INFRASTRUCTURE ONLY. This module is the reference that the CUDA path is
checked against; it shares no code with that path and never calls it. Only
the tests, the smoke check and the benchmark's CPU-baseline leg may import it.

What the layer computes, and where the pages say so:

* Layer structure - "Optimizing Qwen 3.5 397B MoE on Ironwood TPU7x" (Google
  Developers Blog), MoE paragraph of the model description: a router gate
  projects each token, a softmax over experts picks the top-k routed experts,
  and one shared expert runs on every token.
* Permute / unpermute - same page, the SparseCore paragraphs: token rows are
  gathered into expert-contiguous rows without padding, and after the expert
  GEMMs an indirect gather plus local reduction brings them back per token.
* Expert FFN - same page, the GMM V2 paragraph: gate and up projections are
  packed in one grouped GEMM with SwiGLU fused, then the down projection.
* PTPC quantisation - "Ultimate Latency Optimization of Qwen3 and Qwen3-VL on
  AMD MI300X Series" (LMSYS), section 2.1.1 and Figure 3: per-token scales for
  activations, per-output-channel scales for weights, FP8 values.
* Routing metadata - the TPU page's expert-parallel paragraph: expert indices
  (int) and top-k weights (float) are two arrays of shape [tokens, k].
* Routing precision - the TPU page's Numerical Verification Layer paragraph:
  gating is checked against an fp32 reference, so selection uses fp32 logits.

Readings taken where the pages are silent:

* top-k weights are the softmax over all experts restricted to the chosen k and
  renormalised to sum to 1, i.e. a softmax over the k chosen logits;
  selection is on the fp32 logits, ties go to the lower expert index;
* a token's FP8 scale is s = fp32(max(amax, 1e-12) / 448) and its codes are
  e4m3(fp32(v / s)): the quantiser takes its decisions in fp32, the precision
  of the kernel that takes them, with IEEE division;
* the SwiGLU output h is rounded to fp32 before its per-row requantisation
  (the GPU keeps h in fp32; that rounding is where both sides take the
  decision), every other step runs in fp64;
* rows inside one expert keep ascending flat index f = t*k + j (stable);
* the shared expert is group E with the same intermediate size I, gated by
  sigmoid(x . w_g), and fed the same per-token FP8 x;
* the output is one bf16 rounding (nearest even) of the fp64 sum.

Exactness of the contractions: an e4m3 value is a multiple of 2**-9 with at
most 4 significant bits, so each product of two is a multiple of 2**-18 below
448**2 < 2**18 in magnitude, and a sum of up to 2**14 such products needs at
most 18 + 18 + 14 = 50 < 53 bits. The fp64 matrix products of decoded codes
below are therefore exact in any summation order.
"""

import numpy as np

from .fp8 import bf16_round, e4m3_decode, e4m3_encode

QUANT_EPS = np.float32(1e-12)
FP8_MAX = np.float32(448.0)


# ---------------------------------------------------------------------------
# router
# ---------------------------------------------------------------------------
def router_logits_ref(x, w_r):
    """logits[t, e] = x[t] . w_r[e], summed in fp64, rounded once to fp32.

    The router gate projection of the TPU page's MoE paragraph. `x` [T, D] and
    `w_r` [E, D] hold bf16 values (given as fp32 arrays).
    """
    x64 = np.asarray(x, dtype=np.float64)
    w64 = np.asarray(w_r, dtype=np.float64)
    return (x64 @ w64.T).astype(np.float32)


def route_ref(logits, k, renormalize=True):
    """Top-k expert selection and weights for each token.

    Selection: the k largest fp32 logits, ties broken by the lower expert
    index (a stable sort of the negated logits). Weights: the softmax
    probabilities of the chosen experts, renormalised over the k of them when
    `renormalize` (which equals a softmax over the k chosen logits), or the
    plain softmax probabilities over all E experts otherwise. fp64 throughout.

    Returns ids [T, k] int32 (in selection order) and weights [T, k] fp64.
    """
    lg = np.asarray(logits, dtype=np.float32)
    T, E = lg.shape
    if not 1 <= k <= E:
        raise ValueError("k out of range")
    order = np.argsort(-lg, axis=1, kind="stable")
    ids = order[:, :k].astype(np.int32)
    chosen = np.take_along_axis(lg, ids.astype(np.int64), axis=1).astype(np.float64)
    if renormalize:
        m = chosen[:, :1]
        p = np.exp(chosen - m)
        w = p / p.sum(axis=1, keepdims=True)
    else:
        all64 = lg.astype(np.float64)
        m = all64.max(axis=1, keepdims=True)
        z = np.exp(all64 - m).sum(axis=1, keepdims=True)
        w = np.exp(chosen - m) / z
    return ids, w


# ---------------------------------------------------------------------------
# permutation into expert-contiguous rows
# ---------------------------------------------------------------------------
def permute_ref(ids, E):
    """Counting sort of the flat (token, slot) pairs by expert.

    Flat index f = t * k + j. counts[e] = number of f routed to e; offsets is
    the exclusive prefix sum of counts (E + 1 entries); within one expert the
    rows keep ascending f. sorted_to_flat[s] is the flat index stored at
    sorted row s, flat_to_sorted[f] the sorted row of flat index f.
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    R = flat.size
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = offsets[:E].copy()
    sorted_to_flat = np.empty(R, dtype=np.int64)
    flat_to_sorted = np.empty(R, dtype=np.int64)
    for f in range(R):
        e = flat[f]
        s = cursor[e]
        cursor[e] += 1
        sorted_to_flat[s] = f
        flat_to_sorted[f] = s
    return (counts.astype(np.int32), offsets.astype(np.int32),
            sorted_to_flat.astype(np.int32), flat_to_sorted.astype(np.int32))


# ---------------------------------------------------------------------------
# PTPC quantisation
# ---------------------------------------------------------------------------
def quant_rows_ref(v):
    """Per-row FP8 e4m3 quantisation (per token for activations, per output
    channel for a weight matrix stored [N, K]).

    s = fp32(max(amax, 1e-12) / 448); codes = e4m3(fp32(v / s)); both
    divisions are IEEE fp32 divisions. Returns (codes uint8, scales fp32).
    """
    v32 = np.asarray(v, dtype=np.float32)
    amax = np.max(np.abs(v32), axis=1)
    scale = (np.maximum(amax, QUANT_EPS) / FP8_MAX).astype(np.float32)
    ratio = (v32 / scale[:, None]).astype(np.float32)
    return e4m3_encode(ratio), scale


def dequant_rows_ref(codes, scales):
    """Value of quantised rows: e4m3 value times the row's scale (fp64)."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[:, None]


def ptpc_matmul_ref(a_codes, a_scale, w_codes, w_scale):
    """out[r, n] = a_scale[r] * w_scale[n] * sum_k a[r, k] * w[n, k].

    The PTPC identity of section 2.1.1 of the LMSYS page: with one scale per
    row of A and one per row of W (output channel), the dequantisation is a
    rank-1 scaling of the exact FP8 dot products. The dot products are exact
    in fp64 (module docstring).
    """
    acc = e4m3_decode(a_codes) @ e4m3_decode(w_codes).T
    return acc * np.asarray(a_scale, np.float64)[:, None] * \
        np.asarray(w_scale, np.float64)[None, :]


def silu_ref(g):
    """silu(g) = g * sigmoid(g) = g / (1 + exp(-g)), fp64."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def sigmoid_ref(z):
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def expert_ffn_ref(xq, sx, wgu_codes, sgu, wd_codes, sd):
    """One expert on its rows: gate/up GEMM, SwiGLU, requant, down GEMM.

    wgu_codes [2I, K=D]: rows 0..I-1 gate, rows I..2I-1 up (both K-contiguous);
    wd_codes [D, I]. Returns a dict with h (fp64), h rounded to fp32, the
    requantised h (codes, scales) and y (fp64, [rows, D]).
    """
    I = wgu_codes.shape[0] // 2
    gu = ptpc_matmul_ref(xq, sx, wgu_codes, sgu)
    g, u = gu[:, :I], gu[:, I:]
    h = silu_ref(g) * u
    h32 = h.astype(np.float32)
    hq, sh, y = down_from_h_ref(h32, wd_codes, sd)
    return {"g": g, "u": u, "h": h, "h32": h32, "hq": hq, "sh": sh, "y": y}


def down_from_h_ref(h32, wd_codes, sd):
    """The expert's steps after SwiGLU, from fp32 h [rows, I]: per-row FP8
    requantisation (PTPC, per token), then the down GEMM against
    wd_codes [D, I] with its per-channel scales. Returns (hq, sh, y fp64)."""
    hq, sh = quant_rows_ref(h32)
    y = ptpc_matmul_ref(hq, sh, wd_codes, sd)
    return hq, sh, y


# ---------------------------------------------------------------------------
# the whole layer
# ---------------------------------------------------------------------------
def shared_gate_ref(x, w_g):
    """sigmoid(x[t] . w_g) per token, fp64 (x and w_g hold bf16 values)."""
    return sigmoid_ref(np.asarray(x, np.float64) @ np.asarray(w_g, np.float64))


def moe_forward_ref(x, k, expert_weights, E, logits=None, router_w=None,
                    w_g=None, renormalize=True, tokens=None):
    """The layer forward, step by step.

    x: [T, D] bf16 values (fp32 array). Exactly one of `logits` [T, E] fp32 and
    `router_w` [E, D] bf16 values is given. expert_weights(e) returns the
    quantised weights (wgu_codes, sgu, wd_codes, sd) of expert e, with e == E
    the shared expert (present when w_g is given).

    `tokens`: optional subset of token indices whose outputs are computed;
    routing and permutation always cover all T tokens. Every output row
    depends only on its own token once the routing is fixed, so the subset
    gives the same values as the full run.

    Returns a dict with the routing, the permutation, the quantised x, and
    `out` (bf16 values as fp32, rows for `tokens` in order) and `out64`.
    """
    x32 = np.asarray(x, dtype=np.float32)
    T, D = x32.shape
    if (logits is None) == (router_w is None):
        raise ValueError("give exactly one of logits and router_w")
    if logits is None:
        logits = router_logits_ref(x32, router_w)
    logits = np.asarray(logits, dtype=np.float32)
    ids, w = route_ref(logits, k, renormalize)
    counts, offsets, s2f, f2s = permute_ref(ids, E)
    xq, sx = quant_rows_ref(x32)
    gate = shared_gate_ref(x32, w_g) if w_g is not None else None

    sel = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    out64 = np.zeros((sel.size, D), dtype=np.float64)
    # Group the requested (token, slot) pairs by expert, run each expert once.
    pairs = {}
    for n, t in enumerate(sel):
        for j in range(k):
            pairs.setdefault(int(ids[t, j]), []).append((n, int(t), j))
    for e in sorted(pairs):
        wgu, sgu, wd, sd = expert_weights(e)
        rows = np.array([t for _, t, _ in pairs[e]], dtype=np.int64)
        r = expert_ffn_ref(xq[rows], sx[rows], wgu, sgu, wd, sd)
        for i, (n, t, j) in enumerate(pairs[e]):
            out64[n] += w[t, j] * r["y"][i]
    if gate is not None:
        wgu, sgu, wd, sd = expert_weights(E)
        r = expert_ffn_ref(xq[sel], sx[sel], wgu, sgu, wd, sd)
        out64 += gate[sel][:, None] * r["y"]
    return {
        "logits": logits, "ids": ids, "w": w, "counts": counts,
        "offsets": offsets, "sorted_to_flat": s2f, "flat_to_sorted": f2s,
        "xq": xq, "sx": sx, "gate": gate, "tokens": sel,
        "out64": out64, "out": bf16_round(out64),
    }


def moe_flops(T, D, E, k, I, shared):
    """Algorithmic FLOPs of the expert GEMMs (2 per multiply-add)."""
    rows = T * k + (T if shared else 0)
    return 2.0 * rows * D * (2 * I) + 2.0 * rows * I * D


def quantize_expert_ref(w_gu, w_d):
    """PTPC weight quantisation of one expert: per output channel = per row
    of W_gu [2I, D] and of W_d [D, I]."""
    wgu, sgu = quant_rows_ref(w_gu)
    wd, sd = quant_rows_ref(w_d)
    return wgu, sgu, wd, sd


__all__ = [
    "router_logits_ref", "route_ref", "permute_ref", "quant_rows_ref",
    "dequant_rows_ref", "ptpc_matmul_ref", "silu_ref", "sigmoid_ref",
    "expert_ffn_ref", "down_from_h_ref", "shared_gate_ref", "moe_forward_ref",
    "moe_flops",
    "quantize_expert_ref",
]
