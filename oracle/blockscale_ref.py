"""FP8 with per-K-block scales: BlockScale-128 and 512-subchannel, the two
alternatives the PTPC grouped GEMM is compared against.

TEST INFRASTRUCTURE ONLY. This module is part of the reference the CUDA path
is checked against; it shares no code with that path and never calls it.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import it.

Sources:
* "Ultimate Latency Optimization of Qwen3 and Qwen3-VL on AMD MI300X Series"
  (LMSYS), section 2.1.1: BlockScale FP8 ties its scales to a fixed block
  size along K, which the hardware GEMM tile then has to respect; PTPC has
  no such block and was measured 15-30% faster.
* The SGLang / AMD page on DeepSeek-R1 disaggregated inference on MI355X,
  "MoRI Quantized All-to-All" section: FP8 blockwise quantisation uses one
  fp32 scale per 128 elements; its "FlyDSL FusedMoE" section tunes an A8W8
  blockscale GEMM for the expert shapes.
* "Optimizing Qwen 3.5 397B MoE on Ironwood TPU7x" (Google Developers Blog),
  GMM V2 paragraph: FP8 activations quantised per 512-wide subchannel.

None of the pages writes the formats out. The readings taken here:

* Quantiser: the PTPC one (moe_ref.quant_rows_ref) applied to a block,
  s = fp32(max(amax_block, 1e-12) / 448), codes = e4m3(fp32(v / s)).
* BlockScale-128 activations: a 1 x 128 block along K per row, scales
  [rows, K / 128]. Weights W[N, K]: 128 x 128 blocks, scales
  [N / 128, K / 128] (the DeepSeek-V3 layout the MI355X page's model uses).
* 512-subchannel: activations in 1 x 512 blocks along K, scales
  [rows, K / 512]; the page names only the activations, so the weights keep
  their PTPC per-output-channel scales [N].
* GEMM: each block's FP8 dot product is exact (products of e4m3 values are
  multiples of 2^-18 below 2^17, and a block of up to 512 sums to under
  2^27 of those units), and is scaled by its two scales:
      block-128:  y[r, n] = sum_b sa[r, b] * sw[n // 128, b] * P_b[r, n]
      sub-512:    y[r, n] = sw[n] * sum_g sa[r, g] * P_g[r, n]
  where P_b[r, n] = sum over k in block b of qa[r, k] * qw[n, k]. The scaled
  sum over blocks is taken in fp64.
"""

import numpy as np

from .fp8 import e4m3_decode
from .moe_ref import quant_rows_ref

BLOCK_K = 128          # BlockScale block along K (activations and weights)
BLOCK_N = 128          # BlockScale weight block along N
SUBCHANNEL_K = 512     # subchannel width along K (activations only)


def quant_blocks_ref(v, block):
    """Quantise each row of v [R, K] in 1 x `block` pieces along K (K a
    multiple of block). Returns (codes uint8 [R, K], scales fp32
    [R, K // block]); scales[r, b] belongs to v[r, b*block:(b+1)*block]."""
    v32 = np.asarray(v, dtype=np.float32)
    R, K = v32.shape
    if K % block:
        raise ValueError("K must be a multiple of the block")
    nb = K // block
    codes, scales = quant_rows_ref(v32.reshape(R * nb, block))
    return codes.reshape(R, K), scales.reshape(R, nb)


def quant_weight_blocks_ref(w, bn=BLOCK_N, bk=BLOCK_K):
    """Quantise W [N, K] in bn x bk blocks (N, K multiples of them). Returns
    (codes uint8 [N, K], scales fp32 [N // bn, K // bk]); scales[i, b]
    belongs to W[i*bn:(i+1)*bn, b*bk:(b+1)*bk]."""
    w32 = np.asarray(w, dtype=np.float32)
    N, K = w32.shape
    if N % bn or K % bk:
        raise ValueError("N and K must be multiples of the block")
    nn, nk = N // bn, K // bk
    # one row per block, holding that block's bn * bk entries
    blocks = w32.reshape(nn, bn, nk, bk).transpose(0, 2, 1, 3).reshape(nn * nk, bn * bk)
    codes, scales = quant_rows_ref(blocks)
    codes = codes.reshape(nn, nk, bn, bk).transpose(0, 2, 1, 3).reshape(N, K)
    return codes, scales.reshape(nn, nk)


def block_partials_ref(a_codes, w_codes, block):
    """P[b, r, n] = exact sum over k in block b of a[r, k] * w[n, k] (fp64;
    exact, see the module docstring)."""
    a = e4m3_decode(a_codes)
    w = e4m3_decode(w_codes)
    K = a.shape[1]
    return np.stack([a[:, b:b + block] @ w[:, b:b + block].T
                     for b in range(0, K, block)])


def blockscale_matmul_ref(a_codes, a_scale, w_codes, w_scale):
    """BlockScale-128: y[r, n] = sum_b a_scale[r, b] * w_scale[n // 128, b] *
    P_b[r, n] (fp64). a_scale [R, K/128], w_scale [N/128, K/128]."""
    P = block_partials_ref(a_codes, w_codes, BLOCK_K)
    sa = np.asarray(a_scale, np.float64)            # [R, nb]
    sw = np.repeat(np.asarray(w_scale, np.float64), BLOCK_N, axis=0)   # [N, nb]
    y = np.zeros(P.shape[1:], np.float64)
    for b in range(P.shape[0]):
        y += sa[:, b][:, None] * sw[:, b][None, :] * P[b]
    return y


def subchannel_matmul_ref(a_codes, a_scale, w_codes, w_scale, block=SUBCHANNEL_K):
    """512-subchannel: y[r, n] = w_scale[n] * sum_g a_scale[r, g] * P_g[r, n]
    (fp64). a_scale [R, K/block], w_scale [N] (per output channel)."""
    P = block_partials_ref(a_codes, w_codes, block)
    sa = np.asarray(a_scale, np.float64)
    y = np.zeros(P.shape[1:], np.float64)
    for g in range(P.shape[0]):
        y += sa[:, g][:, None] * P[g]
    return y * np.asarray(w_scale, np.float64)[None, :]


def grouped_blockscale_ref(a_codes, a_scale, w_codes, w_scale, offsets, mode, rows=None):
    """The grouped GEMM over experts: group g owns rows
    [offsets[g], offsets[g+1]) and multiplies them by its own W[g].
    mode "block128": w_codes [G, N, K], w_scale [G, N/128, K/128];
    mode "sub512": w_scale [G, N]. `rows`: evaluate only these rows (sorted
    row indices), returning y for them in that order."""
    offsets = np.asarray(offsets, np.int64)
    R = a_codes.shape[0]
    N = w_codes.shape[1]
    want = np.arange(R) if rows is None else np.asarray(rows, np.int64)
    y = np.full((len(want), N), np.nan)
    for g in range(len(offsets) - 1):
        lo, hi = offsets[g], offsets[g + 1]
        sel = np.flatnonzero((want >= lo) & (want < hi))
        if sel.size == 0:
            continue
        r = want[sel]
        if mode == "block128":
            y[sel] = blockscale_matmul_ref(a_codes[r], a_scale[r], w_codes[g], w_scale[g])
        elif mode == "sub512":
            y[sel] = subchannel_matmul_ref(a_codes[r], a_scale[r], w_codes[g], w_scale[g])
        else:
            raise ValueError(mode)
    return y
