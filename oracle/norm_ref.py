"""Add + RMSNorm + per-token FP8 quantisation, the op that produces the MoE
layer's FP8 input straight from the residual stream.

TEST INFRASTRUCTURE ONLY. This module is part of the reference the CUDA path
is checked against; it shares no code with that path and never calls it.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import it.

"Ultimate Latency Optimization of Qwen3 and Qwen3-VL on AMD MI300X Series"
(LMSYS), section 2.1.5 and its fusion table: AllReduce + AddRMSNorm +
per-token quant run as one fused operator in front of the MoE block. On one
GPU there is nothing to all-reduce, and the op is, per token t,

    r_t = x_t + res_t                              the updated residual stream
    v_t = r_t / sqrt(mean_d(r_t[d]^2) + eps) * gamma
    (codes_t, s_t) = the PTPC quantisation of v_t  (moe_ref.quant_rows_ref)

The page gives no formulas. The readings taken here, in the order of the
steps:

* r_t is rounded once to bf16, the residual stream's type:
  r = bf16_rne(fp32(x) + fp32(res)).
* The mean square is ms = fp32(S / D), where S = sum_d r[d]^2 is the exact
  sum of the exact squares (math.fsum of fp64 squares of bf16 values) and
  S / D is one fp64 division.
* inv = the correctly rounded fp32 value of 1 / sqrt(fp32(ms + eps)): one
  fp32 addition, then the exact reciprocal square root rounded once.
* v = fp32(fp32(r * inv) * gamma), two fp32 multiplications. v is not
  rounded to bf16; the quantiser takes it as it is, since that is where the
  code decision is made.
* The shared-expert gate, when present, is sigmoid(sum_d v[d] * w_g[d]).
"""

import math
from decimal import Context, Decimal

import numpy as np

from .fp8 import bf16_round
from .moe_ref import quant_rows_ref, sigmoid_ref


def rsqrt_f32_rn(a):
    """The fp32 number nearest to 1 / sqrt(a) for an fp32 a > 0 (ties to even,
    which cannot occur for fp32 inputs). The exact value is taken to 60
    decimal digits, and the nearest of three fp32 candidates around a
    first guess is chosen."""
    a = float(np.float32(a))
    if a <= 0.0:
        raise ValueError("rsqrt of a non-positive value")
    ctx = Context(prec=60)
    exact = ctx.divide(Decimal(1), ctx.sqrt(Decimal(a)))
    guess = np.float32(1.0 / math.sqrt(a))
    cands = [np.nextafter(guess, np.float32(0.0)), guess,
             np.nextafter(guess, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(Decimal(float(c)) - exact),
                                     int(np.float32(c).view(np.uint32)) & 1))
    return np.float32(best)


def add_rmsnorm_ref(x, res, gamma, eps):
    """r = bf16(x + res) and v = fp32(fp32(r * inv) * gamma) per row, with the
    readings above. x, res [T, D] and gamma [D] hold bf16 values (any float
    dtype). Returns (r fp32 holding bf16 values, v fp32, inv fp32 [T])."""
    x32 = np.asarray(x, dtype=np.float32)
    res32 = np.asarray(res, dtype=np.float32)
    g32 = np.asarray(gamma, dtype=np.float32)
    T, D = x32.shape
    r = bf16_round((x32 + res32).astype(np.float64))     # fp32 add, bf16 RNE
    v = np.empty((T, D), np.float32)
    inv = np.empty(T, np.float32)
    eps32 = np.float32(eps)
    for t in range(T):
        sq = [float(q) * float(q) for q in r[t]]           # exact in fp64
        ms = np.float32(math.fsum(sq) / D)
        inv[t] = rsqrt_f32_rn(np.float32(ms + eps32))
        v[t] = (r[t] * inv[t]).astype(np.float32) * g32
    return r, v, inv


def add_rmsnorm_quant_ref(x, res, gamma, eps, w_g=None):
    """The whole fused op for every row. Returns a dict with
    r (the new residual, bf16 values in fp32), v, codes [T, D] uint8,
    scales [T] fp32 and, when w_g [D] is given, gate [T] (fp64)."""
    r, v, inv = add_rmsnorm_ref(x, res, gamma, eps)
    codes, scales = quant_rows_ref(v)
    out = {"r": r, "v": v, "inv": inv, "codes": codes, "scales": scales}
    if w_g is not None:
        out["gate"] = sigmoid_ref(v.astype(np.float64) @
                                  np.asarray(w_g, dtype=np.float64))
    return out
