"""Grouped FP8 GEMMs with PTPC, 512-subchannel or BlockScale-128 scales, on the
library's one block-scaled engine (moe_grouped_gemm_scaled): quantisation of
weights and activations on the GPU, the GEMM, and a synthetic grouped problem
of a layer workload for comparing the three.

"Ultimate Latency Optimization of Qwen3 and Qwen3-VL on AMD MI300X Series",
section 2.1.1, compares PTPC with BlockScale FP8 (per-128 fp32 scales, the
MI355X DeepSeek-R1 page's "MoRI Quantized All-to-All" section); the Ironwood
TPU page's GMM V2 paragraph quantises activations per 512-wide subchannel.
"""

import torch

from . import binding
from . import synthetic as syn

KINDS = {"ptpc": binding.MOE_SCALE_PTPC, "sub512": binding.MOE_SCALE_SUB512,
         "block128": binding.MOE_SCALE_BLOCK128}


def quantize_weights(mode, w, q=None, s=None):
    """w [G, N, K] fp32 -> (codes [G, N, K], scales): BlockScale-128 in
    128 x 128 blocks [G, N/128, K/128]; otherwise per output channel [G, N]."""
    G, N, K = w.shape
    if mode == "block128":
        q, s = binding.moe_quant_weight_blocks(w, q=q, scales=s)
        return q, s.view(G, N // 128, K // 128)
    q2 = None if q is None else q.view(G * N, K)
    s2 = None if s is None else s.view(G * N)
    q2, s2 = binding.moe_quant_ptpc(w.view(G * N, K), out_q=q2, out_scale=s2)
    return q2.view(G, N, K), s2.view(G, N)


def quantize_activations(mode, x, q=None, s=None):
    """x [R, K] bf16 -> (codes [R, K], scales): per token [R] (PTPC), or per
    1 x 512 ([R, K/512]) or 1 x 128 ([R, K/128]) piece along K."""
    if mode == "ptpc":
        return binding.moe_quant_ptpc(x, out_q=q, out_scale=s)
    return binding.moe_quant_blocks(x, 512 if mode == "sub512" else 128, q=q, scales=s)


def grouped_gemm(mode, qa, sa, qw, sw, offsets, out=None, stream=None):
    return binding.moe_grouped_gemm_scaled(KINDS[mode], qa, sa, qw, sw, offsets,
                                           out=out, stream=stream)


def make_problem(mode, cfg, which="gateup", seed=0, device="cuda"):
    """The grouped GEMM of one layer workload with `mode` scales:
    which="gateup": the token rows of x (bf16) in expert order, routed by the
      workload's seeded logits, times each expert's W_gu [2I, D];
    which="down": R = T k rows of N(0, 1) bf16 activations [R, I] in the same
      groups, times each expert's W_d [D, I].
    Weights and activations are quantised on the device. Returns a dict with
    the operands, the output buffer and accessors of the raw inputs."""
    T, D, E, k, I = cfg.T, cfg.D, cfg.E, cfg.k, cfg.I
    logits = syn.gen_logits(cfg, device, seed)
    ids, _ = binding.moe_route(logits, k, cfg.renormalize)
    _, offsets, s2f, _ = binding.moe_permute(ids, E)
    R = T * k
    if which == "gateup":
        x = syn.gen_x(cfg, device, seed)
        a = x[(s2f // k).long()]                   # row r holds its token's x
        N, K = 2 * I, D
    else:
        a = syn._normal((R, I), 1.0, device, seed, f"hdown/{cfg.name}").to(torch.bfloat16)
        N, K = D, I
    qw = torch.empty((E, N, K), dtype=torch.uint8, device=device)
    sw = (torch.empty((E, N // 128, K // 128), dtype=torch.float32, device=device)
          if mode == "block128" else
          torch.empty((E, N), dtype=torch.float32, device=device))

    def w_raw_dev(e):
        gu, dn = syn.gen_expert_weights(cfg, e, device, seed)
        return gu if which == "gateup" else dn

    for e in range(E):
        quantize_weights(mode, w_raw_dev(e)[None], q=qw[e:e + 1], s=sw[e:e + 1])
    qa, sa = quantize_activations(mode, a)
    out = torch.empty((R, N), dtype=torch.float32, device=device)
    return {"mode": mode, "offsets": offsets, "qa": qa, "sa": sa, "qw": qw, "sw": sw,
            "out": out, "a": a,
            "x_rows": lambda rows: a[torch.as_tensor(rows, device=device).long()]
            .float().cpu().numpy(),
            "w_raw": lambda e: w_raw_dev(e).cpu().numpy()}


def run(prob, stream=None):
    return grouped_gemm(prob["mode"], prob["qa"], prob["sa"], prob["qw"], prob["sw"],
                        prob["offsets"], out=prob["out"], stream=stream)
