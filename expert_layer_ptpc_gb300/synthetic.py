"""Seeded synthetic inputs for the MoE layer: token activations, router logits
or router weights, raw (unquantised) expert weights and the shared-expert gate.

This module only draws random numbers; it holds none of the layer's
arithmetic. Both the CUDA path and the oracle are fed from it. Every tensor
comes from its own torch.Generator, seeded from (seed, tensor name, expert
index), so an expert's weights can be regenerated alone and in any order.
Tensors are generated on the requested device; the same device gives the same
numbers on every run.

Layer shapes follow the pages' Qwen3 / Qwen3.5 MoE layers ("Optimizing Qwen 3.5
397B MoE on Ironwood TPU7x": D = 4096, 512 experts of I = 1024, top-10 plus one
shared expert; "Ultimate Latency Optimization of Qwen3 and Qwen3-VL on AMD
MI300X Series": Qwen3-235B, 128 experts, top-8, I = 1536).
"""

import hashlib
import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class LayerConfig:
    """Dimensions and input recipe of one MoE layer workload.

    T tokens of hidden size D, E routed experts of intermediate size I, top-k
    routing, optional shared expert (intermediate size I, sigmoid-gated).
    `router` picks the logit recipe: "weights" (bf16 router matrix, logits
    computed by the layer), "normal" (N(0,1) logits), "normal_bias" (N(0,1)
    plus a per-expert N(0, 0.5) bias) or "zipf" (Zipf(1.1) expert popularity).
    `t_draw` is the token count the x / logits streams are drawn for; smaller
    T take its first rows, so a token-count sweep shares inputs.
    """
    name: str
    T: int
    D: int
    E: int
    k: int
    I: int
    shared: bool
    router: str
    renormalize: bool = True
    t_draw: int = 0

    @property
    def rows(self):
        """Permuted rows: T*k routed plus T shared."""
        return self.T * self.k + (self.T if self.shared else 0)

    @property
    def groups(self):
        return self.E + (1 if self.shared else 0)

    def with_tokens(self, T):
        return replace(self, T=T, name=f"{self.name.split('@')[0]}@T={T}")


SWEEP_T = (1, 64, 512, 4096, 16384)

CONFIGS = {
    # T=64, D=256, E=8, top-2, I=128, router projection from bf16 weights.
    "tiny": LayerConfig("tiny", 64, 256, 8, 2, 128, False, "weights"),
    # Qwen3-235B-like decode step: 16 tokens, weight streaming.
    "decode": LayerConfig("decode", 16, 4096, 128, 8, 1536, False, "normal"),
    # Qwen3-235B-like prefill chunk: 8192 tokens, mild expert imbalance.
    "prefill": LayerConfig("prefill", 8192, 4096, 128, 8, 1536, False,
                           "normal_bias"),
    # Skewed routing with a shared expert.
    "skewed": LayerConfig("skewed", 4096, 2048, 256, 8, 512, True, "zipf"),
    # Qwen3.5-397B-like layer; T swept over SWEEP_T with shared draws.
    "sweep": LayerConfig("sweep", 16384, 4096, 512, 10, 1024, True, "normal",
                         t_draw=16384),
}


def sweep_config(T):
    return CONFIGS["sweep"].with_tokens(T)


def _seed(seed, tag, index=0):
    h = hashlib.sha256(f"{seed}:{tag}:{index}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed, tag, index=0):
    g = torch.Generator(device=device)
    g.manual_seed(_seed(seed, tag, index))
    return g


def _normal(shape, std, device, seed, tag, index=0):
    g = _gen(device, seed, tag, index)
    return torch.randn(shape, generator=g, device=device,
                       dtype=torch.float32) * std


def gen_x(cfg, device="cpu", seed=0):
    """Token activations x [T, D], N(0, 1), rounded to bf16."""
    t = max(cfg.T, cfg.t_draw)
    x = _normal((t, cfg.D), 1.0, device, seed, f"x/{cfg.name.split('@')[0]}")
    return x[:cfg.T].to(torch.bfloat16).contiguous()


def gen_router_weights(cfg, device="cpu", seed=0):
    """Router gate matrix W_r [E, D], N(0, 0.02), bf16."""
    w = _normal((cfg.E, cfg.D), 0.02, device, seed, f"wr/{cfg.name}")
    return w.to(torch.bfloat16).contiguous()


def gen_logits(cfg, device="cpu", seed=0):
    """Router logits [T, E] fp32 for the "normal", "normal_bias" and "zipf"
    recipes. Zipf: expert popularity ranks are a seeded permutation of 1..E
    and expert e's logits are shifted by log(rank_e**-1.1 / H), H the
    normaliser sum_r r**-1.1, so the softmax prior follows Zipf(1.1)."""
    base = cfg.name.split("@")[0]
    t = max(cfg.T, cfg.t_draw)
    z = _normal((t, cfg.E), 1.0, device, seed, f"logits/{base}")[:cfg.T]
    if cfg.router == "normal":
        out = z
    elif cfg.router == "normal_bias":
        b = _normal((cfg.E,), 0.5, device, seed, f"bias/{base}")
        out = z + b[None, :]
    elif cfg.router == "zipf":
        g = _gen("cpu", seed, f"zipf/{base}")
        rank = (torch.randperm(cfg.E, generator=g) + 1).to(torch.float64)
        harmonic = sum(r ** -1.1 for r in range(1, cfg.E + 1))
        prior = torch.log(rank ** -1.1 / harmonic).to(torch.float32)
        out = z + prior.to(device)[None, :]
    else:
        raise ValueError(f"router recipe {cfg.router!r} has no logits")
    return out.contiguous()


def gen_expert_weights(cfg, e, device="cpu", seed=0):
    """Raw fp32 weights of expert e (e == E is the shared expert).

    W_gu [2I, D]: rows 0..I-1 the gate projection, rows I..2I-1 the up
    projection; W_d [D, I]. Both N(0, 1/sqrt(D)), stored with the reduction
    dimension contiguous (one row per output channel).
    """
    base = cfg.name.split("@")[0]
    std = 1.0 / math.sqrt(cfg.D)
    wgu = _normal((2 * cfg.I, cfg.D), std, device, seed, f"wgu/{base}", e)
    wd = _normal((cfg.D, cfg.I), std, device, seed, f"wd/{base}", e)
    return wgu, wd


def gen_shared_gate(cfg, device="cpu", seed=0):
    """Shared-expert gate vector w_g [D], N(0, 0.02), bf16."""
    base = cfg.name.split("@")[0]
    w = _normal((cfg.D,), 0.02, device, seed, f"wg/{base}")
    return w.to(torch.bfloat16).contiguous()
