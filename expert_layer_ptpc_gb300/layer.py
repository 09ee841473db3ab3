"""One MoE layer's device state: PTPC-quantised weights and a reusable
workspace, with `forward` calling the library's moe_forward.

Weights are quantised on the GPU by moe_quant_ptpc, one scale per output
channel (per row of W_gu [2I, D] and of W_d [D, I]).
"""

import torch

from . import binding
from . import synthetic as syn


class MoELayer:
    def __init__(self, cfg, w_gu, s_gu, w_d, s_d, router_w=None,
                 shared_gate_w=None):
        self.cfg = cfg
        self.w_gu, self.s_gu, self.w_d, self.s_d = w_gu, s_gu, w_d, s_d
        self.router_w = router_w
        self.shared_gate_w = shared_gate_w
        self._ws = None

    @classmethod
    def synthetic(cls, cfg, device="cuda", seed=0):
        """Seeded random weights of `cfg`, quantised on the device."""
        G, I, D = cfg.groups, cfg.I, cfg.D
        w_gu = torch.empty((G, 2 * I, D), dtype=torch.uint8, device=device)
        s_gu = torch.empty((G, 2 * I), dtype=torch.float32, device=device)
        w_d = torch.empty((G, D, I), dtype=torch.uint8, device=device)
        s_d = torch.empty((G, D), dtype=torch.float32, device=device)
        for e in range(G):
            raw_gu, raw_d = syn.gen_expert_weights(cfg, e, device, seed)
            binding.moe_quant_ptpc(raw_gu, out_q=w_gu[e], out_scale=s_gu[e])
            binding.moe_quant_ptpc(raw_d, out_q=w_d[e], out_scale=s_d[e])
        router_w = (syn.gen_router_weights(cfg, device, seed)
                    if cfg.router == "weights" else None)
        gate_w = syn.gen_shared_gate(cfg, device, seed) if cfg.shared else None
        return cls(cfg, w_gu, s_gu, w_d, s_d, router_w, gate_w)

    def dims(self, T):
        c = self.cfg
        return binding.make_dims(T, c.D, c.E, c.k, c.I, c.shared, c.renormalize)

    def workspace(self, T):
        need = max(binding.moe_forward_workspace_size(self.dims(T)), 1)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.w_gu.device)
            self._ws[:min(need, 256)].zero_()   # the forward's error word
        return self._ws

    def status(self, stream=None):
        """(status, error bits) of the most recent forward on this layer's
        workspace (read and cleared; synchronises the stream)."""
        if self._ws is None:
            return 0, 0
        return binding.moe_workspace_status(self._ws, stream)

    def forward(self, x, router_logits=None, out=None, topk_ids=None,
                topk_w=None, stream=None, events=None, residual=None, gamma=None,
                eps=1e-6, residual_out=None):
        """The layer on x (bf16 [T, D]); with `residual` and `gamma` on
        RMSNorm(x + residual) * gamma, the new residual written to
        `residual_out` (default: in place). The pre-normed form needs
        router_logits."""
        T = x.shape[0]
        router_w = self.router_w
        if router_w is not None and residual is None:
            router_logits = None
        elif residual is not None:
            router_w = None
        return binding.moe_forward(
            self.dims(T), x, self.w_gu, self.s_gu, self.w_d, self.s_d,
            router_logits=router_logits, router_w=router_w,
            shared_gate_w=self.shared_gate_w, out=out, ws=self.workspace(T),
            topk_ids=topk_ids, topk_w=topk_w, stream=stream, events=events,
            residual=residual, gamma=gamma, eps=eps, residual_out=residual_out)
