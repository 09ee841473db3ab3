"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes expires, the kernel ends normally, the host reads the expiry from
moe_device_status() (standalone steps) or moe_workspace_status() (a forward's
own workspace), and the context stays usable."""

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_helpers import ensure_library, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    require_gpu()
    ensure_library()


def test_expired_wait_is_reported_and_cleared():
    from expert_layer_ptpc_gb300 import binding as B
    assert B.moe_device_status() == (0, 0)
    B.moe_debug_expire_wait(20000)            # 20 ms limit
    st, bits = B.moe_device_status()
    assert st == -5 and bits & 64, (st, bits)
    assert B.moe_device_status() == (0, 0)    # read once, then cleared


def test_context_usable_after_an_expired_wait():
    from expert_layer_ptpc_gb300 import binding as B
    B.moe_debug_expire_wait(5000)
    assert B.moe_device_status()[0] == -5
    g = torch.Generator().manual_seed(3)
    logits = torch.randn(257, 64, generator=g)
    ids, w = B.moe_route(logits.cuda(), 6)
    assert B.moe_device_status() == (0, 0)
    rid, rw = oracle.route_ref(logits.numpy(), 6)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=1e-5, atol=0)


def test_workspace_errors_stay_with_their_workspace():
    """Two forwards on two streams, each with its own workspace: a bounded
    wait that expires on one stream's workspace is reported there exactly
    once, and neither the other workspace nor the device word sees it."""
    from expert_layer_ptpc_gb300 import binding as B
    from expert_layer_ptpc_gb300 import synthetic as syn
    from expert_layer_ptpc_gb300.layer import MoELayer
    cfg = syn.LayerConfig("ws_err", 256, 512, 16, 4, 256, True, "normal")
    L = MoELayer.synthetic(cfg, "cuda", 0)
    x, lg = syn.gen_x(cfg, "cuda", 0), syn.gen_logits(cfg, "cuda", 0)
    dims = L.dims(cfg.T)
    need = B.moe_forward_workspace_size(dims)
    ws = [torch.empty(need, dtype=torch.uint8, device="cuda") for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for i in range(2):
        outs.append(B.moe_forward(dims, x, L.w_gu, L.s_gu, L.w_d, L.s_d,
                                  router_logits=lg, shared_gate_w=L.shared_gate_w,
                                  ws=ws[i], stream=streams[i]))
    B.moe_debug_expire_wait(20000, ws=ws[0], stream=streams[0])   # 20 ms limit
    st1, bits1 = B.moe_workspace_status(ws[1], streams[1])
    st0, bits0 = B.moe_workspace_status(ws[0], streams[0])
    assert (st1, bits1) == (0, 0)
    assert st0 == -5 and bits0 == 64, (st0, bits0)
    assert B.moe_workspace_status(ws[0], streams[0]) == (0, 0)   # exactly once
    assert B.moe_device_status() == (0, 0)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_forward_clears_its_workspace_word():
    """A forward starts from a clear error word: an expiry recorded in a
    workspace before the forward is not reported after it."""
    from expert_layer_ptpc_gb300 import binding as B
    from expert_layer_ptpc_gb300 import synthetic as syn
    from expert_layer_ptpc_gb300.layer import MoELayer
    cfg = syn.LayerConfig("ws_clr", 64, 256, 8, 2, 128, False, "normal")
    L = MoELayer.synthetic(cfg, "cuda", 0)
    x, lg = syn.gen_x(cfg, "cuda", 0), syn.gen_logits(cfg, "cuda", 0)
    ws = L.workspace(cfg.T)
    B.moe_debug_expire_wait(2000, ws=ws)
    L.forward(x, lg)
    assert L.status() == (0, 0)
