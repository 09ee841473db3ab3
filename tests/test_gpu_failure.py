"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes expires, the kernel ends normally, the host reads the expiry from
moe_device_status(), and the context stays usable."""

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
