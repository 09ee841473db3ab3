"""moe_permute_noalloc, the permutation entry point for callers that cannot
allocate device memory (a host framework that has reserved the device memory
in its own arena, or a serving loop that may not call cudaMalloc/cudaFree
because they synchronise the device). It uses a fixed scratch array inside
the library instead of a workspace argument.

Checked through the C ABI against moe_permute (which takes a caller-supplied
workspace): the permutation is integer work, so the outputs must be equal bit
for bit, on two calls in a row with different routings, and on a routing big
enough to use the scratch (more than one 8192-entry chunk)."""

import ctypes

import numpy as np
import pytest
import torch

from tests.gpu_helpers import ensure_library, require_gpu

pytestmark = pytest.mark.gpu


def _routing(T, E, k, seed):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:, : E // 3] -= 8.0          # some experts empty
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    return torch.from_numpy(order.astype(np.int32)).cuda()


def _outputs(T, E, k):
    dev = "cuda"
    return (torch.full((E,), -7, dtype=torch.int32, device=dev),
            torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
            torch.full((T * k,), -7, dtype=torch.int32, device=dev),
            torch.full((T * k,), -7, dtype=torch.int32, device=dev))


def _call_noalloc(lib, ids, E, outs):
    T, k = ids.shape
    c, o, s2f, f2s = outs
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.moe_permute_noalloc(
        ctypes.c_void_p(ids.data_ptr()), T, E, k,
        ctypes.c_void_p(c.data_ptr()), ctypes.c_void_p(o.data_ptr()),
        ctypes.c_void_p(s2f.data_ptr()), ctypes.c_void_p(f2s.data_ptr()), stream)


@pytest.mark.parametrize("T,E,k", [(20000, 256, 4), (16, 128, 8),
                                   (40000, 1024, 10)])
def test_noalloc_permute_matches_workspace_version(T, E, k):
    require_gpu()
    lib = ensure_library()
    from expert_layer_ptpc_gb300 import binding
    for call, seed in enumerate((T, T + 1)):      # two calls in a row
        ids = _routing(T, E, k, seed)
        outs = _outputs(T, E, k)
        assert _call_noalloc(lib, ids, E, outs) == 0
        ref = binding.moe_permute(ids, E)
        st, bits = binding.moe_device_status()
        assert st == 0, bits
        for got, want in zip(outs, ref):
            assert torch.equal(got, want), f"call {call}"


def test_noalloc_permute_rejects_oversize():
    require_gpu()
    lib = ensure_library()
    # 1 MiB of scratch holds 256 histogram rows of E = 1024: at most 256
    # chunks of 2048 flat entries; one token more is refused
    E, k = 1024, 8
    T = 256 * 2048 // k + 1
    rc = lib.moe_permute_noalloc(ctypes.c_void_p(16), T, E, k,
                                 ctypes.c_void_p(16), ctypes.c_void_p(16),
                                 ctypes.c_void_p(16), ctypes.c_void_p(16), None)
    assert rc == -2
