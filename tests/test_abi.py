"""The C-ABI library builds, loads without a GPU, and exports every entry point
include/moe_ptpc.h declares; host-side argument checks answer without
touching the device."""

import ctypes
import os
import re

import pytest

from expert_layer_ptpc_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include",
                      "moe_ptpc.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def test_header_declares_the_api():
    names = _declared()
    for n in ["moe_route", "moe_permute", "moe_quant_ptpc", "moe_grouped_gemm",
              "moe_combine", "moe_forward"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_covers_the_header(lib):
    assert binding.exported_names() == _declared()


def test_status_strings(lib):
    assert binding.status_string(0) == "ok"
    assert "workspace" in binding.status_string(-4)
    assert lib.moe_version() >= 100


def test_argument_errors_need_no_gpu(lib):
    # invalid k, E too large, misaligned / null pointers: rejected on the host
    assert lib.moe_route(None, 4, 8, 0, 1, None, None, None) == -1
    assert lib.moe_route(None, 4, 2048, 2, 1, None, None, None) == -2
    assert lib.moe_route(None, 0, 8, 2, 1, None, None, None) == 0   # empty
    assert lib.moe_quant_ptpc(None, 0, 4, 100, None, 1, -1, None, None,
                              None) == -1                          # cols % 16
    assert lib.moe_grouped_gemm(0, None, None, 8, None, None, None, 2, 100,
                                256, None, 1, 0, None) == -2       # N % 128
    d = binding.make_dims(16, 4096, 128, 8, 1536, False)
    need = lib.moe_forward_workspace_size(ctypes.byref(d))
    assert need > 16 * 8 * 4
    bad = binding.make_dims(16, 4000, 128, 8, 1536, False)
    assert lib.moe_forward_workspace_size(ctypes.byref(bad)) == 0
    assert lib.moe_forward(ctypes.byref(bad), *([None] * 12), 0, None) == -2
    # the fp16 encoding of y: shapes and pointer sets checked on the host
    assert lib.moe_scale_max(None, -1, 4, None, None) == -1
    assert lib.moe_scale_max(None, 0, 4, None, None) == 0        # no groups
    assert lib.moe_grouped_gemm_down_f16(None, None, 8, None, None, None, None,
                                         2, 100, 256, None, None, 0, None) == -2
    fake16 = ctypes.c_void_p(0x1000)
    assert lib.moe_combine_f16(fake16, fake16, fake16, fake16, 4, 2, 256, fake16,
                               None, None, fake16, None) == -1    # partial shared set
    # the fused router: E > 512, k > 16 or D % 64 go to the unfused ops
    assert lib.moe_router_topk(None, None, 4, 4096, 1024, 8, 1, None, None, None,
                               None) == -2
    assert lib.moe_router_topk(None, None, 4, 4096, 128, 17, 1, None, None, None,
                               None) == -2
    assert lib.moe_router_topk(None, None, 4, 4096, 8, 9, 1, None, None, None,
                               None) == -1                       # k > E
    # block-scaled path: block sizes, kinds and shapes checked on the host
    assert lib.moe_quant_blocks(None, 4, 256, 64, None, None, None) == -1     # block 64
    assert lib.moe_quant_blocks(None, 4, 640, 512, None, None, None) == -1    # K % 512
    assert lib.moe_quant_blocks(None, 0, 256, 128, None, None, None) == 0     # empty
    assert lib.moe_quant_weight_blocks(None, 100, 256, None, None, None) == -1
    assert lib.moe_quant_weight_blocks(None, 128 * 65536, 128, fake16, fake16,
                                       None) == -2
    assert lib.moe_grouped_gemm_scaled(3, None, None, 8, None, None, None, 2, 128,
                                       256, None, None) == -1             # unknown kind
    assert lib.moe_grouped_gemm_scaled(1, None, None, 8, None, None, None, 2, 128,
                                       640, None, None) == -2             # K % 512
    assert lib.moe_grouped_gemm_scaled(2, None, None, 8, None, None, None, 2, 100,
                                       256, None, None) == -2             # N % 128
    assert lib.moe_grouped_gemm_scaled(2, None, None, 0, None, None, None, 2, 128,
                                       256, None, None) == 0              # no rows
    # the failure-detection check validates its limit before touching CUDA
    assert lib.moe_debug_expire_wait(0, None, 0, None) == -1
    assert lib.moe_debug_expire_wait(2000000, None, 0, None) == -1
    # a forward workspace smaller than its error word is refused, unlaunched
    fake16 = ctypes.c_void_p(0x1000)
    assert lib.moe_debug_expire_wait(10, fake16, 128, None) == -1
    assert lib.moe_workspace_status(None, 1024, None, None) == -1
    assert lib.moe_workspace_status(fake16, 255, None, None) == -1
    assert lib.moe_workspace_status(ctypes.c_void_p(0x1008), 4096, None, None) == -1
    # workspace too small is reported before any launch
    fake = ctypes.c_void_p(0x1000)
    rc = lib.moe_forward(ctypes.byref(d), fake, fake, None, fake, fake, fake,
                         fake, None, fake, None, None, fake, 16, None)
    assert rc == -4


def test_permute_workspace_size(lib):
    assert lib.moe_permute_workspace_size(16, 128, 8) == 0          # one block
    assert lib.moe_permute_workspace_size(1024, 128, 8) == 0        # 8192 entries
    # one int histogram row per chunk of 2048 flat entries (ragged last chunk)
    assert lib.moe_permute_workspace_size(8192, 128, 8) == 32 * 128 * 4
    assert lib.moe_permute_workspace_size(1025, 128, 8) == 5 * 128 * 4


@pytest.mark.parametrize("dims_args", [(64, 256, 8, 2, 128, 0), (1000, 1024, 16, 8, 256, 1),
                                       (16384, 4096, 512, 10, 1024, 1), (1, 128, 1, 1, 128, 0)])
def test_workspace_layout_has_guard_bands(lib, dims_args):
    """Sub-buffers of the forward workspace are disjoint, in order, 256-byte
    aligned, each followed by at least 256 guard bytes, inside the size
    moe_forward_workspace_size reports."""
    from expert_layer_ptpc_gb300 import binding
    d = binding.make_dims(*dims_args)
    lay = binding.moe_forward_workspace_layout(d)
    total = lib.moe_forward_workspace_size(ctypes.byref(d))
    assert len(lay) >= 10
    ends = [o for o, _ in lay[1:]] + [total]
    for (o, n), nxt in zip(lay, ends):
        assert o % 256 == 0 and o + n + 256 <= nxt, (o, n, nxt)


def test_checked_build_exports_the_same_symbols():
    """The checked variant (-DMOE_CHECK) compiles and exports exactly the
    header's entry points, like the normal library."""
    import subprocess
    lib = build.build(variant="check")
    out = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True,
                         text=True, check=True).stdout
    names = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert {n for n in names if n.startswith("moe_")} == set(binding.exported_names())


_SINGLE_LAUNCH_PROBE = r"""
import sys
sys.path.insert(0, {root!r})
from expert_layer_ptpc_gb300 import binding as B
q = B.moe_forward_single_launch
print(int(q(B.make_dims(1, 4096, 512, 10, 1024, 1, 1))),           # the T=1 sweep point
      int(q(B.make_dims(4, 1024, 128, 6, 512, 1, 0))),             # four tokens
      int(q(B.make_dims(5, 1024, 128, 6, 512, 1, 1))),             # five: chained
      int(q(B.make_dims(1, 4096, 512, 10, 1024, 1, 1), router_weights=True)),
      int(q(B.make_dims(1, 4096, 512, 10, 1024, 1, 1), prenorm=True)),
      int(q(B.make_dims(4, 8192, 64, 4, 512, 0, 1))))              # x rows too long
"""


@pytest.mark.parametrize("mode,expect", [(None, "0 0 0 0 0 0"), ("1", "1 1 0 0 0 0")])
def test_single_launch_rule_needs_no_gpu(lib, mode, expect):
    """moe_forward_single_launch answers on the host: the one-launch forward
    is off unless MOE_SMALL_FORWARD=1, and then applies to at most 4 tokens
    on given logits without pre-norm, on shapes whose x and h rows fit its
    buffers (child processes: the switch is read once)."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    env.pop("MOE_SMALL_FORWARD", None)
    if mode is not None:
        env["MOE_SMALL_FORWARD"] = mode
    r = subprocess.run([sys.executable, "-c", _SINGLE_LAUNCH_PROBE.format(root=root)],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.split() == expect.split()
    bad = binding.make_dims(1, 100, 8, 2, 128, 0, 1)     # D not a multiple of 128
    assert lib.moe_forward_single_launch(ctypes.byref(bad), 0, 0) < 0
