"""The checked build (libmoe_ptpc_check.so, -DMOE_CHECK) in place of a memory
checker: every data-dependent index (expert ids, row maps, destination rows)
is validated where it is used, and a bad one sets bit 128 of the error word
and skips the access instead of reading or writing out of bounds.

* Forwards through the checked build report no check bit and give outputs
  identical, bit for bit, to the normal build's (the checks change no
  arithmetic).
* Expert ids out of range, handed to the checked build's permutation, are
  reported (MOE_ERR_INVALID_ARG, bit 128) and skipped: nothing faults and the
  context stays usable. The normal build never sees such ids here.

The checked library runs in a child process (one library per process)."""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from tests.gpu_helpers import require_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    ("c1", 300, 512, 16, 4, 256, True),
    ("c2", 1024, 1024, 16, 8, 256, True),     # fp16 y, CTA pairs
    ("c3", 9000, 256, 8, 2, 128, False),      # multi-block permutation
    ("c4", 16, 4096, 128, 8, 1536, False),    # decode-shaped tiles
]

CHILD = r'''
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
from expert_layer_ptpc_gb300 import binding, build
from expert_layer_ptpc_gb300 import synthetic as syn
from expert_layer_ptpc_gb300.layer import MoELayer
build.build(variant=sys.argv[2])
outs = {}
for name, T, D, E, k, I, shared in CASES:
    cfg = syn.LayerConfig(name, T, D, E, k, I, shared, "normal")
    L = MoELayer.synthetic(cfg, "cuda", 0)
    x, lg = syn.gen_x(cfg, "cuda", 0), syn.gen_logits(cfg, "cuda", 0)
    out = L.forward(x, lg)
    st = L.status()
    assert st == (0, 0), (name, st)
    outs[name] = out.view(torch.int16).cpu().numpy()
if sys.argv[2] == "check":
    # ids out of range: reported and skipped
    ids = torch.randint(0, 16, (64, 4), dtype=torch.int32, device="cuda")
    ids[3, 1] = 16
    ids[40, 0] = -2
    binding.moe_permute(ids, 16)
    st = binding.moe_device_status()
    assert st[0] == -1 and st[1] & 128, st
    assert binding.moe_device_status() == (0, 0)
    ok_ids = torch.randint(0, 16, (64, 4), dtype=torch.int32, device="cuda")
    binding.moe_permute(ok_ids, 16)
    assert binding.moe_device_status() == (0, 0)
np.savez(sys.argv[3], **outs)
'''


def _run(variant, path):
    code = "CASES = " + repr(CASES) + "\n" + CHILD
    env = dict(os.environ, MOE_LIBRARY_VARIANT=variant)
    r = subprocess.run([sys.executable, "-c", code, ROOT, variant, path], env=env,
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    return np.load(path)


def test_checked_build_matches_and_catches_bad_ids(tmp_path):
    require_gpu()
    checked = _run("check", str(tmp_path / "check.npz"))
    normal = _run("", str(tmp_path / "normal.npz"))
    for name, *_ in CASES:
        assert np.array_equal(checked[name], normal[name]), name
