"""The byte counts bench.py reports (host arithmetic, no GPU)."""
import numpy as np
import pytest

import bench
from expert_layer_ptpc_gb300 import synthetic as syn


def _configs():
    out = [syn.CONFIGS[n] for n in ("tiny", "decode", "prefill", "skewed")]
    return out + [syn.sweep_config(T) for T in syn.SWEEP_T]


@pytest.mark.parametrize("cfg", _configs(), ids=lambda c: c.name)
def test_implementation_bytes_cover_the_algorithmic_bytes(cfg):
    """Every byte the layer must move (weights, x, out, router input) is
    among the bytes its launches move; the intermediates come on top."""
    rng = np.random.default_rng(0)
    for touched_frac in (1.0, 0.3):
        counts = (rng.random(cfg.E) < touched_frac).astype(np.int64)
        B, touched = bench.algorithmic_bytes(cfg, counts)
        assert bench.implementation_bytes(cfg, touched) >= B


@pytest.mark.parametrize("cfg", _configs(), ids=lambda c: c.name)
def test_prenorm_adds_the_residual_traffic(cfg):
    """The pre-norm forward reads the residual and gamma and writes the new
    residual: 2 T D bf16 reads and writes plus D bf16 of gamma."""
    counts = np.ones(cfg.E, dtype=np.int64)
    _, touched = bench.algorithmic_bytes(cfg, counts)
    extra = bench.implementation_bytes(cfg, touched, pre=True) - \
        bench.implementation_bytes(cfg, touched)
    assert extra == 2 * cfg.T * cfg.D * 2 + 2 * cfg.D

