"""The token sample of the full-size layer parity tests (`parity_tokens`):
it must hold every row where a GEMM tile of the layer changes."""

import numpy as np
import pytest

import oracle
from tests.gpu_helpers import parity_tokens


def _routing(T, E, k, rng, skew=0.0):
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits += (skew * np.log1p(np.arange(E))[::-1]).astype(np.float32)[None, :]
    return oracle.route_ref(logits, k)[0]


@pytest.mark.parametrize("T,E,k,shared,skew", [
    (2048, 32, 8, False, 0.0),     # ~512 rows per expert: 64-row boundaries
    (1500, 64, 6, True, 3.0),      # skewed, with a shared expert
    (300, 128, 4, False, 0.0),     # ~9 rows per expert: 16-row boundaries
])
def test_sample_covers_tile_boundaries(rng, T, E, k, shared, skew):
    ids = _routing(T, E, k, rng, skew)
    tok = parity_tokens(ids, E, shared, n_min=256, seed=1)
    assert np.all(np.diff(tok) > 0) and tok[0] >= 0 and tok[-1] < T
    assert len(tok) >= min(T, 256)
    _, offsets, s2f, _ = oracle.permute_ref(ids, E)
    step = 16 if T * k <= 32 * E else 64
    have = set(tok.tolist())
    for g in range(E):
        a, b = offsets[g], offsets[g + 1]
        must = [a, b - 1] if b > a else []
        for m in range(a + step, b, step):
            must += [m - 1, m]
        for s in must:
            assert s2f[s] // k in have, (g, s)
    if shared:
        assert {0, T - 1, step - 1, step} <= have


def test_sample_is_all_tokens_for_small_batches(rng):
    ids = _routing(100, 16, 2, rng)
    assert np.array_equal(parity_tokens(ids, 16, True, n_min=256), np.arange(100))


def test_bf16_half_ulp_bounds_the_rounding(rng):
    """bf16_half_ulp(v) is the largest move of rounding v to bf16: torch's
    round-to-nearest-even never exceeds it, and a value half-way between two
    bf16 numbers reaches it exactly."""
    import torch
    from tests.gpu_helpers import bf16_half_ulp
    v = rng.standard_normal(200_000) * np.exp2(rng.integers(-20, 20, 200_000))
    r = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
    v32 = v.astype(np.float32).astype(np.float64)
    assert np.all(np.abs(r - v32) <= bf16_half_ulp(v32))
    mid = np.array([1.0 + 2.0 ** -8, 3.0 + 2.0 ** -7, -0.75 - 2.0 ** -9])
    assert np.allclose(bf16_half_ulp(mid), [2.0 ** -8, 2.0 ** -7, 2.0 ** -9])
    r_mid = torch.from_numpy(mid).to(torch.bfloat16).double().numpy()
    assert np.array_equal(np.abs(r_mid - mid), bf16_half_ulp(mid))
    assert bf16_half_ulp(np.array([0.0]))[0] == 0.0
