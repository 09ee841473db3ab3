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


def _oracle_intermediates(cfg, x, ids, qmap, wg):
    """A forward's intermediates as the oracle computes them, laid out like
    the library's workspace (rows in sorted, expert-contiguous order)."""
    import torch
    T, D, E, k, I = cfg.T, cfg.D, cfg.E, cfg.k, cfg.I
    R = T * k
    rows = R + (T if cfg.shared else 0)
    _, offsets, s2f, f2s = oracle.permute_ref(ids, E)
    xq, sx = oracle.quant_rows_ref(x)
    h = np.zeros((rows, I), np.float32)
    srow_tok = np.concatenate([s2f // k, np.arange(T)]) if cfg.shared else s2f // k
    srow_exp = np.concatenate([ids.ravel()[s2f], np.full(T, E)]) if cfg.shared \
        else ids.ravel()[s2f]
    y = np.zeros((rows, D))
    hq = np.zeros((rows, I), np.uint8)
    sh = np.zeros(rows, np.float32)
    for e in np.unique(srow_exp):
        sel = np.flatnonzero(srow_exp == e)
        r = oracle.expert_ffn_ref(xq[srow_tok[sel]], sx[srow_tok[sel]], *qmap[int(e)])
        h[sel], hq[sel], sh[sel], y[sel] = r["h32"], r["hq"], r["sh"], r["y"]
    t = torch.from_numpy
    return {"flat_to_sorted": t(f2s.astype(np.int32)), "xq": t(xq[srow_tok]),
            "sx": t(sx[srow_tok]),
            "h": t(h), "hq": t(hq), "sh": t(sh), "y": t(y.astype(np.float32)),
            "y_fp16": False}


def test_staged_check_accepts_the_oracle_and_catches_a_wrong_code():
    """The staged layer comparison of the GPU tests, run on the CPU with the
    oracle's own intermediates standing in for the GPU's: it passes them, and
    fails when one requantised code, one h value or one output is wrong."""
    from expert_layer_ptpc_gb300 import synthetic as syn
    from tests.gpu_helpers import staged_layer_check
    cfg = syn.LayerConfig("cpu_staged", 40, 256, 8, 2, 128, True, "normal")
    rng = np.random.default_rng(5)
    x = oracle.bf16_round(rng.standard_normal((cfg.T, cfg.D))).astype(np.float32)
    logits = rng.standard_normal((cfg.T, cfg.E)).astype(np.float32)
    ids, w = oracle.route_ref(logits, cfg.k)
    qmap = {e: oracle.quantize_expert_ref(
        (rng.standard_normal((2 * cfg.I, cfg.D)) / 16).astype(np.float32),
        (rng.standard_normal((cfg.D, cfg.I)) / 16).astype(np.float32))
        for e in range(cfg.E + 1)}
    wg = oracle.bf16_round(rng.standard_normal(cfg.D) * 0.02)
    inter = _oracle_intermediates(cfg, x, ids, qmap, wg)
    ref = oracle.moe_forward_ref(x, cfg.k, lambda e: qmap[e], cfg.E, logits=logits,
                                 w_g=wg)
    tokens = np.arange(cfg.T)
    staged_layer_check(cfg, x, ref["out"], ids, w, inter, tokens, qmap, wg)
    bad = dict(inter, hq=inter["hq"].clone())
    bad["hq"][3, 5] ^= 1
    with pytest.raises(AssertionError, match="h codes"):
        staged_layer_check(cfg, x, ref["out"], ids, w, bad, tokens, qmap, wg)
    bad = dict(inter, h=inter["h"].clone())
    bad["h"][7, 2] *= 1.01
    with pytest.raises(AssertionError):
        staged_layer_check(cfg, x, ref["out"], ids, w, bad, tokens, qmap, wg)
    out = ref["out"].copy()
    out[4, 9] += 0.5 * np.sqrt(np.mean(ref["out64"] ** 2))
    with pytest.raises(AssertionError, match="accuracy|max excess"):
        staged_layer_check(cfg, x, out, ids, w, inter, tokens, qmap, wg)
