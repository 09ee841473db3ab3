"""Pins of the add + RMSNorm + quant oracle (MI300X page, section 2.1.5: the
fused AddRMSNorm + per-token quant operator) against exact arithmetic, a
library routine, closed forms and invariants."""

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _bf16(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).float().numpy()


def _case(T, D, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    x = _bf16(rng.standard_normal((T, D)) * scale)
    res = _bf16(rng.standard_normal((T, D)) * scale)
    gamma = _bf16(1.0 + 0.1 * rng.standard_normal(D))
    return x, res, gamma


@pytest.mark.parametrize("a", [1e-6, 0.25, 0.3, 1.0, 2.0, 3.0, 7.5, 1234.5678, 6.02e23,
                               1.1754944e-38, 3.0e38])
def test_rsqrt_is_correctly_rounded(a):
    """r is the correctly rounded fp32 1/sqrt(a) iff the exact value lies
    between the midpoints to its fp32 neighbours, i.e. m_lo^2 a < 1 < m_hi^2 a
    in exact rational arithmetic."""
    a32 = np.float32(a)
    r = oracle.rsqrt_f32_rn(a32)
    lo = np.nextafter(r, np.float32(0.0))
    hi = np.nextafter(r, np.float32(np.inf))
    fa, fr = Fraction(float(a32)), Fraction(float(r))
    m_lo = (Fraction(float(lo)) + fr) / 2
    m_hi = (fr + Fraction(float(hi))) / 2
    assert m_lo * m_lo * fa < 1 < m_hi * m_hi * fa


def test_residual_matches_torch_bf16_add():
    x, res, gamma = _case(33, 256, 1)
    r, _, _ = oracle.add_rmsnorm_ref(x, res, gamma, 1e-6)
    ref = (torch.from_numpy(x).bfloat16() + torch.from_numpy(res).bfloat16()).float()
    assert np.array_equal(r, ref.numpy())


def test_matches_torch_rms_norm():
    x, res, gamma = _case(40, 1024, 2)
    r, v, _ = oracle.add_rmsnorm_ref(x, res, gamma, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(r).double(), (1024,),
                                       torch.from_numpy(gamma).double(), eps=1e-6)
    # four fp32 roundings (mean, rsqrt, two products) of a value of size |v|
    assert np.allclose(v, ref.numpy(), rtol=4 * 2.0 ** -24, atol=0)


def test_constant_row_closed_form():
    """x + res = c everywhere, eps = 0, c a power of two: inv = 1/|c| exactly
    and v = sign(c) * gamma."""
    D = 512
    gamma = _bf16(np.linspace(-2, 2, D))
    for c in (0.5, 2.0, -4.0):
        x = np.full((1, D), c / 2, np.float32)
        res = np.full((1, D), c / 2, np.float32)
        r, v, inv = oracle.add_rmsnorm_ref(x, res, gamma, 0.0)
        assert inv[0] == np.float32(1.0 / abs(c))
        assert np.array_equal(v[0], np.sign(c) * gamma)


def test_scale_invariance_without_eps():
    """Multiplying x and res by 2^k scales r by 2^k (exact in bf16) and leaves
    v unchanged bit for bit when eps = 0."""
    x, res, gamma = _case(8, 384, 3)
    _, v0, _ = oracle.add_rmsnorm_ref(x, res, gamma, 0.0)
    for k in (-3, 5):
        _, vk, _ = oracle.add_rmsnorm_ref(x * 2.0 ** k, res * 2.0 ** k, gamma, 0.0)
        assert np.array_equal(v0, vk)


def test_zero_row_quantises_to_zero():
    D = 256
    x = np.zeros((2, D), np.float32)
    gamma = np.ones(D, np.float32)
    out = oracle.add_rmsnorm_quant_ref(x, x, gamma, 1e-6)
    assert np.all(out["v"] == 0) and np.all(out["codes"] == 0)
    assert np.all(out["scales"] == np.float32(1e-12 / 448))
    assert out["inv"][0] == oracle.rsqrt_f32_rn(np.float32(1e-6))


def test_quant_is_the_ptpc_quantiser_of_v():
    x, res, gamma = _case(16, 512, 4)
    out = oracle.add_rmsnorm_quant_ref(x, res, gamma, 1e-5)
    codes, scales = oracle.quant_rows_ref(out["v"])
    assert np.array_equal(out["codes"], codes)
    assert np.array_equal(out["scales"], scales)
    # dequantised codes reproduce v within half an e4m3 step (3 mantissa bits)
    dq = oracle.e4m3_decode(out["codes"]) * out["scales"][:, None]
    assert np.all(np.abs(dq - out["v"]) <= 2.0 ** -4 * np.abs(out["v"]) + 2.0 ** -10 *
                  out["scales"][:, None] + 1e-30)


def test_gate_is_sigmoid_of_v_dot_wg():
    x, res, gamma = _case(5, 256, 5)
    wg = _bf16(np.random.default_rng(6).standard_normal(256) * 0.02)
    out = oracle.add_rmsnorm_quant_ref(x, res, gamma, 1e-6, w_g=wg)
    z = out["v"].astype(np.float64) @ wg.astype(np.float64)
    assert np.allclose(out["gate"], 1 / (1 + np.exp(-z)), rtol=1e-12)
