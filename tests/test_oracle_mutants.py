"""Planted mistakes in the oracle must each fail at least one pin.

Each mutant replaces one oracle function with a plausibly wrong variant (a
dropped term, a swapped operand, a wrong tie rule ...) on the CPU; the test
runs the relevant pins against the mutated oracle and expects an assertion
failure. This checks that the pins constrain every step of the oracle.
"""

import numpy as np
import pytest

import oracle
import oracle.blockscale_ref as bref
import oracle.moe_ref as ref
import oracle.norm_ref as nref
from tests import test_oracle_blockscale as block_pins
from tests import test_oracle_layer as layer_pins
from tests import test_oracle_norm as norm_pins
from tests import test_oracle_route as route_pins


def _mut_silu(g):
    return ref.sigmoid_ref(g)                       # dropped the g factor


def _mut_expert_ffn_swap(xq, sx, wgu, sgu, wd, sd):
    I = wgu.shape[0] // 2
    gu = ref.ptpc_matmul_ref(xq, sx, wgu, sgu)
    h = ref.silu_ref(gu[:, I:]) * gu[:, :I]         # gate and up swapped
    hq, sh = ref.quant_rows_ref(h.astype(np.float32))
    return {"y": ref.ptpc_matmul_ref(hq, sh, wd, sd)}


def _mut_expert_ffn_no_requant(xq, sx, wgu, sgu, wd, sd):
    I = wgu.shape[0] // 2
    gu = ref.ptpc_matmul_ref(xq, sx, wgu, sgu)
    h = ref.silu_ref(gu[:, :I]) * gu[:, I:]
    wdq = ref.dequant_rows_ref(wd, sd)
    return {"y": h @ wdq.T}                         # h never quantised


def _mut_ptpc_one_scale(a, sa, w, sw):
    acc = ref.e4m3_decode(a) @ ref.e4m3_decode(w).T
    return acc * np.asarray(sa, np.float64)[:, None]   # weight scale dropped


def _mut_route_tie_high(logits, k, renormalize=True):
    lg = np.asarray(logits, np.float32)
    E = lg.shape[1]
    rev = lg[:, ::-1]
    order = (E - 1) - np.argsort(-rev, axis=1, kind="stable")  # ties -> higher
    ids = order[:, :k].astype(np.int32)
    ch = np.take_along_axis(lg, ids.astype(np.int64), 1).astype(np.float64)
    p = np.exp(ch - ch[:, :1])
    return ids, p / p.sum(1, keepdims=True)


def _mut_route_no_renorm(logits, k, renormalize=True):
    ids, _ = _orig_route(logits, k, renormalize)
    lg = np.asarray(logits, np.float64)
    p = np.exp(lg - lg.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    return ids, np.take_along_axis(p, ids.astype(np.int64), 1)


def _mut_permute_unstable(ids, E):
    counts, offsets, s2f, f2s = _orig_permute(ids, E)
    s2f = s2f.copy()
    for e in range(E):
        s2f[offsets[e]:offsets[e + 1]] = s2f[offsets[e]:offsets[e + 1]][::-1]
    f2s = np.empty_like(s2f)
    f2s[s2f] = np.arange(s2f.size, dtype=s2f.dtype)
    return counts, offsets, s2f, f2s


def _mut_quant_wrong_max(v):
    v32 = np.asarray(v, np.float32)
    amax = np.abs(v32).max(1)
    s = (np.maximum(amax, ref.QUANT_EPS) / np.float32(240)).astype(np.float32)
    return ref.e4m3_encode((v32 / s[:, None]).astype(np.float32)), s


def _mut_sigmoid_gate(z):
    return np.ones_like(np.asarray(z, np.float64))       # shared gate ignored


_orig_route = ref.route_ref
_orig_permute = ref.permute_ref


def _norm_variant(no_gamma=False, d_minus_1=False, eps_outside=False, no_bf16=False):
    def f(x, res, gamma, eps):
        x32 = np.asarray(x, np.float32)
        res32 = np.asarray(res, np.float32)
        g32 = np.asarray(gamma, np.float32)
        T, D = x32.shape
        s = (x32 + res32).astype(np.float32)
        r = s if no_bf16 else oracle.bf16_round(s.astype(np.float64))
        v = np.empty((T, D), np.float32)
        inv = np.empty(T, np.float32)
        for t in range(T):
            ms = np.float32(np.sum(r[t].astype(np.float64) ** 2) / (D - 1 if d_minus_1 else D))
            if eps_outside:
                inv[t] = np.float32(1.0 / (np.sqrt(np.float64(ms)) + eps))
            else:
                inv[t] = nref.rsqrt_f32_rn(np.float32(ms + np.float32(eps)))
            v[t] = (r[t] * inv[t]).astype(np.float32) * (np.float32(1) if no_gamma else g32)
        return r, v, inv
    return f


def _mut_rsqrt_two_roundings(a):
    a32 = np.float32(a)
    return np.float32(np.float32(1.0) / np.sqrt(a32))


def _norm_pins():
    for a in [1e-6, 0.25, 0.3, 1.0, 2.0, 3.0, 7.5, 1234.5678, 6.02e23, 1.1754944e-38, 3.0e38]:
        norm_pins.test_rsqrt_is_correctly_rounded(a)
    norm_pins.test_residual_matches_torch_bf16_add()
    norm_pins.test_matches_torch_rms_norm()
    norm_pins.test_constant_row_closed_form()
    norm_pins.test_scale_invariance_without_eps()
    norm_pins.test_zero_row_quantises_to_zero()


def _layer_pins():
    for params in [(25, 128, 6, 3, 128, True, "normal"),
                   (33, 256, 8, 2, 128, False, "weights")]:
        layer_pins.test_layer_matches_dense_evaluation(*params)


def _route_pins():
    rng = np.random.default_rng(7)
    for case in route_pins._cases():
        route_pins.test_golden_cases(case)
    route_pins.test_selection_properties_with_ties(rng, 6, 3)
    route_pins.test_all_equal_logits()


def _permute_pins():
    rng = np.random.default_rng(7)
    route_pins.test_permute_invariants(rng, 37, 8, 2)


def _quant_pins():
    rng = np.random.default_rng(7)
    layer_pins.test_quant_matches_torch_quantiser(rng)


def _mut_quant_blocks_strided(v, block):
    v32 = np.asarray(v, dtype=np.float32)
    R, K = v32.shape
    nb = K // block
    # blocks gathered with stride nb instead of contiguous runs
    pieces = v32.reshape(R, block, nb).transpose(0, 2, 1).reshape(R * nb, block)
    codes, scales = ref.quant_rows_ref(pieces)
    return codes.reshape(R, nb, block).transpose(0, 2, 1).reshape(R, K), scales.reshape(R, nb)


def _mut_weight_blocks_row_strips(w, bn=128, bk=128):
    w32 = np.asarray(w, dtype=np.float32)
    N, K = w32.shape
    # 1 x (bn * bk) strips of consecutive entries instead of bn x bk tiles
    codes, scales = ref.quant_rows_ref(w32.reshape(-1, bn * bk))
    return codes.reshape(N, K), scales.reshape(N // bn, K // bk)


def _mut_blockscale_tiled_weight_scale(a_codes, a_scale, w_codes, w_scale):
    P = bref.block_partials_ref(a_codes, w_codes, 128)
    sa = np.asarray(a_scale, np.float64)
    sw = np.tile(np.asarray(w_scale, np.float64), (128, 1))   # n % nn, not n // 128
    y = np.zeros(P.shape[1:])
    for b in range(P.shape[0]):
        y += sa[:, b][:, None] * sw[:, b][None, :] * P[b]
    return y


def _mut_blockscale_no_activation_scale(a_codes, a_scale, w_codes, w_scale):
    P = bref.block_partials_ref(a_codes, w_codes, 128)
    sw = np.repeat(np.asarray(w_scale, np.float64), 128, axis=0)
    return sum(sw[:, b][None, :] * P[b] for b in range(P.shape[0]))


def _mut_subchannel_first_group_scale(a_codes, a_scale, w_codes, w_scale, block=512):
    P = bref.block_partials_ref(a_codes, w_codes, block)
    sa = np.asarray(a_scale, np.float64)
    y = P.sum(axis=0) * sa[:, 0][:, None]          # one group's scale for all
    return y * np.asarray(w_scale, np.float64)[None, :]


def _blockscale_pins():
    block_pins.test_one_block_per_row_is_the_ptpc_quantiser()
    for b in (128, 512):
        block_pins.test_each_block_is_quantised_on_its_own(b)
    block_pins.test_weight_block_is_a_per_tensor_quantiser()
    block_pins.test_weight_blocks_slice_by_slice()
    block_pins.test_blockscale_matmul_equals_dequantise_first()
    block_pins.test_subchannel_matmul_equals_dequantise_first()
    block_pins.test_equal_block_scales_reduce_to_ptpc()


MUTANTS = {
    "silu_drops_g": (ref, "silu_ref", _mut_silu, _layer_pins),
    "gate_up_swapped": (ref, "expert_ffn_ref", _mut_expert_ffn_swap, _layer_pins),
    "no_requant": (ref, "expert_ffn_ref", _mut_expert_ffn_no_requant, _layer_pins),
    "weight_scale_dropped": (ref, "ptpc_matmul_ref", _mut_ptpc_one_scale,
                             _layer_pins),
    "ties_to_higher_index": (ref, "route_ref", _mut_route_tie_high, _route_pins),
    "no_renormalisation": (ref, "route_ref", _mut_route_no_renorm, _route_pins),
    "unstable_permutation": (ref, "permute_ref", _mut_permute_unstable,
                             _permute_pins),
    "quant_wrong_fp8_max": (ref, "quant_rows_ref", _mut_quant_wrong_max,
                            _quant_pins),
    "shared_gate_ignored": (ref, "sigmoid_ref", _mut_sigmoid_gate, _layer_pins),
    "norm_drops_gamma": (nref, "add_rmsnorm_ref", _norm_variant(no_gamma=True),
                         _norm_pins),
    "norm_mean_over_d_minus_1": (nref, "add_rmsnorm_ref",
                                 _norm_variant(d_minus_1=True), _norm_pins),
    "norm_eps_outside_sqrt": (nref, "add_rmsnorm_ref",
                              _norm_variant(eps_outside=True), _norm_pins),
    "norm_residual_not_bf16": (nref, "add_rmsnorm_ref", _norm_variant(no_bf16=True),
                               _norm_pins),
    "rsqrt_two_roundings": (nref, "rsqrt_f32_rn", _mut_rsqrt_two_roundings,
                            _norm_pins),
    "activation_blocks_strided": (bref, "quant_blocks_ref", _mut_quant_blocks_strided,
                                  _blockscale_pins),
    "weight_blocks_as_strips": (bref, "quant_weight_blocks_ref",
                                _mut_weight_blocks_row_strips, _blockscale_pins),
    "blockscale_weight_scale_tiled": (bref, "blockscale_matmul_ref",
                                      _mut_blockscale_tiled_weight_scale, _blockscale_pins),
    "blockscale_no_activation_scale": (bref, "blockscale_matmul_ref",
                                       _mut_blockscale_no_activation_scale,
                                       _blockscale_pins),
    "subchannel_one_group_scale": (bref, "subchannel_matmul_ref",
                                   _mut_subchannel_first_group_scale, _blockscale_pins),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(monkeypatch, name):
    module, attr, fn, pins = MUTANTS[name]
    monkeypatch.setattr(module, attr, fn)
    # the pin modules imported some oracle functions by name, and the norm
    # pins call them through the package
    if hasattr(oracle, attr):
        monkeypatch.setattr(oracle, attr, fn)
    for pin_mod in (layer_pins, route_pins):
        if hasattr(pin_mod, attr):
            monkeypatch.setattr(pin_mod, attr, fn)
    with pytest.raises(AssertionError):
        pins()
