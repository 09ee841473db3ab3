"""Pins of the oracle's quantiser, PTPC GEMM and whole layer.

The layer pin is a dense evaluation written with torch CPU ops only (torch's
fp8 cast, matmul, topk, softmax, silu): every expert runs on every token and
the routing masks the results. It shares nothing with the oracle's grouped,
permuted evaluation except the definition of the layer.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import (e4m3_decode, moe_forward_ref, ptpc_matmul_ref,
                    quant_rows_ref, router_logits_ref)
from expert_layer_ptpc_gb300 import synthetic as syn


# ---------------------------------------------------------------------------
# quantiser
# ---------------------------------------------------------------------------
def _torch_quant_rows(v32):
    """Per-row e4m3 quantisation written with torch ops (IEEE fp32 division,
    torch's nearest-even fp8 cast)."""
    v = torch.as_tensor(v32, dtype=torch.float32)
    amax = v.abs().amax(dim=1)
    s = torch.clamp(amax, min=1e-12) / 448.0
    q = (v / s[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy(), s.numpy()


def test_quant_matches_torch_quantiser(rng):
    v = (rng.standard_normal((300, 517)) *
         np.exp(rng.uniform(-8, 8, size=(300, 1)))).astype(np.float32)
    q, s = quant_rows_ref(v)
    tq, ts = _torch_quant_rows(v)
    assert np.array_equal(s.view(np.uint32), ts.view(np.uint32))
    assert np.array_equal(q, tq)


def test_quant_row_max_hits_448_and_error_bound(rng):
    v = rng.standard_normal((64, 256)).astype(np.float32)
    q, s = quant_rows_ref(v)
    am = np.abs(v).argmax(axis=1)
    assert np.all((q[np.arange(64), am] & 0x7F) == 0x7E)
    deq = e4m3_decode(q) * s[:, None]
    # half an e4m3 step: relative 2**-4 for normals, 2**-10 * s absolute below
    err = np.abs(deq - v)
    bound = np.maximum(np.abs(v) * 2.0 ** -4, 2.0 ** -10 * s[:, None])
    assert np.all(err <= bound * (1 + 1e-6))


def test_quant_zero_row():
    q, s = quant_rows_ref(np.zeros((2, 8), np.float32))
    assert np.all(q == 0)
    assert s[0] == np.float32(np.float32(1e-12) / np.float32(448))


# ---------------------------------------------------------------------------
# PTPC GEMM
# ---------------------------------------------------------------------------
def test_ptpc_matmul_exact_in_integers(rng):
    a = rng.integers(0, 256, size=(40, 1024), dtype=np.uint8)
    w = rng.integers(0, 256, size=(24, 1024), dtype=np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x11          # no NaN codes
    w[(w & 0x7F) == 0x7F] = 0x22
    sa = rng.uniform(0.5, 2, 40).astype(np.float32)
    sw = rng.uniform(0.5, 2, 24).astype(np.float32)
    # every e4m3 value times 2**9 is an integer: the dot products are exact in
    # int64, then scaled by 2**-18.
    ai = (e4m3_decode(a) * 512).astype(np.int64)
    wi = (e4m3_decode(w) * 512).astype(np.int64)
    acc = (ai @ wi.T).astype(np.float64) * 2.0 ** -18
    ref = acc * sa.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]
    got = ptpc_matmul_ref(a, sa, w, sw)
    assert np.allclose(got, ref, rtol=1e-15, atol=0)


def test_ptpc_equals_dequantise_first(rng):
    x = rng.standard_normal((30, 384)).astype(np.float32)
    W = rng.standard_normal((50, 384)).astype(np.float32)
    xq, sx = quant_rows_ref(x)
    wq, sw = quant_rows_ref(W)
    ref = (e4m3_decode(xq) * sx[:, None].astype(np.float64)) @ \
        (e4m3_decode(wq) * sw[:, None].astype(np.float64)).T
    assert np.allclose(ptpc_matmul_ref(xq, sx, wq, sw), ref, rtol=1e-12,
                       atol=1e-12 * np.abs(ref).max())


def test_router_logits_exactly_rounded(rng):
    x = torch.randn(5, 256).to(torch.bfloat16).float().numpy()
    w = (torch.randn(8, 256) * 0.02).to(torch.bfloat16).float().numpy()
    got = router_logits_ref(x, w)
    for t in range(5):
        for e in range(8):
            exact = math.fsum(float(a) * float(b) for a, b in zip(x[t], w[e]))
            assert got[t, e] == np.float32(exact)


# ---------------------------------------------------------------------------
# whole layer: dense torch evaluation
# ---------------------------------------------------------------------------
def _make_layer(T, D, E, k, I, shared, seed=0, router="normal"):
    cfg = syn.LayerConfig("pin", T, D, E, k, I, shared, router)
    x = syn.gen_x(cfg, seed=seed).float().numpy()
    if router == "weights":
        wr = syn.gen_router_weights(cfg, seed=seed).float().numpy()
        logits = None
    else:
        wr = None
        logits = syn.gen_logits(cfg, seed=seed).numpy()
    raw = [syn.gen_expert_weights(cfg, e, seed=seed)
           for e in range(E + (1 if shared else 0))]
    wg = syn.gen_shared_gate(cfg, seed=seed).float().numpy() if shared else None
    return cfg, x, logits, wr, raw, wg


def _dense_torch(x, logits, wr, raw, wg, k, E):
    """Every expert on every token, masked by the routing (torch fp64)."""
    xt = torch.from_numpy(x).double()
    if logits is None:
        logits = (xt @ torch.from_numpy(wr).double().T).float()
    else:
        logits = torch.from_numpy(logits)
    top_v, top_i = torch.topk(logits, k, dim=1)
    w = torch.softmax(top_v.double(), dim=1)
    mask = torch.zeros(logits.shape, dtype=torch.float64)
    mask.scatter_(1, top_i, w)

    def quant(v32):
        q, s = _torch_quant_rows(v32)
        return (torch.from_numpy(q).view(torch.float8_e4m3fn).double() *
                torch.from_numpy(s).double()[:, None])

    xdq = quant(x)
    out = torch.zeros_like(xt)
    for e in range(len(raw)):
        wgu, wd = raw[e]
        wgu_dq = quant(wgu.numpy())
        wd_dq = quant(wd.numpy())
        I = wgu.shape[0] // 2
        gu = xdq @ wgu_dq.T
        h = F.silu(gu[:, :I]) * gu[:, I:]
        y = quant(h.float().numpy()) @ wd_dq.T
        if e < E:
            out += mask[:, e:e + 1] * y
        else:
            gate = torch.sigmoid(xt @ torch.from_numpy(wg).double())
            out += gate[:, None] * y
    return out.numpy(), top_i.numpy()


def _oracle_run(x, logits, wr, raw, wg, k, E, tokens=None):
    quantised = {}

    def expert_weights(e):
        if e not in quantised:
            wgu, wd = raw[e]
            quantised[e] = oracle.quantize_expert_ref(wgu.numpy(), wd.numpy())
        return quantised[e]
    return moe_forward_ref(x, k, expert_weights, E, logits=logits,
                           router_w=wr, w_g=wg, tokens=tokens)


@pytest.mark.parametrize("T,D,E,k,I,shared,router", [
    (40, 128, 8, 2, 64, False, "normal"),
    (33, 256, 8, 2, 128, False, "weights"),
    (25, 128, 6, 3, 128, True, "normal"),
    (17, 128, 4, 4, 64, True, "normal"),
])
def test_layer_matches_dense_evaluation(T, D, E, k, I, shared, router):
    cfg, x, logits, wr, raw, wg = _make_layer(T, D, E, k, I, shared,
                                              router=router)
    r = _oracle_run(x, logits, wr, raw, wg, k, E)
    dense, top_i = _dense_torch(x, logits, wr, raw, wg, k, E)
    assert np.array_equal(np.sort(r["ids"], 1), np.sort(top_i, 1))
    scale = np.sqrt(np.mean(dense ** 2))
    assert np.max(np.abs(r["out64"] - dense)) <= 1e-12 * scale


def test_single_expert_is_dense_ffn():
    cfg, x, logits, wr, raw, wg = _make_layer(20, 128, 1, 1, 64, False)
    r = _oracle_run(x, logits, wr, raw, wg, 1, 1)
    assert np.allclose(r["w"], 1.0, rtol=0, atol=0)
    dense, _ = _dense_torch(x, logits, wr, raw, wg, 1, 1)
    assert np.max(np.abs(r["out64"] - dense)) <= 1e-12 * np.abs(dense).max()
    ref_bf16 = torch.from_numpy(dense).to(torch.bfloat16).float().numpy()
    # bf16 rounding of fp64 vs torch's of fp64: both nearest-even
    assert np.array_equal(r["out"], ref_bf16)


def test_token_subset_matches_full_run():
    cfg, x, logits, wr, raw, wg = _make_layer(30, 128, 8, 3, 64, True)
    full = _oracle_run(x, logits, wr, raw, wg, 3, 8)
    sub = [29, 0, 7, 7, 15]
    part = _oracle_run(x, logits, wr, raw, wg, 3, 8, tokens=sub)
    assert np.array_equal(part["out64"], full["out64"][sub])


def test_zero_tokens_rows():
    cfg, x, logits, wr, raw, wg = _make_layer(8, 128, 4, 2, 64, True)
    x[3] = 0.0
    r = _oracle_run(x, logits, wr, raw, wg, 2, 4)
    assert np.all(r["xq"][3] == 0)
    assert np.all(r["out64"][3] == 0.0)
