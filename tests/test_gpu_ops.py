"""Per-entry-point parity of the CUDA path against the oracle, through the C
ABI, on seeded inputs small enough for the full oracle: several tiles, ragged
tails, empty experts and the degenerate cases of each step.

Bars: routing ids, counts, offsets, the permutation, FP8 codes and scales are
bit-exact; floating-point outputs stay within bounds derived from fp32
arithmetic (stated at each check)."""

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_helpers import U32, ensure_library, gemm_bound, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    require_gpu()
    ensure_library()


def B():
    from expert_layer_ptpc_gb300 import binding
    return binding


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# ---------------------------------------------------------------------------
# router projection
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,E,D", [(64, 8, 256), (5, 3, 128), (33, 64, 4096)])
def test_router_logits_exact(T, E, D):
    g = torch.Generator().manual_seed(T * 1000 + E)
    x = torch.randn(T, D, generator=g).to(torch.bfloat16)
    w = (torch.randn(E, D, generator=g) * 0.02).to(torch.bfloat16)
    got = B().moe_router_logits(x.cuda(), w.cuda()).cpu().numpy()
    ref = oracle.router_logits_ref(x.float().numpy(), w.float().numpy())
    # fp64 sums of exact products, one rounding: equal except for a double
    # rounding at an fp32 midpoint, which would differ by one ulp
    diff = np.abs(got.view(np.int32).astype(np.int64) - ref.view(np.int32))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.999


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,E,k,renorm,ties", [
    (64, 8, 2, True, False), (100, 128, 8, True, False),
    (37, 512, 10, True, False), (16, 1024, 32, True, False),
    (50, 64, 6, False, False), (200, 16, 5, True, True),
    (31, 32, 32, True, True), (7, 1, 1, True, False), (9, 40, 1, False, True),
])
def test_route(T, E, k, renorm, ties):
    rng = np.random.default_rng(T + E + k)
    if ties:
        logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    else:
        logits = rng.standard_normal((T, E)).astype(np.float32)
    ids, w = B().moe_route(cuda(logits), k, renormalize=renorm)
    rid, rw = oracle.route_ref(logits, k, renormalize=renorm)
    assert np.array_equal(ids.cpu().numpy(), rid)
    # fp32 exp and sum over <= 32 terms: a few ulps relative
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=64 * U32, atol=0)


# ---------------------------------------------------------------------------
# permutation
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,E,k,skew", [
    (64, 8, 2, False), (1, 512, 10, False), (16, 128, 8, False),
    (3000, 64, 6, True), (8192, 128, 8, False), (4096, 256, 8, True),
    (20000, 1024, 4, True), (5, 7, 7, False),
    (2049, 16, 4, False),      # 8196 entries: four past the one-block path
    (5000, 256, 8, "hot"),     # every token picks expert 3 (one counter)
])
def test_permute(T, E, k, skew):
    rng = np.random.default_rng(T * 7 + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    if skew == "hot":
        logits[:, 3] += 30.0
    elif skew:   # many experts empty
        logits[:, : E // 2] -= 20.0
    ids, _ = oracle.route_ref(logits, k)
    counts, offsets, s2f, f2s = B().moe_permute(cuda(ids), E)
    rc, ro, rs, rf = oracle.permute_ref(ids, E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(s2f.cpu().numpy(), rs)
    assert np.array_equal(f2s.cpu().numpy(), rf)


# ---------------------------------------------------------------------------
# quantisation
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,rows,cols", [
    ("bf16", 64, 256), ("bf16", 33, 4096), ("f32", 130, 1536),
    ("f32", 7, 128), ("bf16", 5, 16), ("f32", 3, 8192),
    # one warp per row up to 1024 columns: one or two vectors per lane, a
    # ragged 17-vector row, rows not a multiple of the block's eight warps
    ("f32", 1001, 512), ("f32", 77, 1024), ("bf16", 19, 272), ("f32", 5, 1040),
    ("bf16", 41, 2048), ("f32", 9, 2064),
])
def test_quant_exact(dtype, rows, cols):
    rng = np.random.default_rng(rows * cols)
    v = (rng.standard_normal((rows, cols)) *
         np.exp(rng.uniform(-10, 10, size=(rows, 1)))).astype(np.float32)
    v[0] = 0.0                                   # zero row
    if rows > 2:
        v[1, :] = 1e-30                          # scale from the 1e-12 floor
        v[2, ::3] = 0.0
    t = torch.from_numpy(v)
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
        v = t.float().numpy()
    q, s = B().moe_quant_ptpc(t.cuda())
    rq, rs = oracle.quant_rows_ref(v)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("T,D,k", [
    (40, 512, 3), (45, 2048, 3),
    (21, 256, 31),    # 32 destinations: one lane each
    (21, 256, 32),    # 33 destinations: the block-per-row kernel
])
def test_quant_scatter_with_extra_rows(T, D, k):
    rng = np.random.default_rng(3 + k)
    x = torch.from_numpy(rng.standard_normal((T, D)).astype(np.float32)).to(
        torch.bfloat16)
    perm = rng.permutation(T * k).astype(np.int32)
    R = T * k
    q, s = B().moe_quant_ptpc(x.cuda(), dst_rows=cuda(perm), copies=k,
                              extra_row_base=R, out_rows=R + T)
    rq, rs = oracle.quant_rows_ref(x.float().numpy())
    q = q.cpu().numpy()
    s = s.cpu().numpy()
    for f in range(R):
        assert np.array_equal(q[perm[f]], rq[f // k])
        assert s[perm[f]] == rs[f // k]
    assert np.array_equal(q[R:], rq)
    assert np.array_equal(s[R:], rs)


@pytest.mark.parametrize("T,D,E,k,renorm", [
    (64, 256, 8, 2, True), (300, 4096, 128, 8, True), (1000, 2048, 256, 8, True),
    (129, 4096, 512, 10, False), (17, 1024, 40, 3, True), (5, 4096, 300, 16, True),
    (300, 192, 64, 6, False),       # 3 K blocks: no K split, one CTA per tile
    (600, 192, 300, 8, False),      # no K split, upper column half partly past E
    (33, 256, 8, 1, True), (200, 512, 20, 1, False)])   # k = 1
def test_router_topk(T, D, E, k, renorm):
    """Router GEMM + top-k in one kernel. The logits (fp32 GEMM) lie within
    the fp32 accumulation bound of the exact dot products; the selection and
    weights are moe_route's on exactly those logits (ids bit for bit); and the
    chosen set is valid for the exact logits within twice that bound."""
    rng = np.random.default_rng(T + D + E + k)
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    x = bf(rng.standard_normal((T, D)))
    w = bf(rng.standard_normal((E, D)) * 0.02)
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ids, wts = B().moe_router_topk(x.cuda(), w.cuda(), k, renorm, logits=logits)
    assert B().moe_device_status() == (0, 0)
    xd, wd = x.double().numpy(), w.double().numpy()
    exact = xd @ wd.T
    bound = gemm_bound(np.abs(xd) @ np.abs(wd).T, D)
    got_l = logits.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got_l - exact) <= bound)
    rid, rw = oracle.route_ref(logits.cpu().numpy(), k, renorm)
    ids = ids.cpu().numpy()
    assert np.array_equal(ids, rid)
    np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=1e-5, atol=1e-7)
    for t in range(T):
        chosen = np.zeros(E, bool)
        chosen[ids[t]] = True
        if chosen.all():
            continue
        tol = 2 * bound[t].max()
        assert exact[t, chosen].min() >= exact[t, ~chosen].max() - tol


@pytest.mark.parametrize("name,T", [("prefill", None), ("sweep", 16384)])
def test_router_topk_full_size(name, T):
    """The fused router at the routing shapes `bench.py --router-gemm` times,
    with the benchmark's own inputs: prefill (8192 tokens, 128 experts,
    top-8) and the T = 16384 sweep point (512 experts, top-10). Logits of
    sampled tokens within the fp32 bound of the exact products; ids of every
    token bit-exact and weights within 1e-5 against route_ref on the
    kernel's own logits."""
    from dataclasses import replace
    from expert_layer_ptpc_gb300 import synthetic as syn
    cfg = syn.CONFIGS[name] if T is None else syn.sweep_config(T)
    cfg = replace(cfg, router="weights")
    x = syn.gen_x(cfg, "cuda")
    w = syn.gen_router_weights(cfg, "cuda")
    logits = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device="cuda")
    ids, wts = B().moe_router_topk(x, w, cfg.k, cfg.renormalize, logits=logits)
    assert B().moe_device_status() == (0, 0)
    lg = logits.cpu().numpy()
    rid, rw = oracle.route_ref(lg, cfg.k, cfg.renormalize)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(wts.cpu().numpy(), rw, rtol=1e-5, atol=1e-7)
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(cfg.T, 64, replace=False))
    rows[-1] = cfg.T - 1
    xd = x[torch.as_tensor(rows, device="cuda").long()].double().cpu().numpy()
    wd = w.double().cpu().numpy()
    exact = xd @ wd.T
    bound = gemm_bound(np.abs(xd) @ np.abs(wd).T, cfg.D)
    assert np.all(np.abs(lg[rows].astype(np.float64) - exact) <= bound)


@pytest.mark.parametrize("T,D,k,shared,inplace,wide", [
    (1, 256, 1, False, False, False), (37, 512, 4, True, False, False),
    (300, 4096, 8, False, True, False), (64, 7168, 2, True, True, False),
    (200, 2048, 2, False, False, True),
    (21, 256, 32, True, False, False)])   # 33 destinations, 32-thread blocks
def test_add_rmsnorm_quant(T, D, k, shared, inplace, wide):
    """Fused add + RMSNorm + quant against the oracle: the new residual, the
    codes at every destination row and the scales bit for bit, the gate
    within its fp32 evaluation bound. `wide`: a tenth of the entries are
    scaled by 2^-20, and a few rows are all zero or hold one nonzero entry."""
    rng = np.random.default_rng(T * 7 + D + k)
    bf = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    xa = rng.standard_normal((T, D))
    if wide:
        xa[rng.random((T, D)) < 0.1] *= 2.0 ** -20
        xa[0] = 0.0
        xa[1] = 0.0
        xa[1, 5] = 3.0
    x = bf(xa)
    ra = rng.standard_normal((T, D)) * 0.5
    if wide:
        ra[0] = 0.0
        ra[1] = 0.0
    res = bf(ra)
    gamma = bf(1.0 + 0.2 * rng.standard_normal(D))
    wg = bf(rng.standard_normal(D) * 0.02) if shared else None
    R = T * k
    f2s = rng.permutation(R).astype(np.int32)
    res_d = res.cuda()
    out_rows = R + (T if shared else 0)
    r_out, q, sc, gate = B().moe_add_rmsnorm_quant(
        x.cuda(), res_d, gamma.cuda(), 1e-6, dst_rows=cuda(f2s), copies=k,
        extra_row_base=R if shared else -1, out_rows=out_rows,
        residual_out=res_d if inplace else None,
        gate_w=wg.cuda() if shared else None)
    ref = oracle.add_rmsnorm_quant_ref(x.float().numpy(), res.float().numpy(),
                                       gamma.float().numpy(), 1e-6,
                                       w_g=wg.float().numpy() if shared else None)
    assert np.array_equal(r_out.float().cpu().numpy(), ref["r"])
    q = q.cpu().numpy()
    sc = sc.cpu().numpy()
    for f in range(R):
        assert np.array_equal(q[f2s[f]], ref["codes"][f // k]), f
        assert sc[f2s[f]].view(np.uint32) == ref["scales"][f // k].view(np.uint32)
    if shared:
        assert np.array_equal(q[R:], ref["codes"])
        assert np.array_equal(sc[R:].view(np.uint32), ref["scales"].view(np.uint32))
        v = ref["v"].astype(np.float64)
        absdot = np.abs(v) @ np.abs(wg.float().numpy().astype(np.float64))
        g = ref["gate"]
        bound = D * U32 * absdot * g * (1 - g) + 8 * U32
        assert np.all(np.abs(gate.cpu().numpy() - g) <= bound)


def test_shared_gate():
    rng = np.random.default_rng(4)
    x = torch.from_numpy(rng.standard_normal((70, 2048)).astype(np.float32)).to(
        torch.bfloat16)
    wg = (torch.from_numpy(rng.standard_normal(2048).astype(np.float32)) *
          0.02).to(torch.bfloat16)
    got = B().moe_shared_gate(x.cuda(), wg.cuda()).cpu().numpy()
    ref = oracle.shared_gate_ref(x.float().numpy(), wg.float().numpy())
    # fp32 dot of 2048 exact products (relative to sum|x w|) then expf
    absdot = np.abs(x.float().numpy()) @ np.abs(wg.float().numpy())
    bound = (2048 * U32) * absdot * ref * (1 - ref) + 8 * U32
    assert np.all(np.abs(got - ref) <= bound)


# ---------------------------------------------------------------------------
# grouped GEMMs
# ---------------------------------------------------------------------------
def _grouped_case(G, counts, N, K, gateup, seed):
    rng = np.random.default_rng(seed)
    rows = int(sum(counts))
    a = rng.standard_normal((rows, K)).astype(np.float32)
    aq, sa = oracle.quant_rows_ref(a)
    wn = 2 * N if gateup else N
    w = (rng.standard_normal((G, wn, K)) / np.sqrt(K)).astype(np.float32)
    wq = np.empty((G, wn, K), np.uint8)
    sw = np.empty((G, wn), np.float32)
    for g in range(G):
        wq[g], sw[g] = oracle.quant_rows_ref(w[g])
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return aq, sa, wq, sw, offs


def _ref_grouped(aq, sa, wq, sw, offs, N, gateup):
    G = wq.shape[0]
    rows = aq.shape[0]
    out = np.zeros((rows, N))
    bound = np.zeros((rows, N))
    adec = oracle.e4m3_decode(aq)
    for g in range(G):
        r0, r1 = offs[g], offs[g + 1]
        if r1 == r0:
            continue
        full = oracle.ptpc_matmul_ref(aq[r0:r1], sa[r0:r1], wq[g], sw[g])
        absacc = (np.abs(adec[r0:r1]) @ np.abs(oracle.e4m3_decode(wq[g])).T) * \
            sa[r0:r1, None].astype(np.float64) * sw[g][None, :].astype(np.float64)
        K = aq.shape[1]
        if gateup:
            gg, uu = full[:, :N], full[:, N:]
            eg = gemm_bound(absacc[:, :N], K)
            eu = gemm_bound(absacc[:, N:], K)
            sig = oracle.sigmoid_ref(gg)
            silu = gg * sig
            dsilu = np.abs(sig * (1 + gg * (1 - sig)))
            out[r0:r1] = silu * uu
            # first-order propagation plus the fp32 evaluation of silu * u
            # with the fast exponential and division: CUDA documents at most
            # 2 + floor(1.173 |x|) ulp for __expf(x) and 2 ulp for
            # __fdividef in this range, plus the scaling multiplies
            ulps = 16 + 2 + np.floor(1.173 * np.abs(gg))
            bound[r0:r1] = dsilu * np.abs(uu) * eg + np.abs(silu) * eu + \
                ulps * U32 * np.abs(silu * uu) + 1e-30
        else:
            out[r0:r1] = full
            bound[r0:r1] = gemm_bound(absacc, K) + 1e-30
    return out, bound


@pytest.mark.parametrize("gateup", [True, False])
@pytest.mark.parametrize("G,counts,N,K,hint", [
    (4, [3, 0, 17, 1], 128, 256, 0),                 # BN 16, ragged, empty
    (8, [40, 33, 0, 0, 64, 1, 90, 7], 256, 512, 0),  # BN 32
    (3, [200, 129, 64], 128, 1024, 0),               # BN 128 / 64
    (5, [300, 0, 257, 511, 2], 384, 384, 0),         # BN 128 / 256, tails
    (2, [1000, 24], 128, 4096, 0),                   # long K
    (2, [600, 301], 256, 512, 0),                    # BN 256 (wide tiles)
    (4, [130, 0, 300, 77], 512, 256, 0),             # CTA pairs, BN 128
    (6, [5, 9, 0, 300, 2, 3], 256, 256, 16),         # hint forces BN 16
    (3, [400, 5, 90], 768, 384, 100),                # BN 128; down: 256-channel tiles
    # BN 16 with more possible tiles than two per SM: gate/up one CTA an SM
    (40, [3, 1, 4, 1, 5, 9, 2, 6, 5, 3] * 4, 512, 256, 0),
    # CTA pairs, balanced token tiles of at most 192 rows (gate/up, 256 to
    # 384 rows per expert on average): 160+160, 160+97, 192+192+192+97, 33
    # (MMA 64), 160+160+130, 96
    (6, [320, 257, 673, 33, 450, 96], 256, 512, 0),
])
def test_grouped_gemm(gateup, G, counts, N, K, hint):
    aq, sa, wq, sw, offs = _grouped_case(G, counts, N, K, gateup,
                                         seed=G * 100 + N + K)
    kind = 0 if gateup else 1
    out = B().moe_grouped_gemm(kind, cuda(aq), cuda(sa), cuda(wq), cuda(sw),
                               cuda(offs), rows_hint=hint)
    st, bits = B().moe_device_status()
    assert st == 0, bits
    got = out.cpu().numpy().astype(np.float64)
    ref, bound = _ref_grouped(aq, sa, wq, sw, offs, N, gateup)
    err = np.abs(got - ref)
    bad = err > bound
    assert not bad.any(), (np.argwhere(bad)[:5], err[bad][:5], bound[bad][:5])


def test_grouped_gemm_leaves_other_rows_alone():
    # rows before the first group and after the last are not written
    aq, sa, wq, sw, offs = _grouped_case(3, [10, 0, 20], 128, 256, False, 9)
    offs = offs + 5
    aq = np.concatenate([np.zeros((5, 256), np.uint8), aq,
                         np.zeros((7, 256), np.uint8)])
    sa = np.concatenate([np.ones(5, np.float32), sa, np.ones(7, np.float32)])
    out = torch.full((42, 128), 7.0, device="cuda")
    B().moe_grouped_gemm(1, cuda(aq), cuda(sa), cuda(wq), cuda(sw), cuda(offs),
                         out=out)
    o = out.cpu().numpy()
    assert np.all(o[:5] == 7.0) and np.all(o[35:] == 7.0)


def test_scale_max():
    rng = np.random.default_rng(11)
    sc = rng.uniform(1e-4, 2e-2, (37, 4096)).astype(np.float32)
    sc[5, 4095] = 0.5                      # the maximum in the last column
    got = B().moe_scale_max(cuda(sc)).cpu().numpy()
    assert np.array_equal(got, sc.max(axis=1))


@pytest.mark.parametrize("G,counts,N,K,hint", [
    (4, [3, 0, 17, 1], 128, 256, 0),                 # BN 16, ragged, empty
    (8, [40, 33, 0, 0, 64, 1, 90, 7], 256, 512, 0),  # BN 32
    (3, [200, 129, 64], 128, 1024, 0),               # BN 128
    (5, [300, 0, 257, 511, 2], 384, 384, 0),         # BN 256, tails
    (2, [1000, 24], 256, 1536, 0),                   # long K
    (4, [130, 0, 300, 77], 512, 512, 0),             # BN 128, 256-channel tiles
])
def test_grouped_gemm_down_f16(G, counts, N, K, hint):
    """The fp16 encoding of y: row_scale * y16 against the oracle's y, within
    the fp32 accumulation bound plus fp16 rounding (half an ulp, 2^-11
    relative; 2^-25 absolute below fp16's normal range) and four fp32
    roundings (s_d * rho, the product, a_scale / rho)."""
    aq, sa, wq, sw, offs = _grouped_case(G, counts, N, K, False, seed=G * 7 + N + K)
    bound_w = B().moe_scale_max(cuda(sw))
    y16, rs = B().moe_grouped_gemm_down_f16(cuda(aq), cuda(sa), cuda(wq), cuda(sw),
                                            bound_w, cuda(offs), rows_hint=hint)
    st, bits = B().moe_device_status()
    assert st == 0, bits
    y16 = y16.float().cpu().numpy().astype(np.float64)
    rs = rs.cpu().numpy().astype(np.float64)
    rows = int(offs[-1])
    assert np.all(np.isfinite(y16[:rows])) and np.all(np.abs(y16[:rows]) <= 60000)
    got = rs[:rows, None] * y16[:rows]
    ref, gbound = _ref_grouped(aq, sa, wq, sw, offs, N, False)
    tol = gbound * (1 + 1e-3) + np.abs(ref) * (2.0 ** -11 + 4 * U32) + \
        rs[:rows, None] * 2.0 ** -25 + 1e-30
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), (np.argwhere(bad)[:5], err[bad][:5], tol[bad][:5])


# ---------------------------------------------------------------------------
# combine
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,k,D,shared", [(64, 2, 256, False), (17, 8, 4096, True),
                                          (5, 10, 1024, True), (1, 1, 128, False)])
def test_combine(T, k, D, shared):
    rng = np.random.default_rng(T * k + D)
    R = T * k
    y = rng.standard_normal((R + (T if shared else 0), D)).astype(np.float32)
    f2s = rng.permutation(R).astype(np.int32)
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    gate = rng.uniform(0, 1, T).astype(np.float32) if shared else None
    ys = y[R:] if shared else None
    out = B().moe_combine(cuda(y), cuda(f2s), cuda(w),
                          y_shared=cuda(ys) if shared else None,
                          shared_gate=cuda(gate) if shared else None)
    got = out.float().cpu().numpy().astype(np.float64)
    ref = np.zeros((T, D))
    absref = np.zeros((T, D))
    for t in range(T):
        for j in range(k):
            term = w[t, j].astype(np.float64) * y[f2s[t * k + j]]
            ref[t] += term
            absref[t] += np.abs(term)
        if shared:
            ref[t] += gate[t].astype(np.float64) * ys[t]
            absref[t] += np.abs(gate[t].astype(np.float64) * ys[t])
    # fp32 sum of k+1 products, then one bf16 rounding (half a bf16 ulp)
    bound = (k + 2) * U32 * absref + 2.0 ** -8 * np.abs(ref) * (1 + 1e-6)
    assert np.all(np.abs(got - ref) <= bound + 1e-30)


@pytest.mark.parametrize("T,k,D,shared", [(64, 2, 256, False), (17, 8, 4096, True),
                                          (5, 10, 1024, True), (1, 1, 128, False),
                                          # 8 columns a thread (D not a multiple
                                          # of 16); a ragged third block column
                                          (9, 8, 2056, True), (3, 4, 4112, False)])
def test_combine_f16(T, k, D, shared):
    rng = np.random.default_rng(T * k + D + 1)
    R = T * k
    rows = R + (T if shared else 0)
    y16 = (rng.standard_normal((rows, D)) * 300).astype(np.float16)
    rs = rng.uniform(1e-4, 1e-2, rows).astype(np.float32)
    f2s = rng.permutation(R).astype(np.int32)
    w = rng.uniform(0, 1, (T, k)).astype(np.float32)
    gate = rng.uniform(0, 1, T).astype(np.float32) if shared else None
    out = B().moe_combine_f16(
        cuda(y16), cuda(rs), cuda(f2s), cuda(w),
        y16_shared=cuda(y16[R:]) if shared else None,
        row_scale_shared=cuda(rs[R:]) if shared else None,
        shared_gate=cuda(gate) if shared else None)
    got = out.float().cpu().numpy().astype(np.float64)
    yd = y16.astype(np.float64)
    ref = np.zeros((T, D))
    absref = np.zeros((T, D))
    for t in range(T):
        terms = [(w[t, j].astype(np.float64) * rs[f2s[t * k + j]], yd[f2s[t * k + j]])
                 for j in range(k)]
        if shared:
            terms.append((gate[t].astype(np.float64) * rs[R + t], yd[R + t]))
        for c, yr in terms:
            ref[t] += c * yr
            absref[t] += np.abs(c * yr)
    # one rounding of each coefficient, fp32 sum of k+1 products, one bf16
    # rounding (half a bf16 ulp)
    bound = (k + 3) * U32 * absref + 2.0 ** -8 * np.abs(ref) * (1 + 1e-6)
    assert np.all(np.abs(got - ref) <= bound + 1e-30)


@pytest.mark.parametrize("switches", [
    {"MOE_GEMM_CTA_PAIR": "1"},
    {"MOE_GEMM_CTA_PAIR": "1", "MOE_GEMM_BALANCED": "0", "MOE_GEMM_WIDE": "0"},
    {"MOE_GEMM_CTA_PAIR": "0"},
    {"MOE_GEMM_WIDE": "1"},
    {"MOE_GEMM_WIDE": "0"},
    {"MOE_GEMM_CTA_PAIR": "1", "MOE_GEMM_KATOMS": "1"},
], ids=["pair", "pair-unbalanced", "single", "wide", "no-wide", "pair-katoms1"])
def test_grouped_gemm_cta_pair_variant(switches):
    """The wide-tile cases with the kernel choice forced, in a child process:
    MOE_GEMM_CTA_PAIR=1 runs the CTA-pair (cta_group::2) kernel for every
    shape with more than 64 rows per expert (the down projection included),
    =0 the single-CTA kernel everywhere (the gate/up shapes that otherwise
    take the pair). MOE_GEMM_BALANCED=0 cuts the pair kernel's token tiles
    into full ones and a partial tail instead of equal widths.
    MOE_GEMM_WIDE=1 / =0 turns the 512-token gate/up tiles (two MMAs per K
    step) on / off above 256 rows per expert. MOE_GEMM_KATOMS=1 gives the
    gate/up pair kernel stages of one 128-byte K atom (the form that K not a
    multiple of 256 takes) instead of two."""
    import os
    import subprocess
    import sys
    env = dict(os.environ, **switches)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m",
           "gpu", os.path.join(root, "tests", "test_gpu_ops.py"), "-k",
           "test_grouped_gemm and (counts2 or counts3 or counts4 or counts5 or counts6 "
           "or counts10)"]
    r = subprocess.run(cmd, env=env, cwd=root, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
