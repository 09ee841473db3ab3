"""Parity of the block-scaled FP8 path (BlockScale-128, 512-subchannel and the
same engine's PTPC mode) against the oracle, through the C ABI.

Bars: codes and scales of both block quantisers are bit-exact. The GEMM
outputs stay within the fp32 bound of their evaluation: each scale group's
tensor-core sum of G exact products (G = 128, 512 or K) plus one fma per group
and the scale products, (G + groups + 4) u times the same GEMM on magnitudes."""

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_helpers import ensure_library, gemm_bound, require_gpu

pytestmark = pytest.mark.gpu

MODES = {"ptpc": 0, "sub512": 1, "block128": 2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    require_gpu()
    ensure_library()


def B():
    from expert_layer_ptpc_gb300 import binding
    return binding


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _acts(R, K, seed):
    """bf16 activations with blocks of very different magnitude."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((R, K)).astype(np.float32)
    for r in range(R):
        b = rng.integers(0, K // 128)
        v[r, b * 128:(b + 1) * 128] *= np.float32(2.0 ** rng.integers(-10, 10))
    return torch.from_numpy(v).to(torch.bfloat16)


@pytest.mark.parametrize("R,K,block", [(1, 128, 128), (300, 1024, 128), (77, 4096, 512),
                                       (5, 512, 512), (0, 256, 128)])
def test_quant_blocks(R, K, block):
    x = _acts(max(R, 1), K, R + K)[:R]
    q, s = B().moe_quant_blocks(x.cuda(), block)
    rq, rs = oracle.quant_blocks_ref(x.float().numpy(), block)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_quant_blocks_zero_and_tiny_blocks():
    x = _acts(4, 512, 9)
    x[0] = 0.0                       # all-zero row: scale 1e-12/448, codes 0
    x[1, 128:256] = 0.0              # one zero block
    x[2, 256:384] = 2.0 ** -126      # a block of tiny values
    q, s = B().moe_quant_blocks(x.cuda(), 128)
    rq, rs = oracle.quant_blocks_ref(x.float().numpy(), 128)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("G,N,K", [(1, 128, 128), (3, 256, 640), (2, 384, 4096)])
def test_quant_weight_blocks(G, N, K):
    rng = np.random.default_rng(G * N + K)
    w = (rng.standard_normal((G, N, K)) / np.sqrt(K)).astype(np.float32)
    w[0, :128, :128] *= 100.0
    q, s = B().moe_quant_weight_blocks(cuda(w))
    rq, rs = oracle.quant_weight_blocks_ref(w.reshape(G * N, K))
    assert np.array_equal(q.cpu().numpy().reshape(G * N, K), rq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def _problem(mode, offsets, N, K, seed):
    """Quantised operands of a grouped problem, by the oracle's quantisers."""
    rng = np.random.default_rng(seed)
    offsets = np.asarray(offsets, np.int32)
    G, R = len(offsets) - 1, int(offsets[-1])
    x = _acts(R, K, seed).float().numpy()
    w = (rng.standard_normal((G, N, K)) / np.sqrt(K)).astype(np.float32)
    w[:, :, :128] *= 4.0
    if mode == "block128":
        qa, sa = oracle.quant_blocks_ref(x, 128)
        qw, sw = oracle.quant_weight_blocks_ref(w.reshape(G * N, K))
        sw = sw.reshape(G, N // 128, K // 128)
    elif mode == "sub512":
        qa, sa = oracle.quant_blocks_ref(x, 512)
        qw, sw = oracle.quant_rows_ref(w.reshape(G * N, K))
        sw = sw.reshape(G, N)
    else:
        qa, sa = oracle.quant_rows_ref(x)
        qw, sw = oracle.quant_rows_ref(w.reshape(G * N, K))
        sw = sw.reshape(G, N)
    return offsets, qa, sa, qw.reshape(G, N, K), sw


def _expected(mode, offsets, qa, sa, qw, sw, rows=None):
    """Oracle output and its error bound on the given rows."""
    K = qa.shape[1]
    mag_a, mag_w = qa & 0x7F, qw & 0x7F          # |e4m3| codes
    if mode == "ptpc":
        want = np.arange(qa.shape[0]) if rows is None else np.asarray(rows)
        y = np.full((len(want), qw.shape[1]), np.nan)
        mag = np.full_like(y, np.nan)
        for g in range(len(offsets) - 1):
            sel = np.flatnonzero((want >= offsets[g]) & (want < offsets[g + 1]))
            if sel.size:
                r = want[sel]
                y[sel] = oracle.ptpc_matmul_ref(qa[r], sa[r], qw[g], sw[g])
                mag[sel] = oracle.ptpc_matmul_ref(mag_a[r], sa[r], mag_w[g], sw[g])
        return y, gemm_bound(mag, K + 5)
    y = oracle.grouped_blockscale_ref(qa, sa, qw, sw, offsets, mode, rows=rows)
    mag = oracle.grouped_blockscale_ref(mag_a, sa, mag_w, sw, offsets, mode, rows=rows)
    gsize = 128 if mode == "block128" else 512
    return y, gemm_bound(mag, gsize + K // gsize + 4)


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("offsets,N,K", [
    ([0, 130, 130, 300, 301, 420], 256, 1024),   # empty group, 1-row group, ragged tails
    ([0, 64], 128, 512),
    ([0, 0, 257], 384, 2048),
])
def test_grouped_gemm_scaled(mode, offsets, N, K):
    offsets, qa, sa, qw, sw = _problem(mode, offsets, N, K, len(offsets) * N + K)
    R = qa.shape[0]
    out = torch.full((R, N), float("nan"), dtype=torch.float32, device="cuda")
    B().moe_grouped_gemm_scaled(MODES[mode], cuda(qa), cuda(sa), cuda(qw), cuda(sw),
                                cuda(offsets), out=out)
    assert B().moe_device_status() == (0, 0)
    got = out.cpu().numpy().astype(np.float64)
    y, bound = _expected(mode, offsets, qa, sa, qw, sw)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - y) <= bound)


@pytest.mark.parametrize("mode", ["ptpc", "block128"])
def test_grouped_gemm_scaled_odd_k_blocks(mode):
    """K = 640: five 128-wide blocks, an odd number of scale groups for
    BlockScale-128 (512-subchannel needs K a multiple of 512)."""
    offsets, qa, sa, qw, sw = _problem(mode, [0, 70, 200], 256, 640, 41)
    out = torch.full((200, 256), float("nan"), dtype=torch.float32, device="cuda")
    B().moe_grouped_gemm_scaled(MODES[mode], cuda(qa), cuda(sa), cuda(qw), cuda(sw),
                                cuda(offsets), out=out)
    assert B().moe_device_status() == (0, 0)
    y, bound = _expected(mode, offsets, qa, sa, qw, sw)
    assert np.all(np.abs(out.cpu().numpy().astype(np.float64) - y) <= bound)


def test_sub512_rejects_k_off_its_blocks():
    offsets, qa, sa, qw, sw = _problem("ptpc", [0, 8], 128, 640, 5)
    with pytest.raises(B().MoeError) as e:
        B().moe_grouped_gemm_scaled(MODES["sub512"], cuda(qa), cuda(np.ones((8, 1), np.float32)),
                                    cuda(qw), cuda(sw), cuda(offsets))
    assert e.value.status == -2          # MOE_ERR_UNSUPPORTED, before any launch


def test_rows_outside_every_group_untouched():
    offsets, qa, sa, qw, sw = _problem("block128", [0, 100], 128, 256, 3)
    qa = np.concatenate([qa, qa[:28]])            # 28 rows owned by no group
    sa = np.concatenate([sa, sa[:28]])
    out = torch.full((128, 128), 7.0, dtype=torch.float32, device="cuda")
    B().moe_grouped_gemm_scaled(2, cuda(qa), cuda(sa), cuda(qw), cuda(sw), cuda(offsets),
                                out=out)
    assert torch.all(out[100:] == 7.0)


@pytest.mark.parametrize("mode", sorted(MODES))
@pytest.mark.parametrize("which", ["gateup", "down"])
def test_scaled_gemm_prefill_shape_sampled(mode, which):
    """The launches the block-scale comparison times: the prefill workload's
    gate/up-shaped (N = 3072, K = 4096) and down-shaped (N = 4096, K = 1536)
    grouped GEMMs over 65536 routed rows and 128 experts, operands quantised
    on the GPU. On sampled rows: the activation codes and scales against the
    oracle's quantiser, the weights of the experts they use against the
    oracle's, and the outputs against the oracle GEMM."""
    from expert_layer_ptpc_gb300 import scaled
    from expert_layer_ptpc_gb300 import synthetic as syn
    prob = scaled.make_problem(mode, syn.CONFIGS["prefill"], which)
    out = scaled.run(prob)
    torch.cuda.synchronize()
    assert B().moe_device_status() == (0, 0)
    offsets = prob["offsets"].cpu().numpy()
    R = int(offsets[-1])
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(R, 5, replace=False))
    rows[-1] = R - 1
    ridx = torch.as_tensor(rows, device="cuda").long()
    x = prob["x_rows"](rows)
    qa = prob["qa"][ridx].cpu().numpy()
    sa = prob["sa"][ridx].cpu().numpy()
    if mode == "ptpc":
        rq, rs = oracle.quant_rows_ref(x)
    else:
        rq, rs = oracle.quant_blocks_ref(x, 128 if mode == "block128" else 512)
    assert np.array_equal(qa, rq)
    assert np.array_equal(sa.view(np.uint32), rs.view(np.uint32))
    got = out[ridx].cpu().numpy().astype(np.float64)
    for i, r in enumerate(rows):
        g = int(np.searchsorted(offsets, r, side="right") - 1)
        qw = prob["qw"][g].cpu().numpy()
        sw = prob["sw"][g].cpu().numpy()
        w = prob["w_raw"](g)
        if mode == "block128":
            wq, ws = oracle.quant_weight_blocks_ref(w)
        else:
            wq, ws = oracle.quant_rows_ref(w)
        assert np.array_equal(qw, wq)
        assert np.array_equal(sw.view(np.uint32), ws.view(np.uint32))
        one = np.array([0, 1])
        y, bound = _expected(mode, one, qa[i:i + 1], sa[i:i + 1], qw[None], sw[None])
        assert np.all(np.abs(got[i] - y[0]) <= bound[0]), (mode, which, r)
