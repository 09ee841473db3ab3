"""Pins of the BlockScale-128 and 512-subchannel oracle (MI300X page, section
2.1.1; the MI355X page's per-128 fp32 blockwise scales; the TPU page's 512
subchannel activations) against special cases that reduce to the pinned PTPC
quantiser and GEMM, exact rational arithmetic, a dequantise-first evaluation
and invariants."""

from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle.fp8 import e4m3_decode


def _rows(R, K, seed, outliers=True):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((R, K)).astype(np.float32)
    if outliers:   # blocks of very different magnitude, where block scales matter
        for r in range(R):
            b = rng.integers(0, K // 128)
            v[r, b * 128:(b + 1) * 128] *= np.float32(2.0 ** rng.integers(-12, 12))
    return v


def test_one_block_per_row_is_the_ptpc_quantiser():
    """A block as wide as the row is the per-token quantiser."""
    v = _rows(9, 256, 1)
    c, s = oracle.quant_blocks_ref(v, 256)
    rc, rs = oracle.quant_rows_ref(v)
    assert np.array_equal(c, rc)
    assert np.array_equal(s[:, 0].view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("block", [128, 512])
def test_each_block_is_quantised_on_its_own(block):
    """Slice by slice: block b of row r is the per-token quantiser applied to
    v[r, b*block:(b+1)*block] alone."""
    v = _rows(5, 1024, 2)
    c, s = oracle.quant_blocks_ref(v, block)
    assert s.shape == (5, 1024 // block)
    for r in range(5):
        for b in range(1024 // block):
            sl = v[r:r + 1, b * block:(b + 1) * block]
            rc, rs = oracle.quant_rows_ref(sl)
            assert np.array_equal(c[r:r + 1, b * block:(b + 1) * block], rc)
            assert s[r, b] == rs[0]


def test_block_scale_invariance():
    """Multiplying one block by 2^j multiplies only its scale by 2^j; every
    code stays the same (the quantiser is exact under powers of two away
    from the clamp)."""
    v = _rows(4, 512, 3, outliers=False)
    c0, s0 = oracle.quant_blocks_ref(v, 128)
    w = v.copy()
    w[2, 256:384] *= np.float32(2.0 ** 7)
    c1, s1 = oracle.quant_blocks_ref(w, 128)
    assert np.array_equal(c0, c1)
    expect = s0.copy()
    expect[2, 2] *= np.float32(2.0 ** 7)
    assert np.array_equal(s1, expect)


def test_weight_block_is_a_per_tensor_quantiser():
    """A 128 x 128 weight matrix is one block: one scale from its global amax
    (the per-token quantiser on the flattened matrix as a single row)."""
    w = _rows(128, 128, 4)
    c, s = oracle.quant_weight_blocks_ref(w)
    rc, rs = oracle.quant_rows_ref(w.reshape(1, -1))
    assert s.shape == (1, 1) and s[0, 0] == rs[0]
    assert np.array_equal(c, rc.reshape(128, 128))


def test_weight_blocks_slice_by_slice():
    w = _rows(256, 384, 5)
    c, s = oracle.quant_weight_blocks_ref(w)
    assert s.shape == (2, 3)
    for i in range(2):
        for b in range(3):
            blk = w[i * 128:(i + 1) * 128, b * 128:(b + 1) * 128]
            rc, rs = oracle.quant_rows_ref(blk.reshape(1, -1))
            assert s[i, b] == rs[0]
            assert np.array_equal(c[i * 128:(i + 1) * 128, b * 128:(b + 1) * 128],
                                  rc.reshape(128, 128))


def test_quantisation_error_bound():
    """e4m3 keeps 3 mantissa bits: every dequantised entry is within 2^-4 of
    its value relative, plus half the subnormal spacing (2^-10) times the
    scale."""
    v = _rows(6, 512, 6)
    for block in (128, 512):
        c, s = oracle.quant_blocks_ref(v, block)
        deq = e4m3_decode(c) * np.repeat(s.astype(np.float64), block, axis=1)
        err = np.abs(deq - v.astype(np.float64))
        bound = 2.0 ** -4 * np.abs(v) + np.repeat(s.astype(np.float64), block, axis=1) * 2.0 ** -10
        assert np.all(err <= bound * (1 + 1e-12))


def test_block_scales_beat_per_token_scales_on_outlier_blocks():
    """The reason for block scales: in a row whose one block is 2^16 larger,
    the other blocks fall into e4m3's subnormals under one per-token scale,
    and keep 3 mantissa bits under per-block scales."""
    rng = np.random.default_rng(7)
    v = rng.standard_normal((1, 512)).astype(np.float32)
    v[0, :128] *= np.float32(65536.0)
    cb, sb = oracle.quant_blocks_ref(v, 128)
    cp, sp = oracle.quant_rows_ref(v)
    small = slice(128, 512)
    eb = np.abs(e4m3_decode(cb)[0, small] * np.repeat(sb[0], 128)[small] - v[0, small])
    ep = np.abs(e4m3_decode(cp)[0, small] * sp[0] - v[0, small])
    assert eb.mean() * 5 < ep.mean()


def _quantised_pair(R, N, K, seed, mode):
    rng = np.random.default_rng(seed)
    a = _rows(R, K, seed)
    w = (rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32)
    w[:, :128] *= np.float32(8.0)
    if mode == "block128":
        qa, sa = oracle.quant_blocks_ref(a, 128)
        qw, sw = oracle.quant_weight_blocks_ref(w)
    else:
        qa, sa = oracle.quant_blocks_ref(a, 512)
        qw, sw = oracle.quant_rows_ref(w)
    return qa, sa, qw, sw


def test_blockscale_matmul_equals_dequantise_first():
    """Scaling each exact block product by its scales equals multiplying the
    dequantised matrices (an independent evaluation: no block sums)."""
    qa, sa, qw, sw = _quantised_pair(7, 256, 512, 8, "block128")
    y = oracle.blockscale_matmul_ref(qa, sa, qw, sw)
    A = e4m3_decode(qa) * np.repeat(sa.astype(np.float64), 128, axis=1)
    swf = np.repeat(np.repeat(sw.astype(np.float64), 128, axis=0), 128, axis=1)
    W = e4m3_decode(qw) * swf
    np.testing.assert_allclose(y, A @ W.T, rtol=1e-12, atol=1e-12 * np.abs(A @ W.T).max())


def test_subchannel_matmul_equals_dequantise_first():
    qa, sa, qw, sw = _quantised_pair(6, 128, 1024, 9, "sub512")
    y = oracle.subchannel_matmul_ref(qa, sa, qw, sw)
    A = e4m3_decode(qa) * np.repeat(sa.astype(np.float64), 512, axis=1)
    W = e4m3_decode(qw) * sw.astype(np.float64)[:, None]
    np.testing.assert_allclose(y, A @ W.T, rtol=1e-12, atol=1e-12 * np.abs(A @ W.T).max())


def test_equal_block_scales_reduce_to_ptpc():
    """With one scale per row repeated over its blocks, and one per weight
    block row repeated over K, both variants are the pinned PTPC GEMM."""
    rng = np.random.default_rng(10)
    R, N, K = 5, 256, 1024
    qa = rng.integers(0, 256, (R, K)).astype(np.uint8)
    qw = rng.integers(0, 256, (N, K)).astype(np.uint8)
    qa[(qa & 0x7f) == 0x7f] = 0      # no NaN codes
    qw[(qw & 0x7f) == 0x7f] = 0
    s_row = (rng.random(R) + 0.5).astype(np.float32)
    s_blk = (rng.random(N // 128) + 0.5).astype(np.float32)
    ref = oracle.ptpc_matmul_ref(qa, s_row, qw, np.repeat(s_blk, 128))
    y = oracle.blockscale_matmul_ref(qa, np.repeat(s_row[:, None], K // 128, 1), qw,
                                     np.repeat(s_blk[:, None], K // 128, 1))
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=0)
    s_ch = (rng.random(N) + 0.5).astype(np.float32)
    ref = oracle.ptpc_matmul_ref(qa, s_row, qw, s_ch)
    y = oracle.subchannel_matmul_ref(qa, np.repeat(s_row[:, None], K // 512, 1), qw, s_ch)
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=0)


def test_block_products_are_exact():
    """The block partial sums equal exact rational sums of the decoded codes
    (brute force on a tiny case)."""
    rng = np.random.default_rng(11)
    qa = rng.integers(0, 256, (2, 256)).astype(np.uint8)
    qw = rng.integers(0, 256, (2, 256)).astype(np.uint8)
    qa[(qa & 0x7f) == 0x7f] = 1
    qw[(qw & 0x7f) == 0x7f] = 1
    sa = np.array([[0.5, 3.0], [1.25, 0.125]], np.float32)
    sw = np.array([[2.0, 0.75]], np.float32)
    y = oracle.blockscale_matmul_ref(qa, sa, np.concatenate([qw] * 64), sw)[:, :2]
    da, dw = e4m3_decode(qa), e4m3_decode(qw)
    for r in range(2):
        for n in range(2):
            tot = Fraction(0)
            for b in range(2):
                p = sum(Fraction(float(da[r, k])) * Fraction(float(dw[n, k]))
                        for k in range(b * 128, (b + 1) * 128))
                tot += Fraction(float(sa[r, b])) * Fraction(float(sw[0, b])) * p
            assert abs(Fraction(float(y[r, n])) - tot) <= abs(tot) * Fraction(1, 2 ** 50)


def test_grouped_reference_uses_each_groups_weights():
    rng = np.random.default_rng(12)
    R, N, K, G = 40, 128, 256, 3
    qa, sa = oracle.quant_blocks_ref(_rows(R, K, 13), 128)
    qws, sws = [], []
    for g in range(G):
        q, s = oracle.quant_weight_blocks_ref(rng.standard_normal((N, K)).astype(np.float32))
        qws.append(q)
        sws.append(s)
    offs = np.array([0, 11, 11, 40])
    y = oracle.grouped_blockscale_ref(qa, sa, np.stack(qws), np.stack(sws), offs, "block128")
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        if hi > lo:
            np.testing.assert_array_equal(
                y[lo:hi], oracle.blockscale_matmul_ref(qa[lo:hi], sa[lo:hi], qws[g], sws[g]))
    rows = np.array([0, 10, 11, 39])
    ys = oracle.grouped_blockscale_ref(qa, sa, np.stack(qws), np.stack(sws), offs,
                                       "block128", rows=rows)
    np.testing.assert_array_equal(ys, y[rows])
