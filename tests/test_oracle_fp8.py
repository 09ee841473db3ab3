"""Pins of the oracle's number formats against the e4m3 specification values,
torch's own fp8 / bf16 conversions, and properties that fix the rounding."""

import os

import numpy as np
import pytest
import torch

from oracle import bf16_round, e4m3_decode, e4m3_encode

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_values.txt")


def _golden():
    out = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            code, val = line.split()
            out.append((int(code, 16), float(val)))
    return out


def test_decode_matches_spec_values():
    for code, val in _golden():
        got = e4m3_decode(np.array([code], np.uint8))[0]
        assert got == val and np.signbit(got) == np.signbit(val), hex(code)


def test_decode_nan_codes():
    v = e4m3_decode(np.array([0x7F, 0xFF], np.uint8))
    assert np.isnan(v).all()


def test_decode_monotone_and_roundtrip():
    codes = np.arange(0, 0x7F, dtype=np.uint8)          # all non-negative finite
    vals = e4m3_decode(codes)
    assert np.all(np.diff(vals) > 0)
    assert np.array_equal(e4m3_encode(vals), codes)
    neg = codes | 0x80
    assert np.array_equal(e4m3_encode(e4m3_decode(neg)), neg)


def test_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_decode(codes.numpy())
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(got[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(ref), np.isnan(got))


def test_encode_matches_torch_in_range(rng):
    # torch's fp32 -> float8_e4m3fn cast rounds to nearest even inside the
    # finite range; compare on random values spanning every binade.
    mag = np.exp2(rng.uniform(-12, np.log2(448.0), size=200_000))
    v = (mag * rng.choice([-1.0, 1.0], size=mag.size)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode(v), ref)


def test_encode_ties_to_even():
    vals = e4m3_decode(np.arange(0, 0x7E, dtype=np.uint8))
    nxt = e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8))
    mid = ((vals + nxt) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (vals + nxt) / 2)  # exact
    got = e4m3_encode(mid)
    lo = np.arange(0, 0x7E)
    expect = np.where(lo % 2 == 0, lo, lo + 1)   # the even mantissa wins
    assert np.array_equal(got, expect.astype(np.uint8))


def test_encode_saturates():
    v = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, np.inf,
                  -448.5, -1e30, -np.inf], np.float32)
    got = e4m3_encode(v)
    assert list(got[:7]) == [0x7E] * 7
    assert list(got[7:]) == [0xFE] * 3
    assert e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


def test_encode_subnormal_and_zero():
    q = 2.0 ** -9
    v = np.array([0.0, -0.0, q * 0.49, q * 0.5, q * 0.51, q * 1.5, q * 2.5,
                  q * 7.5, q * 7.49], np.float32)
    got = e4m3_encode(v)
    assert list(got) == [0x00, 0x80, 0x00, 0x00, 0x01, 0x02, 0x02, 0x08, 0x07]


@pytest.mark.parametrize("scale", [1.0, 1e-3, 1e3, 1e-30, 1e30])
def test_bf16_round_matches_torch(rng, scale):
    v = (rng.standard_normal(100_000) * scale).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(bf16_round(v.astype(np.float64)), ref)


def test_bf16_round_ties_to_even():
    # 1 + 2^-8 lies half way between bf16 1.0 and 1 + 2^-7: even is 1.0.
    assert bf16_round(np.array([1.0 + 2 ** -8]))[0] == 1.0
    assert bf16_round(np.array([1.0 + 3 * 2 ** -8]))[0] == 1.0 + 2 ** -6


# ---------------------------------------------------------------------------
# exhaustive: every fp32 bit pattern
# ---------------------------------------------------------------------------
_EXH_CHUNK_BITS = 24


def _exhaustive_chunk(c):
    """Mismatches between the oracle's encoder and torch's float8_e4m3fn cast
    over the 2^24 fp32 bit patterns of chunk c. torch's cast rounds to
    nearest even inside the finite range but is not saturating (it gives NaN
    beyond it), so its input is first clipped to +-448, which the OCP
    saturating rule maps every larger magnitude to. NaN inputs must give a
    NaN code (exponent and mantissa all ones) on both sides."""
    import numpy as np
    import torch
    torch.set_num_threads(1)
    from oracle import e4m3_encode
    bits = np.arange(c << _EXH_CHUNK_BITS, (c + 1) << _EXH_CHUNK_BITS,
                     dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    got = e4m3_encode(v)
    ref = torch.from_numpy(np.clip(v, -448.0, 448.0)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    nan = np.isnan(v)
    bad = (got != ref) & ~nan
    bad |= nan & ((got & 0x7F) != 0x7F)
    first = int(bits[np.flatnonzero(bad)[0]]) if bad.any() else -1
    return int(bad.sum()), first


def test_encode_exhaustive_all_fp32():
    """The encoder on all 2^32 fp32 bit patterns (both zeros, every
    subnormal and normal, both infinities, every NaN) against torch's cast
    with saturation, in 256 chunks over a spawn-started process pool."""
    import multiprocessing as mp
    n_chunks = 1 << (32 - _EXH_CHUNK_BITS)
    workers = max(1, min(16, os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(workers) as pool:
        res = pool.map(_exhaustive_chunk, range(n_chunks), chunksize=1)
    bad = [(c, n, f) for c, (n, f) in enumerate(res) if n]
    assert not bad, f"mismatching chunks (chunk, count, first bits): {bad[:5]}"
