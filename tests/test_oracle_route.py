"""Pins of the oracle's routing and permutation: hand-worked cases, properties
that determine the answer uniquely, and library special cases."""

import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

from oracle import permute_ref, route_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "route_cases.txt")


def _cases():
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        k, lg, ids, ws = [p.strip() for p in line.split("|")]
        logits = [np.log(float(tok[1:])) for tok in lg.split()]
        yield (int(k), np.array([logits], np.float32),
               [int(i) for i in ids.split()],
               [float(Fraction(w)) for w in ws.split()])


@pytest.mark.parametrize("case", list(_cases()))
def test_golden_cases(case):
    k, logits, ids, ws = case
    got_ids, got_w = route_ref(logits, k)
    assert list(got_ids[0]) == ids
    assert np.allclose(got_w[0], ws, rtol=1e-6, atol=0)


def _check_selection_properties(logits, ids, k):
    """The k-subset and its order are fixed by: every chosen expert beats every
    unchosen one under (higher logit, then lower index); the chosen list is
    ordered by the same rule; ids are distinct."""
    T, E = logits.shape
    for t in range(T):
        sel = [int(e) for e in ids[t]]
        assert len(set(sel)) == k
        rest = [e for e in range(E) if e not in sel]

        def beats(a, b):
            la, lb = logits[t, a], logits[t, b]
            return la > lb or (la == lb and a < b)
        for a in sel:
            for b in rest:
                assert beats(a, b), (t, a, b)
        for a, b in zip(sel, sel[1:]):
            assert beats(a, b), (t, a, b)


@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (6, 3), (8, 8), (16, 5)])
def test_selection_properties_with_ties(rng, E, k):
    # Small integer logits make ties common.
    logits = rng.integers(-2, 3, size=(200, E)).astype(np.float32)
    ids, w = route_ref(logits, k)
    _check_selection_properties(logits, ids, k)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_all_equal_logits():
    ids, w = route_ref(np.zeros((3, 10), np.float32), 4)
    assert (ids == np.arange(4)).all()
    assert np.allclose(w, 0.25, rtol=0, atol=1e-15)


def test_k_equals_E_is_full_softmax(rng):
    logits = rng.standard_normal((50, 12)).astype(np.float32)
    ids, w = route_ref(logits, 12)
    dense = np.zeros_like(w)
    np.put_along_axis(dense, ids.astype(np.int64), w, axis=1)
    ref = scipy.special.softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(dense, ref, rtol=1e-13, atol=0)


def test_no_renormalise_is_plain_softmax(rng):
    logits = rng.standard_normal((50, 16)).astype(np.float32)
    ids, w = route_ref(logits, 3, renormalize=False)
    ref = scipy.special.softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(ref, ids.astype(np.int64), 1),
                       rtol=1e-13, atol=0)


def test_renormalised_weight_ratios(rng):
    logits = (rng.standard_normal((100, 32)) * 3).astype(np.float32)
    ids, w = route_ref(logits, 6)
    chosen = np.take_along_axis(logits.astype(np.float64),
                                ids.astype(np.int64), 1)
    assert np.allclose(w[:, 1:] / w[:, :1], np.exp(chosen[:, 1:] - chosen[:, :1]),
                       rtol=1e-12)


@pytest.mark.parametrize("T,E,k", [(1, 4, 1), (37, 8, 2), (300, 64, 6),
                                   (64, 5, 5)])
def test_permute_invariants(rng, T, E, k):
    logits = rng.standard_normal((T, E)).astype(np.float32)
    ids, _ = route_ref(logits, k)
    counts, offsets, s2f, f2s = permute_ref(ids, E)
    R = T * k
    flat = ids.reshape(-1)
    assert counts.sum() == R
    assert offsets[0] == 0 and offsets[-1] == R
    assert np.all(np.diff(offsets) == counts)
    assert np.array_equal(np.sort(s2f), np.arange(R))
    assert np.array_equal(s2f[f2s], np.arange(R))         # mutually inverse
    assert np.array_equal(f2s[s2f], np.arange(R))
    for e in range(E):
        seg = s2f[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)                   # stable: ascending f
    # permute then unpermute is the identity on row payloads
    payload = rng.standard_normal((R, 3))
    permuted = payload[s2f]
    assert np.array_equal(permuted[f2s], payload)
    # the stable library sort gives the same order
    assert np.array_equal(s2f, np.argsort(flat, kind="stable"))


def test_permute_empty_experts():
    ids = np.array([[3, 1], [3, 0], [1, 3]], np.int32)
    counts, offsets, s2f, f2s = permute_ref(ids, 6)
    assert list(counts) == [1, 2, 0, 3, 0, 0]
    assert list(offsets) == [0, 1, 3, 3, 6, 6, 6]
    assert list(s2f) == [3, 1, 4, 0, 2, 5]
    # f0->3, f1->1, f2->4, f3->0, f4->2, f5->5
    assert list(f2s) == [3, 1, 4, 0, 2, 5]
