"""A host model of the CTA-pair GEMM's stage ring, checked under random
interleavings (no GPU).

The kernel's producer warps take turns by stage: warp p of a box issues the
stages q with q % P == p into slot q % S, after waiting for the slot's
previous stage to be consumed; the MMA issuer consumes the stages in order;
at the end each warp waits for the consumption of its own last stage. Every
wait is an mbarrier parity wait: "the phase with parity b has completed" is
read as "the barrier's current phase has the other parity", which equals
the intended condition only while the barrier is at most one phase away
from the one the waiter means. The model drives every wait by that parity
rule, compares it with the intended condition at each evaluation, and
checks that the two never differ for the producer counts and ring depths
the kernel instantiates (P <= S), and that they do differ in some
interleaving when P > S, so the check has teeth.
"""
import random

import pytest


def parity_wait(completed, parity):
    """mbarrier try_wait.parity: true when the current phase (index =
    completed phases) does not have the given parity."""
    return (completed & 1) != parity


def simulate(S, P, boxes, stages, seed):
    """One random interleaving of `boxes` x `P` producer warps and the MMA
    issuer over `stages` stages in an S-slot ring. Returns (mismatches,
    finished)."""
    rng = random.Random(seed)
    full = [0] * S          # completed phases: a stage's boxes all landed
    arrivals = [0] * S
    empty = [0] * S         # completed phases: a stage consumed
    bad = []
    nxt = {(b, p): p for b in range(boxes) for p in range(P)}
    last = {k: -1 for k in nxt}
    drained = {k: False for k in nxt}
    consumed = 0

    def check(hw, intended, what):
        if hw != intended:
            bad.append(what)
        return hw

    def producer(k):
        q = nxt[k]
        if q >= stages:                      # drain on the last own stage
            lq = last[k]
            if lq < 0:
                drained[k] = True
                return
            s, j = lq % S, lq // S
            if check(parity_wait(empty[s], j & 1), empty[s] >= j + 1,
                     ("drain", k, lq, empty[s])):
                drained[k] = True
            return
        s, j = q % S, q // S
        # the slot's previous stage (q - S) consumed: empty[s] reached j
        if not check(parity_wait(empty[s], (j & 1) ^ 1), empty[s] >= j,
                     ("produce", k, q, empty[s])):
            return
        arrivals[s] += 1
        if arrivals[s] == boxes:
            arrivals[s] = 0
            full[s] += 1
        last[k] = q
        nxt[k] = q + P

    def mma():
        nonlocal consumed
        q = consumed
        if q >= stages:
            return
        s, j = q % S, q // S
        if check(parity_wait(full[s], j & 1), full[s] >= j + 1,
                 ("consume", q, full[s])):
            empty[s] += 1
            consumed += 1

    actors = list(nxt) + ["mma"]
    for _ in range(stages * (len(actors) + 2) * 60):
        if bad or (consumed >= stages and all(drained.values())):
            break
        a = rng.choice(actors)
        if a == "mma":
            mma()
        elif not drained[a]:
            producer(a)
    return bad, consumed >= stages and all(drained.values())


# (ring slots S, producer warps per box P, boxes) the kernel instantiates:
# one-atom stages (two warps per box with an even S, else one) and two-atom
# stages (BN 192: S = 3, P = 3, 2 boxes; BN 128: S = 4, P = 3, 2 boxes;
# BN 256: S = 3, P = 2, 3 boxes)
CONFIGS = [(7, 1, 2), (6, 2, 3), (8, 2, 2), (10, 2, 2), (4, 1, 5),
           (3, 3, 2), (4, 3, 2), (3, 2, 3), (3, 1, 2)]


@pytest.mark.parametrize("S,P,boxes", CONFIGS)
def test_ring_waits_never_alias(S, P, boxes):
    for seed in range(30):
        for stages in sorted({1, 2, S - 1, S, S + 1, 3 * S + 2, 48}):
            bad, done = simulate(S, P, boxes, stages, seed * 1000 + stages)
            assert not bad, (S, P, boxes, stages, seed, bad[:3])
            assert done, (S, P, boxes, stages, seed)


def test_more_turns_than_slots_aliases():
    """With P > S a warp can reach a slot two uses ahead of its barrier,
    where the parity wait passes wrongly: the model must catch it."""
    assert any(simulate(2, 3, 1, 30, seed)[0] for seed in range(300))
