"""Host models of the grouped GEMMs' mbarrier protocols, checked under
random interleavings (no GPU): the CTA-pair stage ring, the accumulator
buffers between the MMA issuer and the epilogue warps, and the scheduler's
tile ring.

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


def simulate_accumulators(A, warps, tiles, seed):
    """The accumulator buffers between the MMA issuer and the epilogue warps:
    tile i uses buffer i % A; the issuer waits until every epilogue warp has
    released the buffer's previous tile (acce), then commits it full (accf);
    each epilogue warp waits for accf, reads, and arrives on acce."""
    rng = random.Random(seed)
    accf = [0] * A           # completed phases: a tile's accumulators ready
    acce = [0] * A           # completed phases: every warp released a tile
    arrivals = [0] * A
    bad = []
    mma_next = 0
    epi_next = [0] * warps

    def check(hw, intended, what):
        if hw != intended:
            bad.append(what)
        return hw

    def mma():
        nonlocal mma_next
        i = mma_next
        if i >= tiles:
            return
        b, j = i % A, i // A
        if check(parity_wait(acce[b], (j & 1) ^ 1), acce[b] >= j, ("mma", i, acce[b])):
            accf[b] += 1
            mma_next += 1

    def epi(w):
        i = epi_next[w]
        if i >= tiles:
            return
        b, j = i % A, i // A
        if check(parity_wait(accf[b], j & 1), accf[b] >= j + 1, ("epi", w, i, accf[b])):
            arrivals[b] += 1
            if arrivals[b] == warps:
                arrivals[b] = 0
                acce[b] += 1
            epi_next[w] += 1

    for _ in range(tiles * (warps + 2) * 60):
        if bad or (mma_next >= tiles and min(epi_next) >= tiles):
            break
        a = rng.randrange(warps + 1)
        if a == warps:
            mma()
        else:
            epi(a)
    return bad, mma_next >= tiles and min(epi_next) >= tiles


def simulate_tile_ring(R, consumers, tiles, seed):
    """The scheduler's tile ring: the scheduler publishes tiles 0..tiles-1
    and the end marker into slot n % R once every consumer has read the
    slot's previous entry; each consumer reads every entry in order. One
    consumer (the first producer) also marks each tile it takes, and the
    scheduler waits for that mark before it asks for the next tile."""
    rng = random.Random(seed)
    full = [0] * R
    empty = [0] * R
    arrivals = [0] * R
    taken = 0
    bad = []
    published = 0              # entries published (tiles, then the marker)
    waits_taken = 0
    pending_take = False
    read = [0] * consumers
    ring = [None] * R

    def check(hw, intended, what):
        if hw != intended:
            bad.append(what)
        return hw

    def sched():
        nonlocal published, waits_taken, pending_take
        if published > tiles:
            return
        if pending_take:
            m = waits_taken
            if not check(parity_wait(taken, m & 1), taken >= m + 1, ("taken", m, taken)):
                return
            waits_taken += 1
            pending_take = False
            return
        n = published
        s, r = n % R, n // R
        if not check(parity_wait(empty[s], (r & 1) ^ 1), empty[s] >= r,
                     ("publish", n, empty[s])):
            return
        ring[s] = n if n < tiles else -1
        full[s] += 1
        published += 1
        pending_take = n < tiles

    def consume(c):
        nonlocal taken
        n = read[c]
        if n > tiles:
            return
        s, r = n % R, n // R
        if not check(parity_wait(full[s], r & 1), full[s] >= r + 1, ("read", c, n, full[s])):
            return
        t = ring[s]
        if t != (n if n < tiles else -1):
            bad.append(("value", c, n, t))
        arrivals[s] += 1
        if arrivals[s] == consumers:
            arrivals[s] = 0
            empty[s] += 1
        if c == 0 and t >= 0:
            taken += 1
        read[c] += 1

    for _ in range((tiles + 2) * (consumers + 2) * 80):
        if bad or (published > tiles and min(read) > tiles):
            break
        a = rng.randrange(consumers + 1)
        if a == consumers:
            sched()
        else:
            consume(a)
    return bad, published > tiles and min(read) > tiles


@pytest.mark.parametrize("A,warps", [(1, 4), (2, 4), (2, 8), (2, 16), (1, 16)])
def test_accumulator_buffers_never_alias(A, warps):
    for seed in range(30):
        for tiles in (1, 2, 3, 7, 33):
            bad, done = simulate_accumulators(A, warps, tiles, seed * 100 + tiles)
            assert not bad, (A, warps, tiles, seed, bad[:3])
            assert done, (A, warps, tiles, seed)


@pytest.mark.parametrize("consumers", [5, 11, 15, 19])
def test_tile_ring_never_aliases(consumers):
    """kRing = 4 slots; consumers as sched_init counts them (producer warps,
    epilogue warps and, in the leader, the MMA issuer)."""
    for seed in range(20):
        for tiles in (0, 1, 3, 4, 5, 17):
            bad, done = simulate_tile_ring(4, consumers, tiles, seed * 100 + tiles)
            assert not bad, (consumers, tiles, seed, bad[:3])
            assert done, (consumers, tiles, seed)
