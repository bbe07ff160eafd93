"""The block-score kernel's barrier protocol, modelled on the CPU.

Producer, MMA issuers and epilogue warps run as processes in random
interleavings over mbarriers that count arrivals and transaction bytes by
phase, as the hardware does (expect-tx raises the byte count before its own
arrival, and a phase completes when both reach zero).  The model checks:
  - an arrival or a copy's bytes never land on a stage barrier while its
    previous phase is still open (they would complete the wrong tile);
  - every tile is issued, and nothing deadlocks;
  - a stage ring shallower than the accumulator ring breaks the first rule, and so
    does an odd stage ring with two issuers.

Protocol (one stage barrier per operand stage): tile j waits on go[j % S];
that phase completes when the producer's copies for tile j have landed and
all epilogue warps have released the accumulator tile j - A used (they arrive
on go[(i + A) % S] when they release tile i; the first A tiles are released at
start).  Tiles are issued by I issuers in turn (tile j by issuer j % I)."""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pend, self.tx, self.phase, self.tag = count, count, 0, 0, None

    def arrive(self, tag, n=1):
        if self.tag is not None and self.tag != tag:
            raise AssertionError(f"arrival for {tag} while the open phase belongs to {self.tag}")
        self.tag = tag
        self.pend -= n
        self._check()

    def expect_tx(self, tag, nbytes):  # raises the byte count, then arrives (one step in hardware)
        self.tx += nbytes
        self.arrive(tag)

    def complete_tx(self, tag, nbytes):
        if self.tag is not None and self.tag != tag:
            raise AssertionError(f"bytes for {tag} while the open phase belongs to {self.tag}")
        self.tag = tag
        self.tx -= nbytes
        self._check()

    def _check(self):
        if self.pend == 0 and self.tx == 0:
            self.phase += 1
            self.pend, self.tag = self.count, None

    def done(self, parity):  # the phase of this parity has completed
        return (self.phase & 1) != parity


def run(S, A, n_tiles, seed, warps=4, issuers=1):
    rnd = random.Random(seed)
    go = [Bar(1 + warps) for _ in range(S)]
    empty = [Bar(1) for _ in range(S)]
    acc_full = [Bar(1) for _ in range(A)]
    for j in range(A):
        for _ in range(warps):
            go[j % S].arrive(("tile", j))
    prod = 0
    copies = []                      # (tile, half) copies in flight
    nxt = [i for i in range(issuers)]  # next tile of each issuer
    in_pipe = []                     # issued, not yet complete (tensor pipe is in order)
    epi = [0] * warps
    for _ in range(10 ** 6):
        acts = []
        if prod < n_tiles and empty[prod % S].done(((prod // S) & 1) ^ 1):
            acts.append(("produce",))
        if copies:
            acts.append(("land",))
        for k in range(issuers):
            j = nxt[k]
            if j < n_tiles and go[j % S].done((j // S) & 1):
                acts.append(("issue", k))
        if in_pipe:
            acts.append(("complete",))
        for w in range(warps):
            i = epi[w]
            if i < n_tiles and acc_full[i % A].done((i // A) & 1):
                acts.append(("release", w))
        if not acts:
            assert prod == n_tiles and all(j >= n_tiles for j in nxt) and all(i == n_tiles for i in epi), "deadlock"
            return
        a = rnd.choice(acts)
        if a[0] == "produce":
            go[prod % S].expect_tx(("tile", prod), 2)
            copies += [(prod, 0), (prod, 1)]
            prod += 1
        elif a[0] == "land":
            j, _ = copies.pop(rnd.randrange(len(copies)))
            go[j % S].complete_tx(("tile", j), 1)
        elif a[0] == "issue":
            j = nxt[a[1]]
            in_pipe.append(j)
            nxt[a[1]] += issuers
        elif a[0] == "complete":
            j = in_pipe.pop(0)          # the tensor pipe retires MMAs in issue order
            empty[j % S].arrive(("tile", j))
            acc_full[j % A].arrive(("tile", j))
        else:
            w = a[1]
            i = epi[w]
            go[(i + A) % S].arrive(("tile", i + A))
            epi[w] += 1
    raise AssertionError("did not finish")


@pytest.mark.parametrize("S,issuers", [(2, 1), (3, 1), (4, 1), (6, 1), (2, 2), (4, 2), (6, 2)])
def test_stage_barrier_protocol_holds(S, issuers):
    for seed in range(150):
        run(S, 2, 29, seed, issuers=issuers)


def test_shallow_stage_ring_breaks_it():
    with pytest.raises(AssertionError, match="open phase belongs to"):
        for seed in range(300):
            run(1, 2, 20, seed)


def test_odd_stage_ring_with_two_issuers_breaks_it():
    """With S odd a stage serves both issuers; one skipping the other's phases can take an
    older phase of the stage barrier for its own (the kernel asserts kNS % 2 == 0)."""
    with pytest.raises(AssertionError):
        for seed in range(300):
            run(3, 2, 29, seed, issuers=2)
