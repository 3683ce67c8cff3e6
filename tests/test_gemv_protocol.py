"""Model check of the streaming GEMV's barrier protocol.

`k_gemv` (gemv_mul_mm_gb300/csrc/k_gemv.cu) streams weight chunks through a
ring of S shared-memory stages: one producer thread issues the bulk copies in
chunk order and, before reusing a stage, waits for its `empty` barrier; the
consumer warps form NW / nwu groups that take a row group's chunks
round-robin, wait for the stage's `full` barrier, decode it and arrive on
`empty` (nwu arrivals). After each row group every warp leaves its partial
sums in one of two reduction buffers and a rotating writer warp adds them up
(`red_full`, NW arrivals; `red_empty`, released by the writer). Every wait is
a parity wait, which is only right while the barrier is at the awaited phase
or the next one. The launch planner makes S a multiple of the number of
groups so that each stage belongs to one group, whose warps meet its uses in
order.

The model replays that schedule under random interleavings (every warp an
actor, copies landing in any order), asserts the phase window at every poll
and tracks the contents of every stage and reduction slot; the producer's
final drain of the last copy of each stage is included. The sabotage case
gives the ring a stage count that is not a multiple of the groups and must
fail.
"""
import random

import pytest

from .test_gemm_protocol import Barrier, Violation, Wait, simulate


class GemvModel:
    def __init__(self, ngroups, nwu, S, cpr, nitems):
        self.ngroups, self.nwu, self.S, self.cpr, self.nitems = ngroups, nwu, S, cpr, nitems
        self.NW = ngroups * nwu
        self.full = [Barrier(f"full[{i}]", 1) for i in range(S)]
        self.empty = [Barrier(f"empty[{i}]", nwu) for i in range(S)]
        self.red_full = [Barrier(f"red_full[{p}]", self.NW) for p in range(2)]
        self.red_empty = [Barrier(f"red_empty[{p}]", 1) for p in range(2)]
        self.stage = [None] * S
        self.red = [[None] * self.NW for _ in range(2)]
        self.loads = []
        self.fifo = []

    def complete(self):
        raise AssertionError("no in-order completions in this model")

    def producer(self):
        it = 0
        for _ in range(self.nitems):
            for _c in range(self.cpr):
                s, use = it % self.S, it // self.S
                if use > 0:
                    yield Wait(self.empty[s], use - 1)

                def land(it=it, s=s):
                    self.stage[s] = it
                    self.full[s].arrive()
                self.loads.append(land)
                it += 1
        # every issued copy lands before the CTA retires
        issued = it
        for s in range(min(self.S, issued)):
            yield Wait(self.full[s], (issued - 1 - s) // self.S)

    def consumer(self, warp):
        grp = warp // self.nwu
        it_base = 0
        for gi in range(self.nitems):
            c = (grp - it_base % self.ngroups + self.ngroups) % self.ngroups
            while c < self.cpr:
                it = it_base + c
                s, use = it % self.S, it // self.S
                yield Wait(self.full[s], use)
                for _ in range(2):                          # decode, then re-check before the release
                    if self.stage[s] != it:
                        raise Violation(f"warp {warp}: stage {s} holds chunk {self.stage[s]}, wanted {it}")
                    yield None
                self.empty[s].arrive()
                c += self.ngroups
            p, use = gi & 1, gi >> 1
            if use > 0:
                yield Wait(self.red_empty[p], use - 1)
            self.red[p][warp] = gi
            self.red_full[p].arrive()
            if warp == gi % self.NW:
                yield Wait(self.red_full[p], use)
                for _ in range(2):
                    if any(v != gi for v in self.red[p]):
                        raise Violation(f"writer of row group {gi}: reduction buffer {p} holds {self.red[p]}")
                    yield None
                self.red_empty[p].arrive()
            it_base += self.cpr

    def run(self, rng):
        actors = [self.producer()] + [self.consumer(w) for w in range(self.NW)]
        simulate(self, actors, rng)


# (groups, warps per group, stages): the shapes the planner produces (stages a
# multiple of the groups, at least two), over item lengths that do and do not
# divide by the groups
SHAPES = [(g, nwu, S) for g, nwu in ((1, 8), (2, 4), (2, 8), (4, 2), (8, 1))
          for S in range(max(2, g), 9) if S % g == 0]


@pytest.mark.parametrize("ngroups,nwu,S", SHAPES)
@pytest.mark.parametrize("cpr", [1, 3, 4])
def test_gemv_ring_protocol_holds(ngroups, nwu, S, cpr):
    for seed in range(15):
        GemvModel(ngroups, nwu, S, cpr, nitems=5).run(random.Random(seed))


@pytest.mark.parametrize("ngroups,S", [(2, 3), (4, 6)])
def test_gemv_ring_sabotage_is_caught(ngroups, S):
    """A stage count that is not a multiple of the groups lets two groups
    share a stage, and some interleaving breaks the protocol."""
    caught = 0
    for seed in range(100):
        try:
            GemvModel(ngroups, 2, S, cpr=3, nitems=5).run(random.Random(seed))
        except Violation:
            caught += 1
    assert caught > 0
