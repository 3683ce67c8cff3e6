"""Model check of the tensor-core GEMMs' barrier protocols.

`k_gemm_sb` and `k_gemm_tc` (gemv_mul_mm_gb300/csrc/k_gemm_tc.cu) run their roles as separate
warps that hand stages to one another through mbarriers, and every wait is a
PARITY wait: it passes when the barrier's current phase has the other parity
than the phase it waits for. Such a wait is only right while the barrier is at
the awaited phase T or the next one (T + 1); at T - 1 it would pass before
phase T completes, at T + 2 it would wait for the wrong phase.

This test replays the kernel's schedule of waits, arrivals, commits and
asynchronous copy completions as a discrete-event model under random
interleavings (every warp an actor, copies landing in any order, MMA groups
completing in issue order at random times), for every pipeline shape the
kernel instantiates: two or four stages, two to four raw-weight stages, one or
two decoder sets, with and without the min term. At every poll it asserts that
the barrier is at T or T + 1, and it tracks the contents of every buffer so
that a stage read after it was overwritten, or overwritten while an MMA still
reads it, fails. The sabotage cases replay the protocol with one completion
barrier per stage and no raw-stage release wait, and must fail: that is the
race two decoder sets would have with two stages or three raw stages. The
per-32 kernel's model is checked the same way, with a sabotage case that
drops the accumulator wait of a sub-step's second block.
"""
import random

import pytest

NDEC_WARPS = 4      # warps per decoder set (one per TMEM lane quadrant)
NEPI_WARPS = 8      # epilogue warps
SCD = 4             # scale buffers
NDONE = 4           # completion barriers, done[h % 4]


class Violation(AssertionError):
    pass


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phase = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending < 0:
            raise Violation(f"{self.name}: more arrivals than its count")
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count


class Wait:
    """A parity wait for the completion of phase `target` of `bar`."""

    def __init__(self, bar, target):
        self.bar, self.target = bar, target

    def poll(self):
        c = self.bar.phase
        if not (self.target <= c <= self.target + 1):
            raise Violation(f"{self.bar.name}: waiting for phase {self.target} while at {c}")
        return c == self.target + 1


def simulate(model, actors, rng):
    """Runs `actors` (generators that yield a Wait, or None to let others
    run) against the model's asynchronous work: `model.loads` (callables,
    landing in any order) and `model.fifo` (completed in order by
    `model.complete()`). Each actor and each kind of completion gets its own
    speed, so that one role can run far ahead of another."""
    speed = [rng.uniform(0.02, 1.0) for _ in range(len(actors) + 2)]
    blocked = [None] * len(actors)
    live = list(range(len(actors)))
    idle = 0
    while live or model.loads or model.fifo:
        cand = [("a", k) for k in live] + [("l", None)] * bool(model.loads) + [("m", None)] * bool(model.fifo)
        w = [speed[k] if t == "a" else speed[-1 if t == "l" else -2] for t, k in cand]
        t, k = rng.choices(cand, weights=w)[0]
        if t == "l":
            model.loads.pop(rng.randrange(len(model.loads)))()
            idle = 0
            continue
        if t == "m":
            model.complete()
            idle = 0
            continue
        if blocked[k] is not None:
            if not blocked[k].poll():
                idle += 1
                if idle > 200000:
                    raise Violation("no progress: the protocol deadlocks")
                continue
            blocked[k] = None
        idle = 0
        try:
            req = next(actors[k])
        except StopIteration:
            live.remove(k)
            continue
        if isinstance(req, Wait):
            blocked[k] = req


class Model:
    def __init__(self, nsup, NS, RS, sets, mins, per_stage_done=False, raw_prewait=True):
        self.nsup, self.NS, self.RS, self.sets, self.mins = nsup, NS, RS, sets, mins
        self.per_stage_done = per_stage_done
        self.raw_prewait = raw_prewait
        nd = NS if per_stage_done else NDONE
        B = Barrier
        self.raw_full = [B(f"raw_full[{i}]", 1) for i in range(RS)]
        self.raw_empty = [B(f"raw_empty[{i}]", NDEC_WARPS) for i in range(RS)]
        self.a_full = [B(f"a_full[{i}]", NDEC_WARPS) for i in range(NS)]
        self.x_full = [B(f"x_full[{i}]", 1) for i in range(NS)]
        self.done = [B(f"done[{i}]", 1) for i in range(nd)]
        self.d_empty = [B(f"d_empty[{i}]", NEPI_WARPS) for i in range(2)]
        self.sc_full = [B(f"sc_full[{i}]", NDEC_WARPS) for i in range(SCD)]
        self.sc_empty = [B(f"sc_empty[{i}]", NEPI_WARPS) for i in range(SCD)]
        # buffer contents
        self.raw = [None] * RS
        self.A = [[None] * NDEC_WARPS for _ in range(NS)]
        self.X = [None] * NS
        self.amin = [None] * NDEC_WARPS
        self.bmin = None
        self.sc = [[None] * NDEC_WARPS for _ in range(SCD)]
        self.D1 = [None, None]
        self.D2 = None
        self.handoff = None          # half-step handed from the waiter to the issuer
        self.fifo = []               # issued MMA groups, completing in order
        self.loads = []              # copies in flight, landing in any order

    # which completion barrier and phase signal "half-step h has completed"
    def done_of(self, h):
        if self.per_stage_done:
            return self.done[h % self.NS], h // self.NS
        return self.done[h % NDONE], h // NDONE

    # ---------------------------------------------------------------- actors
    def producer_raw(self):
        for s in range(self.nsup):
            rs = s % self.RS
            if s >= self.RS:
                yield Wait(self.raw_empty[rs], s // self.RS - 1)

            def land(s=s, rs=rs):
                self.raw[rs] = s
                self.raw_full[rs].arrive()
            self.loads.append(land)

    def producer_x(self):
        for h in range(2 * self.nsup):
            i, half, s = h % self.NS, h & 1, h >> 1
            if h >= self.NS:
                yield Wait(*self.done_of(h - self.NS))

            def land(h=h, i=i, half=half, s=s):
                self.X[i] = h
                if self.mins and half:
                    self.bmin = s
                self.x_full[i].arrive()
            self.loads.append(land)

    def decoder(self, dset, q):
        step = self.sets
        for s in range(dset, self.nsup, step):
            rs = s % self.RS
            if self.raw_prewait and self.RS % step != 0 and s >= self.RS:
                yield Wait(self.raw_empty[rs], s // self.RS - 1)
            yield Wait(self.raw_full[rs], s // self.RS)
            if self.raw[rs] != s:
                raise Violation(f"decoder read raw stage {rs} holding {self.raw[rs]} for super-step {s}")
            if s >= SCD:
                yield Wait(self.sc_empty[s % SCD], s // SCD - 1)
            self.sc[s % SCD][q] = s
            self.sc_full[s % SCD].arrive()
            for half in range(2):
                h = 2 * s + half
                i = h % self.NS
                yield None                                   # the decode itself
                if h >= self.NS:
                    yield Wait(*self.done_of(h - self.NS))
                if self.mins and half:
                    self.amin[q] = s
                self.A[i][q] = h
                self.a_full[i].arrive()
            if self.raw[rs] != s:
                raise Violation(f"raw stage {rs} overwritten while super-step {s} was decoded")
            self.raw_empty[rs].arrive()

    def waiter(self):
        for h in range(2 * self.nsup):
            i, half, s = h % self.NS, h & 1, h >> 1
            yield Wait(self.a_full[i], h // self.NS)
            yield Wait(self.x_full[i], h // self.NS)
            if self.mins:
                if half and s >= 1:
                    yield Wait(self.d_empty[(s - 1) & 1], (s - 1) >> 1)
            else:
                if not half and s >= 2:
                    yield Wait(self.d_empty[s & 1], (s - 2) >> 1)
            self.handoff = h
            while self.handoff is not None:                 # rendezvous with the issuer
                yield None

    def issuer(self):
        for h in range(2 * self.nsup):
            while self.handoff != h:
                yield None
            self.handoff = None
            self.check_operands(h)
            self.fifo.append(h)

    def check_operands(self, h):
        i, half, s = h % self.NS, h & 1, h >> 1
        if any(a != h for a in self.A[i]):
            raise Violation(f"MMA {h}: A stage {i} holds {self.A[i]}")
        if self.X[i] != h:
            raise Violation(f"MMA {h}: activation stage {i} holds {self.X[i]}")
        if self.mins and half:
            if any(m != s for m in self.amin) or self.bmin != s:
                raise Violation(f"MMA {h}: min tiles hold {self.amin} / {self.bmin}")

    def complete(self):
        h = self.fifo.pop(0)
        self.check_operands(h)                              # nothing overwritten in flight
        half, s = h & 1, h >> 1
        b = s & 1
        if half == 0:
            self.D1[b] = (s, 1)
        else:
            if self.D1[b] != (s, 1):
                raise Violation(f"MMA {h}: accumulator {b} holds {self.D1[b]}")
            self.D1[b] = (s, 2)
            if self.mins:
                self.D2 = s
        self.done_of(h)[0].arrive()

    def epilogue(self, e):
        for s in range(self.nsup):
            yield Wait(self.sc_full[s % SCD], s // SCD)
            yield Wait(*self.done_of(2 * s + 1))
            for _ in range(2):                              # reads, then re-checks before the hand-back
                if any(v != s for v in self.sc[s % SCD]):
                    raise Violation(f"epilogue {e}: scales of {s} read as {self.sc[s % SCD]}")
                if self.D1[s & 1] != (s, 2):
                    raise Violation(f"epilogue {e}: accumulator of {s} holds {self.D1[s & 1]}")
                if self.mins and self.D2 != s:
                    raise Violation(f"epilogue {e}: min term of {s} holds {self.D2}")
                yield None
            self.d_empty[s & 1].arrive()
            self.sc_empty[s % SCD].arrive()

    def run(self, rng):
        actors = [self.producer_raw(), self.producer_x(), self.waiter(), self.issuer()]
        actors += [self.decoder(d, q) for d in range(self.sets) for q in range(NDEC_WARPS)]
        actors += [self.epilogue(e) for e in range(NEPI_WARPS)]
        simulate(self, actors, rng)


# (stages, raw stages, decoder sets, min term): every combination the kernel
# instantiates (two stages exactly for the formats with the min term)
SHAPES = [(NS, RS, sets, NS == 2) for NS in (2, 4) for RS in (2, 3, 4) for sets in (1, 2)]


@pytest.mark.parametrize("NS,RS,sets,mins", SHAPES)
def test_sb_protocol_holds(NS, RS, sets, mins):
    for seed in range(60):
        Model(nsup=10, NS=NS, RS=RS, sets=sets, mins=mins).run(random.Random(seed))


@pytest.mark.parametrize("NS,RS", [(2, 4), (4, 3)])
def test_sb_protocol_sabotage_is_caught(NS, RS):
    """Two decoder sets with one completion barrier per stage (two stages) or
    without the raw-stage release wait (three raw stages): some interleaving
    must break the protocol."""
    caught = 0
    for seed in range(300):
        m = Model(nsup=10, NS=NS, RS=RS, sets=2, mins=NS == 2, per_stage_done=NS == 2, raw_prewait=False)
        try:
            m.run(random.Random(seed))
        except Violation:
            caught += 1
    assert caught > 0


# ---------------------------------------------------------------------------
# The per-32 kernel (`k_gemm_tc`: Q8_0, Q4_0, Q5_0, IQ4_NL, Q4_1, Q5_1, Q8_1).
# One decoder set; the unit is a sub-step (64 elements, two 32-element blocks,
# each with its own accumulator), handed from the waiter to the issuer; A
# stages (AS) are released per sub-step, activation stages (XS) per two
# sub-steps, accumulators (ND) per block by the epilogue; the formats with the
# per-block min (ND = 2) add a min MMA at the super-step's last sub-step, with
# double-buffered min tiles.
# ---------------------------------------------------------------------------
SUBS = 4            # sub-steps per super-step
AS32 = 4            # A stages


class Model32:
    def __init__(self, nsup, RS, XS, ND, mins, skip_second_wait=False):
        self.nsup, self.RS, self.XS, self.ND, self.mins = nsup, RS, XS, ND, mins
        self.skip_second_wait = skip_second_wait
        B = Barrier
        self.raw_full = [B(f"raw_full[{i}]", 1) for i in range(RS)]
        self.raw_empty = [B(f"raw_empty[{i}]", NDEC_WARPS) for i in range(RS)]
        self.a_full = [B(f"a_full[{i}]", NDEC_WARPS) for i in range(AS32)]
        self.a_empty = [B(f"a_empty[{i}]", 1) for i in range(AS32)]
        self.x_full = [B(f"x_full[{i}]", 1) for i in range(XS)]
        self.x_empty = [B(f"x_empty[{i}]", 1) for i in range(XS)]
        self.amin_full = [B(f"amin_full[{i}]", NDEC_WARPS) for i in range(2)]
        self.amin_empty = [B(f"amin_empty[{i}]", 1) for i in range(2)]
        self.bmin_full = [B(f"bmin_full[{i}]", 1) for i in range(2)]
        self.bmin_empty = [B(f"bmin_empty[{i}]", 1) for i in range(2)]
        self.d_full = [B(f"d_full[{i}]", 1) for i in range(ND)]
        self.d_empty = [B(f"d_empty[{i}]", NEPI_WARPS) for i in range(ND)]
        self.sc_full = [B(f"sc_full[{i}]", NDEC_WARPS) for i in range(2)]
        self.sc_empty = [B(f"sc_empty[{i}]", NEPI_WARPS) for i in range(2)]
        self.raw = [None] * RS
        self.A = [[None] * NDEC_WARPS for _ in range(AS32)]
        self.X = [None] * XS
        self.amin = [[None] * NDEC_WARPS for _ in range(2)]
        self.bmin = [None, None]
        self.sc = [[None] * NDEC_WARPS for _ in range(2)]
        self.D = [None] * ND
        self.D2 = None
        self.handoff = None
        self.fifo = []       # issued MMAs and commits, completing in order
        self.loads = []

    def producer_raw(self):
        for s in range(self.nsup):
            rs = s % self.RS
            if s >= self.RS:
                yield Wait(self.raw_empty[rs], s // self.RS - 1)

            def land(s=s, rs=rs):
                self.raw[rs] = s
                self.raw_full[rs].arrive()
            self.loads.append(land)
            if self.mins:
                b = s & 1
                if s >= 2:
                    yield Wait(self.bmin_empty[b], s // 2 - 1)

                def land_min(s=s, b=b):
                    self.bmin[b] = s
                    self.bmin_full[b].arrive()
                self.loads.append(land_min)

    def producer_x(self):
        for sx in range(self.nsup * SUBS // 2):
            xs = sx % self.XS
            if sx >= self.XS:
                yield Wait(self.x_empty[xs], sx // self.XS - 1)

            def land(sx=sx, xs=xs):
                self.X[xs] = sx
                self.x_full[xs].arrive()
            self.loads.append(land)

    def decoder(self, q):
        for s in range(self.nsup):
            rs = s % self.RS
            yield Wait(self.raw_full[rs], s // self.RS)
            if self.raw[rs] != s:
                raise Violation(f"decoder read raw stage {rs} holding {self.raw[rs]} for super-step {s}")
            if s >= 2:
                yield Wait(self.sc_empty[s & 1], s // 2 - 1)
            self.sc[s & 1][q] = s
            self.sc_full[s & 1].arrive()
            if self.mins:
                b = s & 1
                if s >= 2:
                    yield Wait(self.amin_empty[b], s // 2 - 1)
                self.amin[b][q] = s
                self.amin_full[b].arrive()
            for qq in range(SUBS):
                sub = SUBS * s + qq
                a = sub % AS32
                yield None                                   # the decode
                if sub >= AS32:
                    yield Wait(self.a_empty[a], sub // AS32 - 1)
                self.A[a][q] = sub
                self.a_full[a].arrive()
            if self.raw[rs] != s:
                raise Violation(f"raw stage {rs} overwritten while super-step {s} was decoded")
            self.raw_empty[rs].arrive()

    def waiter(self):
        for s in range(self.nsup):
            for qq in range(SUBS):
                sub = SUBS * s + qq
                a, xi = sub % AS32, sub >> 1
                yield Wait(self.a_full[a], sub // AS32)
                if sub % 2 == 0:
                    yield Wait(self.x_full[xi % self.XS], xi // self.XS)
                for h in range(1 if self.skip_second_wait else 2):
                    u = 8 * s + 2 * qq + h
                    if u >= self.ND:
                        yield Wait(self.d_empty[u % self.ND], u // self.ND - 1)
                if self.mins and qq == SUBS - 1:
                    yield Wait(self.amin_full[s & 1], s // 2)
                    yield Wait(self.bmin_full[s & 1], s // 2)
                self.handoff = sub
                while self.handoff is not None:
                    yield None

    def issuer(self):
        for s in range(self.nsup):
            for qq in range(SUBS):
                sub = SUBS * s + qq
                while self.handoff != sub:
                    yield None
                self.handoff = None
                a, xi = sub % AS32, sub >> 1
                for h in range(2):
                    u = 8 * s + 2 * qq + h
                    self.fifo.append(("mma", u, a, sub, xi % self.XS, xi))
                    if h == 1 and self.mins and qq == SUBS - 1:
                        self.fifo.append(("min", s))
                        self.fifo.append(("commit", self.amin_empty[s & 1]))
                        self.fifo.append(("commit", self.bmin_empty[s & 1]))
                    self.fifo.append(("commit", self.d_full[u % self.ND]))
                self.fifo.append(("commit", self.a_empty[a]))
                if sub % 2 == 1:
                    self.fifo.append(("commit", self.x_empty[xi % self.XS]))

    def complete(self):
        ev = self.fifo.pop(0)
        if ev[0] == "commit":
            ev[1].arrive()
        elif ev[0] == "mma":
            _, u, a, sub, xs, xi = ev
            if any(v != sub for v in self.A[a]):
                raise Violation(f"MMA of block {u}: A stage {a} holds {self.A[a]}")
            if self.X[xs] != xi:
                raise Violation(f"MMA of block {u}: activation stage {xs} holds {self.X[xs]}")
            self.D[u % self.ND] = u
        else:
            s = ev[1]
            if any(v != s for v in self.amin[s & 1]) or self.bmin[s & 1] != s:
                raise Violation(f"min MMA of {s}: tiles hold {self.amin[s & 1]} / {self.bmin[s & 1]}")
            self.D2 = s

    def epilogue(self, e):
        for s in range(self.nsup):
            yield Wait(self.sc_full[s & 1], s // 2)
            for j in range(8):
                u = 8 * s + j
                b = u % self.ND
                yield Wait(self.d_full[b], u // self.ND)
                for _ in range(2):
                    if self.D[b] != u:
                        raise Violation(f"epilogue {e}: accumulator {b} holds {self.D[b]} for block {u}")
                    if any(v != s for v in self.sc[s & 1]):
                        raise Violation(f"epilogue {e}: scales of {s} read as {self.sc[s & 1]}")
                    if self.mins and j == 7 and self.D2 != s:
                        raise Violation(f"epilogue {e}: min term of {s} holds {self.D2}")
                    yield None
                self.d_empty[b].arrive()
            self.sc_empty[s & 1].arrive()

    def run(self, rng):
        actors = [self.producer_raw(), self.producer_x(), self.waiter(), self.issuer()]
        actors += [self.decoder(q) for q in range(NDEC_WARPS)]
        actors += [self.epilogue(e) for e in range(NEPI_WARPS)]
        simulate(self, actors, rng)


# (raw stages, activation stages, accumulators, min term): the stage counts the
# per-32 formats get (three or four of each; two accumulators with the min term)
SHAPES32 = [(RS, XS, 2 if mins else 3, mins) for RS in (3, 4) for XS in (3, 4) for mins in (False, True)]


@pytest.mark.parametrize("RS,XS,ND,mins", SHAPES32)
def test_per32_protocol_holds(RS, XS, ND, mins):
    for seed in range(40):
        Model32(nsup=6, RS=RS, XS=XS, ND=ND, mins=mins).run(random.Random(seed))


@pytest.mark.parametrize("ND,mins", [(3, False), (2, True)])
def test_per32_protocol_sabotage_is_caught(ND, mins):
    """Without the wait for the second block's accumulator, some interleaving
    overwrites an accumulator the epilogue has not read yet."""
    caught = 0
    for seed in range(100):
        try:
            Model32(nsup=6, RS=4, XS=3, ND=ND, mins=mins, skip_second_wait=True).run(random.Random(seed))
        except Violation:
            caught += 1
    assert caught > 0
