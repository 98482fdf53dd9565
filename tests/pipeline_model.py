"""A model of the GEMM kernel's mbarrier protocol, for randomized checking.

Each role of one block of `qlin_gemm_kernel` (the weight producer, the
activation and scale producer, the two MMA issuers, the eight converter warps
and the epilogue warps) is a generator that yields the kernel's
synchronisation actions in program order: waits on an mbarrier phase parity,
arrivals, expect-tx arrivals, TMA loads (asynchronous, completing their
transaction bytes later), MMAs (asynchronous) and `tcgen05.commit` (an
arrival once every MMA its thread issued before it has completed).  A
scheduler runs one random runnable role, or completes one random pending
asynchronous operation, per tick.

mbarriers follow the PTX rules: an arrival count per phase and a transaction
count; `try_wait.parity P` succeeds when the current phase's parity is not P.
A wait that sees a barrier two phases behind therefore passes, which is the
failure mode this model looks for.

The checker reports
- a deadlock: no role can run and nothing is in flight;
- a hazard: a buffer written while a reader or another writer of it is
  outstanding (weight stages, activation slots, A buffers in TMEM, scale
  slots, accumulators);
- an exit with a copy or an MMA still in flight.

Only tests use this module; it shares nothing with the kernel source beyond
restating its waits and arrivals.
"""
import random
from collections import defaultdict

CHUNK = 8        # scale groups per scale-ring load
SCALE_SLOTS = 4
PRE_W = 3        # weight loads issued before the block's set-up barrier


class _Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.done = name, count, count, 0, 0

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count

    def arrive(self, sim):
        self.pending -= 1
        if self.pending < 0:
            sim.fail(f"{self.name}: arrival overflow in phase {self.done}")
        self._check()

    def ready(self, parity):
        return (self.done & 1) != parity


class _Sim:
    def __init__(self, seed):
        self.rng = random.Random(seed)
        self.bars = {}
        self.agents = []
        self.inflight = []
        self.failed = None
        self.res = defaultdict(lambda: {"w": 0, "r": 0})
        self.mmas = defaultdict(list)
        self.commits = []

    def bar(self, name, count=1):
        self.bars[name] = _Bar(name, count)

    def fail(self, msg):
        if self.failed is None:
            self.failed = msg

    def _begin(self, r, kind, who):
        st = self.res[r]
        if kind == "w" and (st["w"] or st["r"]):
            self.fail(f"hazard: {who} writes {r} while it is in use")
        if kind == "r" and st["w"]:
            self.fail(f"hazard: {who} reads {r} while it is written")
        st[kind] += 1

    def _end(self, r, kind):
        self.res[r][kind] -= 1

    def _flush_commits(self):
        keep = []
        for prior, name in self.commits:
            if all(m["done"] for m in prior):
                self.bars[name].arrive(self)
            else:
                keep.append((prior, name))
        self.commits = keep

    def run(self, max_ticks=500000):
        for _ in range(max_ticks):
            if self.failed:
                return self.failed
            runnable = [a for a in self.agents if not a["done"] and
                        (a["wait"] is None or self.bars[a["wait"][0]].ready(a["wait"][1]))]
            choices = [("a", a) for a in runnable] + [("o", o) for o in self.inflight]
            if not choices:
                live = [(a["name"], a["wait"]) for a in self.agents if not a["done"]]
                return f"deadlock: {live[:4]}" if live else None
            if all(a["done"] for a in self.agents) and (self.inflight or self.commits):
                # the block would exit (and free its TMEM) with copies or
                # MMAs still in flight
                return f"exit with {len(self.inflight)} operations in flight"
            kind, x = self.rng.choice(choices)
            if kind == "o":
                self.inflight.remove(x)
                x()
                self._flush_commits()
            else:
                self._step(x)
        return "no progress bound reached"

    def _step(self, a):
        a["wait"] = None
        try:
            act = next(a["gen"])
        except StopIteration:
            a["done"] = True
            return
        op = act[0]
        if op == "wait":
            a["wait"] = (act[1], act[2])
        elif op == "arrive":
            self.bars[act[1]].arrive(self)
        elif op == "expect":
            b = self.bars[act[1]]
            b.tx += 1
            b.arrive(self)
        elif op == "tma":
            _, name, res = act
            self._begin(res, "w", a["name"])

            def land(name=name, res=res):
                self._end(res, "w")
                b = self.bars[name]
                b.tx -= 1
                b._check()
            self.inflight.append(land)
        elif op == "mma":
            _, issuer, reads = act
            for r in reads:
                self._begin(r, "r", a["name"])
            rec = {"done": False}

            def finish(rec=rec, reads=reads):
                for r in reads:
                    self._end(r, "r")
                rec["done"] = True
            self.mmas[issuer].append(rec)
            self.inflight.append(finish)
        elif op == "commit":
            _, issuer, name = act
            self.commits.append(([m for m in self.mmas[issuer] if not m["done"]], name))
            self._flush_commits()
        elif op == "read":
            self._begin(act[1], "r", a["name"])
            self._end(act[1], "r")
        elif op == "write":
            self._begin(act[1], "w", a["name"])
            self._end(act[1], "w")


def steps(s0, s1, G):
    """The (tile, group) steps s0 .. s1-1 of one block, tiles of G steps."""
    out = []
    n = s1 - s0
    for j, s in enumerate(range(s0, s1)):
        g = s % G
        out.append({"g": g, "first": j == 0 or g == 0, "last": j == n - 1 or g == G - 1})
    return out


class _Chunk:
    """Scale chunks: CHUNK steps of a segment share one scale-ring load."""

    def __init__(self):
        self.cg, self.ci = 0, -1

    def begin(self, seg_first):
        if seg_first:
            self.cg = 0
        starts = self.cg % CHUNK == 0
        if starts:
            self.ci += 1
        return starts

    def row(self):
        return self.cg % CHUNK

    def ends(self, seg_last):
        return seg_last or self.cg % CHUNK == CHUNK - 1

    def advance(self):
        self.cg += 1


def _roles(c, st):
    """The block's roles for configuration c over the step list st.

    c["mode"]: "wo" (W4A16 / W8A16: scales read by the converters, the whole
    segment accumulated per issuer), "w8" (W8A8 with 16-bit token tiles), or
    "w8x" (W8A8 with int8 token tiles expanded by the converters).  NB: A
    buffers; ND: accumulators (segment buffers for "wo"); stages: weight
    ring; NX: token operand slots; NXR: the ring the activation producer
    fills (int8 staging for "w8x")."""
    WO, XC = c["mode"] == "wo", c["mode"] == "w8x"
    NB, ND, ST, NX = c["NB"], c["ND"], c["stages"], c["NX"]
    NXR = c.get("NXR", NX)
    # A buffers freed by commits of their own (weight-only formats, and W8A8
    # with fewer D buffers than A buffers); else by the step's D commit
    ACOMMIT = WO or ND < NB
    n = len(st)
    pre = min(n, PRE_W, ST)

    def weight_producer():
        for j in range(pre):
            yield ("expect", f"wfull{j}")
            yield ("tma", f"wfull{j}", f"W{j}")
        for j in range(pre, n):
            if WO and j == pre:
                yield ("wait", "x_go", 0)
            yield ("wait", f"empty{j % ST}", ((j // ST) & 1) ^ 1)
            yield ("expect", f"wfull{j % ST}")
            yield ("tma", f"wfull{j % ST}", f"W{j % ST}")
        for j in range(max(0, n - ST), n):
            yield ("wait", f"wfull{j % ST}", (j // ST) & 1)

    def activation_producer():
        ch, issued, go, loads = _Chunk(), 0, False, 0
        first = min(n, NXR)
        for j in range(n):
            if ch.begin(j == 0 or st[j]["g"] == 0):
                slot, ph = ch.ci % SCALE_SLOTS, (ch.ci // SCALE_SLOTS) & 1
                if not go and ch.ci >= SCALE_SLOTS and not c.get("no_early_x_go"):
                    yield ("arrive", "x_go")
                    go = True
                yield ("wait", f"sempty{slot}", ph ^ 1)
                yield ("expect", f"sfull{slot}")
                yield ("tma", f"sfull{slot}", f"S{slot}")
                loads += 1
            yield ("wait", f"xempty{j % NXR}", ((j // NXR) & 1) ^ 1)
            yield ("expect", f"xfull{j % NXR}")
            yield ("tma", f"xfull{j % NXR}", f"XI{j % NXR}" if XC else f"X{j % NXR}")
            issued += 1
            if not go and issued == first:
                yield ("arrive", "x_go")
                go = True
            ch.advance()
        if not go:
            yield ("arrive", "x_go")
        for j in range(max(0, issued - NXR), issued):
            yield ("wait", f"xfull{j % NXR}", (j // NXR) & 1)
        for k in range(max(0, loads - SCALE_SLOTS), loads):
            yield ("wait", f"sfull{k % SCALE_SLOTS}", (k // SCALE_SLOTS) & 1)

    def issuer(me):
        seg, started = 0, False
        for j in range(n):
            ab, abph = j % NB, (j // NB) & 1
            if st[j]["first"]:
                started = False
            didx = seg if WO else j
            db, dbph = didx % ND, (didx // ND) & 1
            if (j & 1) == me:
                if not XC:
                    yield ("wait", f"xfull{j % NX}", (j // NX) & 1)
                yield ("wait", f"afull{ab}", abph)
                if not (WO and started):
                    yield ("wait", f"dempty{db}", dbph ^ 1)
                yield ("mma", me, [f"A{ab}", f"X{j % NX}"])
                if ACOMMIT:
                    yield ("commit", me, f"aempty{ab}")
                if not XC:
                    yield ("commit", me, f"xempty{j % NX}")
                if not WO:
                    yield ("commit", me, f"dfull{db}")
                started = True
            if WO and st[j]["last"]:
                if started:
                    yield ("commit", me, f"dfull{db}")
                else:
                    yield ("wait", f"dempty{db}", dbph ^ 1)
                    yield ("arrive", f"dfull{db}")
                seg += 1
        yield ("commit", me, "mma_done")
        yield ("wait", "mma_done", 0)

    def converter(grp):
        ch, ready = _Chunk(), False
        for j in range(n):
            if WO and ch.begin(j == 0 or st[j]["g"] == 0):
                ready = False
            if (j & 1) == grp:
                ab, abph = j % NB, (j // NB) & 1
                yield ("wait", f"wfull{j % ST}", (j // ST) & 1)
                # the weights go to registers first and the slot is released
                # before the A buffer is waited for
                yield ("read", f"W{j % ST}")
                yield ("arrive", f"empty{j % ST}")
                if ACOMMIT:
                    yield ("wait", f"aempty{ab}", abph ^ 1)
                elif j >= NB:
                    yield ("wait", f"dfull{(j - NB) % ND}", ((j - NB) // ND) & 1)
                if XC:
                    yield ("wait", f"xfull{j % NXR}", (j // NXR) & 1)
                if WO:
                    slot = ch.ci % SCALE_SLOTS
                    if not ready:
                        yield ("wait", f"sfull{slot}", (ch.ci // SCALE_SLOTS) & 1)
                    ready = True
                    yield ("read", f"S{slot}")
                if XC:
                    yield ("read", f"XI{j % NXR}")
                    yield ("write", f"X{ab}")
                yield ("write", f"A{ab}")
                if XC:
                    yield ("arrive", f"xempty{j % NXR}")
                yield ("arrive", f"afull{ab}")
            if WO and ch.ends(st[j]["last"]):
                slot = ch.ci % SCALE_SLOTS
                if not c.get("release_without_landing") and not ready:
                    yield ("wait", f"sfull{slot}", (ch.ci // SCALE_SLOTS) & 1)
                yield ("arrive", f"sempty{slot}")
            ch.advance()

    def epilogue(w):
        ch, seg = _Chunk(), 0
        for j in range(n):
            if not WO or st[j]["last"]:
                idx = seg if WO else j
                b, bph = idx % ND, (idx // ND) & 1
                if not WO:
                    ch.begin(st[j]["first"])
                    slot = ch.ci % SCALE_SLOTS
                    if ch.row() == 0:
                        yield ("wait", f"sfull{slot}", (ch.ci // SCALE_SLOTS) & 1)
                    yield ("read", f"S{slot}")
                    if ch.ends(st[j]["last"]):
                        yield ("arrive", f"sempty{slot}")
                yield ("wait", f"dfull{b}", bph)
                yield ("read", f"D{b}")
                yield ("arrive", f"dempty{b}")
            if WO and st[j]["last"]:
                seg += 1
            if not WO:
                ch.advance()
        if w == 0:   # the split-tile fix-up stages partials over both rings
            for i in range(ST):
                yield ("write", f"W{i}")
            for i in range(NX):
                yield ("write", f"X{i}")

    roles = [("weight producer", weight_producer()), ("activation producer", activation_producer()),
             ("issuer 0", issuer(0)), ("issuer 1", issuer(1))]
    for grp in range(2):
        for w in range(4):
            roles.append((f"converter {grp}.{w}", converter(grp)))
    for w in range(c.get("EPI", 8)):
        roles.append((f"epilogue {w}", epilogue(w)))
    return roles


def run(c, s0, s1, G, seed):
    """One randomized run of one block; None if it finished cleanly."""
    sim = _Sim(seed)
    WO, XC = c["mode"] == "wo", c["mode"] == "w8x"
    NXR = c.get("NXR", c["NX"])
    for i in range(c["stages"]):
        sim.bar(f"wfull{i}")
        sim.bar(f"empty{i}", 4)
    for i in range(NXR):
        sim.bar(f"xfull{i}")
        sim.bar(f"xempty{i}", 4 if XC else 1)
    for i in range(c["NB"]):
        sim.bar(f"afull{i}", 4)
        sim.bar(f"aempty{i}")
    for i in range(c["ND"]):
        sim.bar(f"dfull{i}", 2 if WO else 1)
        sim.bar(f"dempty{i}", c.get("EPI", 8))
    for i in range(SCALE_SLOTS):
        sim.bar(f"sfull{i}")
        # released by the eight converter warps (weight-only) or every
        # epilogue warp (W8A8)
        sim.bar(f"sempty{i}", 8 if WO else c.get("EPI", 8))
    sim.bar("mma_done", 2)
    sim.bar("x_go")
    for name, gen in _roles(c, steps(s0, s1, G)):
        sim.agents.append({"name": name, "gen": gen, "wait": None, "done": False})
    return sim.run()
