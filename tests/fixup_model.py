"""A model of the GEMM's cross-block split-tile protocol, for randomized checking.

Stream-K gives block c the steps [c*W//C, (c+1)*W//C) of the W = tiles * G
(tile, group) steps.  A tile whose G steps fall to several blocks is split.
The counter of a split tile is the one of its first contributing block (a
block is the first contributor of at most one split tile: the tile its range
ends in).  A contributor whose range starts in the tile (slot 0: the tile's
later groups, or all of a block whose range lies inside the tile) publishes
its fp32 partial to its workspace slot, then arrives on the counter with an
acquire-release atomic add, and looks at the count it got only after its
last step.  The first contributor, whose range ends in the tile (slot 1),
arrives only after its last step: if its arrival completes the count it
finishes the tile from its own registers and the others' partials; if not,
it publishes its partial to slot 1 and then adds a published flag (bit 16)
to the counter with release semantics.  The block whose arrival completed
the count reads every contributor's partial in ascending block order -- the
first contributor's slot 1 only once the flag is set -- writes the tile's
output and sets the counter back to zero for the next call.  Consecutive calls that share
the workspace are ordered by the grid dependency: a block writes partials,
counters or outputs only once the previous call has completed.

Each block of each call is an agent yielding its global-memory actions in
program order.  Stores become visible at a random later tick, or at the
latest when the same block performs a release (the arrival atomic).  A
scheduler runs one random runnable agent, or makes one random pending store
visible, per tick.

The checker reports a finisher reading a partial that is not the current
call's partial of that tile, a split tile finished zero or several times, an
output written twice, a counter left non-zero after a call, two split tiles
sharing a counter, and an agent that can never run.  A wait on the flag runs
forever in the model when nothing will set it (a deadlock is then reported
as no progress).

Only tests use this module; it restates the protocol, not the kernel code.
"""
import random

FLAG = 1 << 16     # published-partial flag of the first contributor
MASK = FLAG - 1


def ranges(W, C):
    """Block c's steps [s0, s1)."""
    return [(c * W // C, (c + 1) * W // C) for c in range(C)]


def block_of_step(s, W, C):
    """The block whose range holds step s (by search over the ranges)."""
    for c, (s0, s1) in enumerate(ranges(W, C)):
        if s0 <= s < s1:
            return c
    raise ValueError(s)


def segments(s0, s1, G):
    """(tile, first group, last group) of each run of one tile in [s0, s1)."""
    out = []
    s = s0
    while s < s1:
        t = s // G
        e = min(s1, (t + 1) * G)
        out.append((t, s - t * G, e - 1 - t * G))
        s = e
    return out


class _Sim:
    def __init__(self, seed):
        self.rng = random.Random(seed)
        self.mem = {}          # visible global memory
        self.pending = []      # (block key, address, value) not yet visible
        self.failed = None
        self.outputs = {}
        self.finishes = {}

    def fail(self, msg):
        if self.failed is None:
            self.failed = msg

    def store(self, who, addr, value):
        self.pending.append((who, addr, value))

    def flush(self, who):
        keep = []
        for w, a, v in self.pending:
            if w == who:
                self.mem[a] = v
            else:
                keep.append((w, a, v))
        self.pending = keep

    def flush_one(self):
        i = self.rng.randrange(len(self.pending))
        _, a, v = self.pending.pop(i)
        self.mem[a] = v


def _block(sim, call, c, W, G, C, opts, done):
    """Program order of block c's epilogue in call `call`."""
    s0, s1 = ranges(W, C)[c]
    segs = segments(s0, s1, G)
    first_tile = s0 // G
    me = (call, c)
    pend = []
    waited = False
    for t, g0, g1 in segs:
        # the segment's steps run here; nothing global happens before its end
        yield "step"
        if not waited and not opts.get("no_grid_wait"):
            # outputs and workspace may still be in use by the previous call
            while not all(done.get((call - 1, b), call == 0) for b in range(C)):
                yield "wait"
        waited = True
        if g0 == 0 and g1 == G - 1:
            key = (call, "y", t)
            if key in sim.outputs:
                sim.fail(f"call {call}: tile {t} written twice")
            sim.outputs[key] = c
            continue
        slot = 0 if t == first_tile else 1
        c_first = block_of_step(t * G, W, C)
        if slot == 1 and not opts.get("publish_first_everywhere"):
            pend.append((t, None, "end"))     # arrives after its last step
            yield "step"
            continue
        if opts.get("arrive_before_publish"):
            old = sim.mem.get(("cnt", c_first), 0)
            sim.mem[("cnt", c_first)] = old + 1
            yield "step"
            sim.store(me, ("part", c, slot), (call, t, g0, g1))
        else:
            sim.store(me, ("part", c, slot), (call, t, g0, g1))
            yield "step"
            if not opts.get("relaxed_arrival"):
                sim.flush(me)          # release: the partial before the count
            old = sim.mem.get(("cnt", c_first), 0)
            sim.mem[("cnt", c_first)] = old + 1
        pend.append((t, old, "start"))
        yield "step"
    # the end piece first (its partial is still in registers), then the start
    # piece
    pend.sort(key=lambda e: e[2] != "end")
    for t, old, kind in pend:
        c_first = block_of_step(t * G, W, C)
        c_last = block_of_step(t * G + G - 1, W, C)
        own = None
        if kind == "end":
            sim.flush(me)                              # acquire-release arrival
            old = sim.mem.get(("cnt", c_first), 0)
            sim.mem[("cnt", c_first)] = old + 1
            yield "step"
            s_own = segments(*ranges(W, C)[c], G)[-1]
            if (old & MASK) != c_last - c_first:
                sim.store(me, ("part", c, 1), (call, t, s_own[1], s_own[2]))
                yield "step"
                if not opts.get("flag_before_flush"):
                    sim.flush(me)                      # release: the partial before the flag
                sim.mem[("cnt", c_first)] = sim.mem.get(("cnt", c_first), 0) + FLAG
                yield "step"
                continue
            own = (call, t, s_own[1], s_own[2])
        elif (old & MASK) != c_last - c_first:
            continue
        # the last arrival: every contributor's partial, ascending blocks
        covered = []
        for cc in range(c_first, c_last + 1):
            slot = 0 if (ranges(W, C)[cc][0] // G) == t else 1
            if cc == c and own is not None:
                v = own
            else:
                if slot == 1 and not opts.get("publish_first_everywhere") \
                        and not opts.get("skip_flag_wait"):
                    # the first contributor publishes after its arrival
                    while not (sim.mem.get(("cnt", c_first), 0) & FLAG):
                        yield "wait"
                v = sim.mem.get(("part", cc, slot))
            if v is None or v[0] != call or v[1] != t:
                sim.fail(f"call {call}: block {c} finishing tile {t} read block {cc}'s "
                         f"slot {slot} = {v}")
                return
            covered.append((v[2], v[3]))
            yield "step"
        groups = sorted(covered)
        if groups[0][0] != 0 or groups[-1][1] != G - 1 or any(
                a[1] + 1 != b[0] for a, b in zip(groups, groups[1:])):
            sim.fail(f"call {call}: tile {t} partials cover groups {groups}")
        key = (call, "y", t)
        if key in sim.outputs:
            sim.fail(f"call {call}: tile {t} written twice")
        sim.outputs[key] = c
        sim.finishes[(call, t)] = sim.finishes.get((call, t), 0) + 1
        if not opts.get("no_reset"):
            sim.store(me, ("cnt", c_first), 0)
        yield "step"
    sim.flush(me)              # the call completes with every store visible


def run(W, G, C, calls, seed, **opts):
    """Randomized run of `calls` consecutive calls; None if all checks pass."""
    sim = _Sim(seed)
    done = {}
    agents = []
    for call in range(calls):
        for c in range(C):
            agents.append({"key": (call, c), "gen": _block(sim, call, c, W, G, C, opts, done)})
    split = {}
    for t in range(W // G):
        a, b = block_of_step(t * G, W, C), block_of_step(t * G + G - 1, W, C)
        if a != b:
            if a in split:
                sim.fail(f"tiles {split[a]} and {t} share block {a}'s counter")
            split[a] = t
    live = list(agents)
    for _ in range(200000):
        if sim.failed:
            return sim.failed
        if not live and not sim.pending:
            break
        if sim.pending and (not live or sim.rng.random() < 0.3):
            sim.flush_one()
            continue
        a = sim.rng.choice(live)
        try:
            next(a["gen"])
        except StopIteration:
            done[a["key"]] = True
            live.remove(a)
    else:
        return "no progress bound reached"
    if sim.failed:
        return sim.failed
    for call in range(calls):
        for t in range(W // G):
            if (call, "y", t) not in sim.outputs:
                return f"call {call}: tile {t} never written"
        for t in split.values():
            n = sim.finishes.get((call, t), 0)
            if n != 1:
                return f"call {call}: split tile {t} finished {n} times"
    left = {k: v for k, v in sim.mem.items() if k[0] == "cnt" and v != 0}
    if left:
        return f"counters left non-zero: {left}"
    return None
