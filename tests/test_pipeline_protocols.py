"""The prefill kernels' barrier protocols, model-checked on the CPU.

Each role of the scan kernel and of the output kernel is written here as a
sequence of the waits, arrivals and asynchronous operations it issues, with
the same barrier counts, parities and buffer indices as the CUDA source
(csrc/gdn_prefill_scan.cu, csrc/gdn_prefill_out.cu; the scan CTA runs its
chains in turn, counting steps over all of them).  A random scheduler
interleaves the roles and completes the asynchronous operations (tensor-map
and bulk copies in any order, each thread's tcgen05 commits in issue order)
at random times, for many seeds and sizes.  It checks that:
  * an mbarrier parity wait passes only once the phase it stands for has
    completed (the hardware test is "current phase parity differs", so a
    waiter one phase ahead, or two phases behind, would be caught);
  * a named-barrier arrival always lands in the generation it is meant for;
  * no run deadlocks;
  * no buffer (copy stage, z / output slot, TMEM accumulator, S operand) is
    written while a reader that still needs it is using it, and every
    reader sees the unit it expects.
These are the properties the kernels' pipelines rely on; the memory-model
side (proxy fences, visibility) is not modelled.
"""
import random

import pytest


class Violation(AssertionError):
    pass


class MBar:
    """mbarrier: `count` arrivals complete a phase; parity test as in PTX."""

    def __init__(self, name, count):
        self.name, self.count, self.arrived, self.done = name, count, 0, 0

    def arrive(self):
        self.arrived += 1
        if self.arrived == self.count:
            self.arrived = 0
            self.done += 1

    def passes(self, parity):
        return (self.done & 1) != parity


class NamedBar:
    """bar.arrive / bar.sync on one hardware barrier: a generation completes
    when `count` warps have arrived; arrivals carry the generation their
    thread means, which must be the one the hardware is counting."""

    def __init__(self, count):
        self.count, self.arrived, self.gen = count, 0, 0

    def arrive(self, gen):
        if gen != self.gen:
            raise Violation(f"named-barrier arrival for generation {gen} while {self.gen} is counting")
        self.arrived += 1
        if self.arrived == self.count:
            self.arrived = 0
            self.gen += 1


class Buffers:
    """Readers and writers of each buffer, with the unit each holds."""

    def __init__(self):
        self.writers, self.readers, self.content = {}, {}, {}

    def begin_write(self, buf, unit, who):
        if self.readers.get(buf):
            raise Violation(f"{who} writes {buf} (unit {unit}) under readers {self.readers[buf]}")
        if buf in self.writers:
            raise Violation(f"{who} writes {buf} while {self.writers[buf]} writes it")
        self.writers[buf] = (who, unit)

    def end_write(self, buf, unit):
        del self.writers[buf]
        self.content[buf] = unit

    def begin_read(self, buf, unit, who):
        if buf in self.writers:
            raise Violation(f"{who} reads {buf} (unit {unit}) while {self.writers[buf]} writes it")
        if self.content.get(buf) != unit:
            raise Violation(f"{who} reads {buf} expecting unit {unit}, holds {self.content.get(buf)}")
        self.readers.setdefault(buf, set()).add((who, unit))

    def end_read(self, buf, unit, who):
        self.readers[buf].discard((who, unit))


class Sim:
    """Random interleaving of roles (generators of actions) and async ops."""

    def __init__(self, rng):
        self.rng, self.roles, self.asyncs, self.buf = rng, {}, [], Buffers()
        self.stores = {}   # bulk groups still reading shared memory, per thread
        # how often a completion may be taken while a role can still move:
        # from copies that land at once to copies that lag far behind
        self.async_rate = rng.choice([0.02, 0.1, 0.5, 1.0])

    def add(self, name, gen):
        self.roles[name] = [gen, None]   # generator, pending action

    def launch(self, who, ops, ordered=False):
        """An asynchronous operation: `ops` run when it completes.  Ordered
        ones (a thread's tcgen05 commits) complete in issue order."""
        self.asyncs.append((who, ordered, ops))

    def run(self, max_steps=400000):
        # some roles run far behind the others (a warp that is rarely
        # scheduled), so that waits covering long lags are exercised too
        slow = {name for name in self.roles if self.rng.random() < 0.15}
        for _ in range(max_steps):
            choices = []
            for name, st in self.roles.items():
                if st[1] is None:
                    try:
                        st[1] = next(st[0])
                    except StopIteration:
                        st[1] = ("done",)
                act = st[1]
                if act[0] == "done":
                    continue
                if act[0] == "wait" and not act[1].passes(act[2]):
                    continue
                if act[0] == "sync" and act[1].gen <= act[2]:
                    continue
                if act[0] == "stores_read" and self.stores.get(act[1]):
                    continue
                choices.append(("role", name))
            if not choices or self.rng.random() < self.async_rate:
                first_ordered = set()
                for idx, (who, ordered, _) in enumerate(self.asyncs):
                    if ordered:
                        if who in first_ordered:
                            continue
                        first_ordered.add(who)
                    choices.append(("async", idx))
            if not choices:
                if all(st[1] == ("done",) for st in self.roles.values()):
                    return
                raise Violation("deadlock: " + ", ".join(f"{n}: {st[1][:1]}" for n, st in self.roles.items()
                                                          if st[1] != ("done",)))
            weights = [0.03 if (k == "role" and n in slow) else 1.0 for k, n in choices]
            kind, key = self.rng.choices(choices, weights)[0]
            if kind == "async":
                _, _, ops = self.asyncs.pop(key)
                for op in ops:
                    op()
                continue
            st = self.roles[key]
            act, st[1] = st[1], None
            if act[0] == "wait":
                bar, parity, phase = act[1], act[2], act[3]
                if bar.done != phase + 1:
                    raise Violation(f"{key} passed {bar.name} for phase {phase} with {bar.done} completed")
            elif act[0] == "do":
                act[1]()
        raise Violation("no progress bound reached")


def wait(bar, phase):
    return ("wait", bar, phase & 1, phase)


# ---------------------------------------------------------------------------
# Output kernel: record loader, z loader, MMA issuer, two epilogue groups
# ---------------------------------------------------------------------------

def out_protocol(sim, nj, norm, whole):
    B = sim.buf
    full = [MBar(f"full{i}", 1) for i in range(2)]
    rfree = [MBar(f"rfree{i}", 1) for i in range(2)]
    zfull = [MBar(f"zfull{i}", 1) for i in range(4)]
    zfree = [MBar(f"zfree{i}", 1) for i in range(4)]
    afull = [MBar(f"afull{i}", 1) for i in range(4)]
    efree = [MBar(f"efree{i}", 1) for i in range(4)]

    def loader():
        for j in range(nj):
            rs = j & 1
            if j >= 2:
                yield wait(rfree[rs], (j >> 1) - 1)

            def issue(j=j, rs=rs):
                B.begin_write(f"run{rs}", j, "loader")
                sim.launch("tma", [lambda: B.end_write(f"run{rs}", j), full[rs].arrive])
            yield ("do", issue)

    def zloader():
        for j in range(nj):
            g, i = j & 1, j >> 1
            zid = 2 * g + (i & 1)
            if i >= 2:
                yield wait(zfree[zid], (i >> 1) - 1)

            def issue(j=j, zid=zid):
                B.begin_write(f"slot{zid}", j, "zloader")
                sim.launch("tma", [lambda: B.end_write(f"slot{zid}", j), zfull[zid].arrive])
            yield ("do", issue)

    def issuer():
        for j in range(nj):
            rs, a = j & 1, j & 3
            yield wait(full[rs], j >> 1)
            if j >= 4:
                yield wait(efree[a], (j >> 2) - 1)

            def mma(j=j, rs=rs, a=a):
                B.begin_read(f"run{rs}", j, "mma")
                B.begin_write(f"acc{a}", j, "mma")
                sim.launch("issuer", [lambda: B.end_read(f"run{rs}", j, "mma"),
                                      lambda: B.end_write(f"acc{a}", j),
                                      afull[a].arrive, rfree[rs].arrive], ordered=True)
            yield ("do", mma)

    def epilogue(g):
        i = 0
        for j in range(g, nj, 2):
            a, zid = j & 3, 2 * g + (i & 1)
            yield ("stores_read", g)          # the lead's wait for its stores
            if i >= 1:
                yield ("do", zfree[2 * g + ((i - 1) & 1)].arrive)
            if norm:
                yield wait(zfull[zid], i >> 1)
            yield wait(afull[a], j >> 2)

            def use(j=j, a=a, zid=zid):
                B.begin_read(f"acc{a}", j, f"epi{g}")
                if norm:
                    B.begin_read(f"slot{zid}", j, f"epi{g}")
                    B.end_read(f"slot{zid}", j, f"epi{g}")
                B.begin_write(f"slot{zid}", ("out", j), f"epi{g}")   # outputs over the z values
            yield ("do", use)

            def finish(j=j, a=a, zid=zid):
                B.end_write(f"slot{zid}", ("out", j))
                B.end_read(f"acc{a}", j, f"epi{g}")
                efree[a].arrive()
                if whole:
                    B.begin_read(f"slot{zid}", ("out", j), f"store{g}")
                    sim.stores.setdefault(g, set()).add(j)

                    def stored(j=j, zid=zid):
                        B.end_read(f"slot{zid}", ("out", j), f"store{g}")
                        sim.stores[g].discard(j)
                    sim.launch(f"store{g}", [stored])
            yield ("do", finish)
            i += 1
        yield ("stores_read", g)

    sim.add("loader", loader())
    if norm:
        sim.add("zloader", zloader())
    sim.add("issuer", issuer())
    sim.add("epi0", epilogue(0))
    sim.add("epi1", epilogue(1))


@pytest.mark.parametrize("nj", [1, 2, 3, 4, 5, 7, 9, 12])
@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("whole", [True, False])
def test_output_kernel_protocol(nj, norm, whole):
    for seed in range(60):
        sim = Sim(random.Random(1000 * nj + 10 * seed + norm + 2 * whole))
        out_protocol(sim, nj, norm, whole)
        sim.run()


# ---------------------------------------------------------------------------
# Scan kernel: stage loader, two MMA issuers, eight state warps
# ---------------------------------------------------------------------------

def scan_protocol(sim, nck, NS, issuers=2, state_warps=8):
    """The persistent scan CTA: `nck` is the chunk count of one chain or a
    list of them (the chains the CTA runs in turn).  Every role counts the
    steps g over all chains; buffers, stages and parities follow g."""
    B = sim.buf
    lens = [nck] if isinstance(nck, int) else list(nck)
    nck = sum(lens)   # total steps
    firsts = set()    # steps that start a chain
    g = 0
    for L in lens:
        if L:
            firsts.add(g)
        g += L
    full = [MBar(f"full{i}", 1) for i in range(NS)]
    sfree = [MBar(f"sfree{i}", state_warps + issuers) for i in range(NS)]
    chain = MBar("chain", issuers)
    bar_s = NamedBar(state_warps + issuers)

    def loader():
        for c in range(nck):
            st = c % NS
            if c >= NS:
                yield wait(sfree[st], c // NS - 1)

            def issue(c=c, st=st):
                B.begin_write(f"stage{st}", c, "loader")
                sim.launch("tma", [lambda: B.end_write(f"stage{st}", c), full[st].arrive])
            yield ("do", issue)

    def issuer(ii):
        for c in range(nck):
            b, st = c & 1, c % NS
            if ii == 0:
                yield ("stores_read", "copy")   # the copy of S(c-1) has read its buffer
            yield wait(full[st], c // NS)
            yield ("do", lambda c=c: bar_s.arrive(c))
            yield ("sync", bar_s, c)            # S(c) operand written

            def mma(c=c, b=b, st=st):
                B.begin_read(f"stage{st}", c, f"mma{ii}")
                B.begin_read(f"S{b}", c, f"mma{ii}")
                B.begin_write(f"acc{ii}_{b}", c, f"mma{ii}")
                sim.launch(f"issuer{ii}", [lambda: B.end_read(f"stage{st}", c, f"mma{ii}"),
                                           lambda: B.end_read(f"S{b}", c, f"mma{ii}"),
                                           lambda: B.end_write(f"acc{ii}_{b}", c),
                                           chain.arrive, sfree[st].arrive], ordered=True)
                if ii == 0:   # S(c) -> workspace
                    B.begin_read(f"S{b}", c, "copy")
                    sim.stores.setdefault("copy", set()).add(c)

                    def copied(c=c, b=b):
                        B.end_read(f"S{b}", c, "copy")
                        sim.stores["copy"].discard(c)
                    sim.launch("copy", [copied])
            yield ("do", mma)
        if ii == 0:
            yield ("stores_read", "copy")

    def state(w):
        def put(c):
            B.begin_write(f"S{c & 1}", (c, w), f"state{w}")
            B.end_write(f"S{c & 1}", (c, w))
            bar_s.arrive(c)

        for c in range(nck):
            if c in firsts:   # a chain starts: its initial state is the operand of its first step
                yield ("do", lambda c=c: put(c))
            st = c % NS
            yield wait(full[st], c // NS)
            yield wait(chain, c)

            def read(c=c, st=st):
                for ii in range(issuers):
                    B.begin_read(f"acc{ii}_{c & 1}", c, f"state{w}")
                B.begin_read(f"stage{st}", c, f"state{w}")
            yield ("do", read)

            def update(c=c, st=st):
                for ii in range(issuers):
                    B.end_read(f"acc{ii}_{c & 1}", c, f"state{w}")
                if c + 1 < nck and c + 1 not in firsts:   # the chain goes on
                    put(c + 1)
                B.end_read(f"stage{st}", c, f"state{w}")   # released after the fence
                sfree[st].arrive()
            yield ("do", update)

    sim.add("loader", loader())
    for ii in range(issuers):
        sim.add(f"issuer{ii}", issuer(ii))
    for w in range(state_warps):
        sim.add(f"state{w}", state(w))
    return state_warps


def _scan_buffers_hold_whole_states(sim):
    # every state warp writes its part of S(c); the model stores (c, warp)
    # as the content, so readers compare against the chunk only
    orig = sim.buf.begin_read

    def begin_read(buf, unit, who):
        if buf.startswith("S"):
            got = sim.buf.content.get(buf)
            if got is None or got[0] != unit:
                raise Violation(f"{who} reads {buf} expecting S({unit}), holds {got}")
            sim.buf.readers.setdefault(buf, set()).add((who, unit))
            if buf in sim.buf.writers:
                raise Violation(f"{who} reads {buf} while {sim.buf.writers[buf]} writes it")
            return
        orig(buf, unit, who)
    sim.buf.begin_read = begin_read


@pytest.mark.parametrize("nck", [1, 2, 3, 4, 5, 8, 11])
@pytest.mark.parametrize("NS", [4])
def test_scan_kernel_protocol(nck, NS):
    for seed in range(40):
        sim = Sim(random.Random(100 * nck + 7 * seed + NS))
        _scan_buffers_hold_whole_states(sim)
        scan_protocol(sim, nck, NS)
        sim.run()


@pytest.mark.parametrize("lens", [[1, 1, 1], [2, 0, 3], [3, 1, 0, 2, 5], [1, 4, 1, 4], [0, 0, 2]],
                         ids=lambda l: "-".join(map(str, l)))
@pytest.mark.parametrize("NS", [4])
def test_persistent_scan_runs_chains_in_turn(lens, NS):
    """A CTA running several chains back to back (empty ones included): the
    stages and S buffers carry over the chain boundaries by the step count."""
    for seed in range(40):
        sim = Sim(random.Random(31 * sum(lens) + 7 * seed + NS + len(lens)))
        _scan_buffers_hold_whole_states(sim)
        scan_protocol(sim, lens, NS)
        sim.run()


def test_the_model_catches_a_parity_slip():
    """A waiter that skips a phase (here the loader waiting for the previous
    use's phase plus one) is reported, so the checks above are not vacuous."""
    sim = Sim(random.Random(5))
    full = MBar("full", 1)
    free = MBar("free", 1)

    def producer():
        for j in range(4):
            if j >= 1:
                yield wait(free, j)     # should be j - 1
            yield ("do", full.arrive)

    def consumer():
        for j in range(4):
            yield wait(full, j)
            yield ("do", free.arrive)

    sim.add("producer", producer())
    sim.add("consumer", consumer())
    with pytest.raises(Violation):
        sim.run()


# ---------------------------------------------------------------------------
# Planted slips in the protocols above are reported.  Each is applied to a
# copy of this file's source (the first occurrence of the text, which is the
# protocol code: this list comes after it) and the copy's checks must fail.
# ---------------------------------------------------------------------------
PROTOCOL_SLIPS = [
    ("out", "z slot released for the unit in use",
     'yield ("do", zfree[2 * g + ((i - 1) & 1)].arrive)', 'yield ("do", zfree[zid].arrive)'),
    ("out", "accumulator reused two units early",
     "            if j >= 4:\n                yield wait(efree[a], (j >> 2) - 1)",
     "            if j >= 8:\n                yield wait(efree[a], (j >> 2) - 2)"),
    ("out", "run stage refilled without waiting",
     "            if j >= 2:\n                yield wait(rfree[rs], (j >> 1) - 1)", "            pass"),
    ("out", "z tile used without waiting",
     "            if norm:\n                yield wait(zfull[zid], i >> 1)\n", ""),
    ("scan", "S buffer rewritten before its copy has read it",
     '                yield ("stores_read", "copy")   # the copy', "                pass   # the copy"),
    ("scan", "stage released one arrival short",
     'sfree = [MBar(f"sfree{i}", state_warps + issuers)', 'sfree = [MBar(f"sfree{i}", state_warps + issuers - 1)'),
    ("scan", "stage released before it is read",
     "            yield wait(chain, c)\n", "            yield wait(chain, c)\n            yield (\"do\", sfree[c % NS].arrive)\n"),
]


@pytest.mark.parametrize("kind,name,find,repl", PROTOCOL_SLIPS, ids=[s[1] for s in PROTOCOL_SLIPS])
def test_planted_protocol_slip_is_reported(kind, name, find, repl):
    with open(__file__) as f:
        src = f.read()
    assert src.index(find) < src.index("PROTOCOL_SLIPS = ["), f"site of '{name}' not in the protocol code"
    ns = {"__name__": "protocol_copy"}
    exec(compile(src.replace(find, repl, 1), "protocol_copy", "exec"), ns)
    with pytest.raises(AssertionError):
        for seed in range(100):
            for size in (3, 6, 9):
                sim = ns["Sim"](random.Random(seed * 31 + size))
                if kind == "out":
                    ns["out_protocol"](sim, size, True, True)
                else:
                    ns["_scan_buffers_hold_whole_states"](sim)
                    ns["scan_protocol"](sim, size, 4)
                sim.run()
