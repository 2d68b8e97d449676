"""A small executable model of mbarrier-synchronised kernels, for the protocol tests.

A kernel's roles are Python generators that yield while they wait. The machine holds the
mbarriers, the TMA copies in flight and one in-order queue of tensor-core operations per issuing
thread. Each tick it resumes a random role whose wait would pass, completes a random copy, or
retires the head of a random non-empty MMA queue; a commit in a queue arrives on its barrier when
it reaches the head (it completes after every earlier operation of that thread).

mbarrier rule (as on the hardware): a phase completes when the expected arrivals and the expected
transaction bytes are all in, and the barrier moves to the next phase; try_wait.parity(P) passes
iff the current phase's parity differs from P. A waiter that falls two phases behind therefore
waits for a phase that may never come.
"""
import random


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phase, self.tx = name, count, count, 0, 0

    def arrive(self, n=1):
        self.pending -= n
        if self.pending < 0:
            raise AssertionError(f"{self.name}: more arrivals than the count")
        self._maybe()

    def expect_tx(self, b):
        self.tx += b
        self.arrive()

    def tx_done(self, b):
        self.tx -= b
        self._maybe()

    def _maybe(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def passes(self, parity):
        return (self.phase & 1) != parity


class Machine:
    def __init__(self, seed, abort_p=0.0):
        self.rnd = random.Random(seed)
        # Bounded waits: with probability abort_p a blocked wait runs out; from then on (the CTA's
        # abort flag is set) every wait returns at once, as in the kernels.
        self.abort_p = abort_p
        self.aborted = False
        self.B = {}
        self.loads = []  # (barrier, bytes, record)
        self.pipe = {}
        self.done = set()  # completed copies, MMAs and other recorded events
        self.errors = []

    def bar(self, name, count):
        self.B[name] = Bar(name, count)

    def need(self, cond, msg):
        if not cond:
            self.errors.append(msg)

    def wait(self, name, parity):
        """Generator; its return value is True once the phase has completed, False if the wait ran
        out (or the abort flag was already set)."""
        while not self.B[name].passes(parity):
            if self.aborted or (self.abort_p and self.rnd.random() < self.abort_p):
                self.aborted = True
                return False
            yield (name, parity)
        return True

    def load(self, name, nbytes, record):
        """One arrival with its byte count, and the copy that delivers the bytes."""
        self.B[name].expect_tx(nbytes)
        self.loads.append((name, nbytes, record))

    def expect(self, name, nbytes):
        """arrive.expect_tx for several copies issued with copy()."""
        self.B[name].expect_tx(nbytes)

    def copy(self, name, nbytes, record):
        self.loads.append((name, nbytes, record))

    def mma(self, who, label):
        self.pipe.setdefault(who, []).append(("mma", label))

    def commit(self, who, name):
        self.pipe.setdefault(who, []).append(("commit", name))

    def run(self, roles, max_ticks=400000, final=None):
        """'ok', 'deadlock' (nothing can move while a role is unfinished) or 'timeout'.
        final: a generator function started as one more role once every other role has finished
        (code after a CTA-wide barrier, e.g. an exit drain), while copies may still be in flight."""
        roles = dict(roles)
        blocked = {k: None for k in roles}
        alive = set(roles)
        for _ in range(max_ticks):
            if not alive and final is not None:
                roles["exit"], blocked["exit"], final = final(), None, None
                alive.add("exit")
            # With bounded waits a blocked role stays schedulable: resumed, its wait may run out.
            cands = [("role", k) for k in sorted(alive)
                     if blocked[k] is None or self.abort_p or self.B[blocked[k][0]].passes(blocked[k][1])]
            if self.loads:
                cands.append(("load", None))
            cands += [("pipe", w) for w in sorted(self.pipe) if self.pipe[w]]
            if not cands:
                if alive:
                    self.errors.append(f"deadlock: {sorted((k, blocked[k]) for k in alive)}")
                    return "deadlock"
                return "ok"
            c = self.rnd.choice(cands)
            if c[0] == "role":
                try:
                    blocked[c[1]] = next(roles[c[1]])
                except StopIteration:
                    alive.discard(c[1])
            elif c[0] == "load":
                name, b, record = self.loads.pop(self.rnd.randrange(len(self.loads)))
                self.done.add(record)
                self.B[name].tx_done(b)
            else:
                op = self.pipe[c[1]].pop(0)
                if op[0] == "mma":
                    self.done.add(op[1])
                else:
                    self.B[op[1]].arrive()
        return "timeout"
