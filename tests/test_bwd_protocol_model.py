"""A model of the backward main kernel's barrier protocol, checked over random interleavings.

The roles of bwd_tc_kernel (exact_io_aware_38_gb300/csrc/fa_bwd_sm103.cu) are modelled as
generators with the kernel's waits, arrivals and commits: the TMA producer with the key-tile queue,
the S^T/dP^T issuer, the gradient issuer, the elementwise and dQ warpgroups. Each tick resumes a
random role whose wait would pass, completes a random TMA copy, or retires the head of either
issuer's in-order MMA queue (a commit arrives when it reaches the head). mbarriers follow the
hardware rule: a phase completes when its arrivals and transaction bytes are in, and
try_wait.parity(P) passes iff the current phase's parity differs from P, so a waiter that falls
two phases behind waits forever. Checked: no deadlock, and no writer issued while readers of the
data it overwrites are unfinished (a Q/dO stage or K/V reloaded, TMEM columns or the dS tile
rewritten, the dK/dV accumulators overwritten before their read-out).

The same model with the earlier producer release (waiting on the two dq_full barriers for step
i - 3) must deadlock on some interleaving: that aliasing hang is what the per-stage release fixes,
and finding it shows the model can see that class of error.

Abort path: waits that run out at random. After the CTA's abort flag is set every role keeps its
loops (a failed wait returns false at once; the issuers and warpgroups carry on with stale data,
which only spoils the outputs of a call that has already failed, so hazards after the abort are not
errors). What must hold: no barrier gets an arrival beyond its count (a second arrive.expect_tx on
an open phase), every role ends, and no copy is in flight when the producer has drained at exit.
The producer guarantees the first on its own: before reloading a stage (or K/V) it checks that the
stage's previous copy has landed, and it issues nothing once the abort flag is set.

single: the single mode that d = 64 runs (two CTAs per SM): one tensor-memory buffer, a two-deep
Q/dO ring, one K/V buffer, one issuer for the whole step chain and one warpgroup that writes P^T
and dS^T, reads out dQ^T and both accumulators. Its issue order per step is dP^T, S^T (after the
previous dQ^T's read-out: dQ^T accumulates over the S^T columns), then dV, dQ^T, dK. Overwrites that
the in-order MMA queue orders (dQ^T of step s over the P^T that dV of step s reads, dP^T of step s
over the dS^T that dK of step s - 1 reads) are checked as "issued earlier in the same queue".
"""
import random

import pytest
from mbarrier_model import Machine

KST, NB = 3, 2


def run(tiles, seed, release="stage", abort_p=0.0, unguarded=False, single=False):
    """unguarded: the earlier producer, which reloaded a stage once its release arrived, without
    checking its own previous copy or the abort flag."""
    KST, NB = (2, 1) if single else (3, 2)
    M = Machine(seed, abort_p)
    B, bar, wait, done, mma, commit = M.B, M.bar, M.wait, M.done, M.mma, M.commit

    def need(cond, msg):  # a hazard matters only before the abort (afterwards the outputs are void)
        if not M.aborted:
            M.need(cond, msg)

    bar("kv", 1)
    bar("done", 1)
    for i in range(KST):
        bar(f"full{i}", 1)
        bar(f"empty{i}", 1)
    for i in range(NB):
        for n in ("sfull", "dqfull", "sfree"):
            bar(f"{n}{i}", 1)
        bar(f"pready{i}", 1)  # 128 elementwise threads, modelled as one arrival
        bar(f"dqfree{i}", 1)  # 128 dQ threads
    for i in range(2):
        bar(f"tqfull{i}", 1)
        bar(f"tqempty{i}", 2 if single else 4)  # the issuers and the warpgroups' leaders
    bar("accfree", 1 if single else 2)  # the warpgroups
    bar("drain", 1 if single else 2)

    ntiles = len(tiles)
    tile_q = [None, None]
    counter = [0]
    grid = 1
    def take_tile(w):
        ok = yield from wait(f"tqfull{w & 1}", (w >> 1) & 1)
        t = tile_q[w & 1] if ok else ntiles  # a wait that ran out ends the role's tile loop
        B[f"tqempty{w & 1}"].arrive()
        return t

    # step -> work-tile index, filled by the producer (all roles walk the same sequence)
    step_tile = {}

    last_par = {}  # "kv" or stage -> parity of the last phase the producer issued copies for

    def drain():
        """At exit, after an abort: wait (ignoring the abort flag) for the last phase of every
        barrier that got copies; with at most one phase in flight each, no copy is left."""
        if not M.aborted:
            return
        for name, par in last_par.items():
            while not B[name].passes(par):
                yield (name, par)
        M.need(not M.loads, "the CTA exits with copies in flight")

    def landed(name):
        """The producer's own previous copy into this barrier has landed (only it arrives there)."""
        if unguarded or name not in last_par:
            return True
        return (yield from wait(name, last_par[name]))

    def producer():
        yield from producer_loop()
        yield from drain()

    def producer_loop():
        i, wt, w = 0, 0, 0
        while True:
            if w >= 2:
                ok = yield from wait(f"tqempty{w & 1}", ((w - 2) >> 1) & 1)
                if not ok:
                    return  # the producer stops taking tiles; the readers' waits run out too
            t = w if w == 0 else grid + counter[0]
            if w > 0:
                counter[0] += 1
            t = ntiles if M.aborted and not unguarded else min(t, ntiles)  # after an abort: the end marker
            tile_q[w & 1] = t
            B[f"tqfull{w & 1}"].arrive()
            w += 1
            yield None
            if t >= ntiles:
                return
            n = tiles[t]
            if n == 0:
                continue
            kv_issued = False

            def issue_kv():
                if wt >= 1:
                    if not (yield from wait("done", (wt - 1) & 1)):
                        return  # the kernel skips the copy after a wait that ran out
                if not (yield from landed("kv")) or (M.aborted and not unguarded):
                    return
                if wt >= 1:
                    # every MMA of the previous work tile has completed (they read K and V)
                    for s in [s for s, tt in step_tile.items() if tt == wt - 1]:
                        for k in ("S", "dP", "dQ"):
                            need((k, s) in done, f"K/V of work tile {wt} loaded before {k}{s} completed")
                M.load("kv", 2, ("kv", wt))
                last_par["kv"] = wt & 1

            if wt == 0:
                yield from issue_kv()
                kv_issued = True
            for l in range(n):
                if l == 2 and not kv_issued:
                    yield from issue_kv()
                    kv_issued = True
                st, j = i % KST, i - KST
                ok = True
                if j >= 0:
                    if release == "stage":  # the kernel: one release barrier per stage
                        ok = yield from wait(f"empty{j % KST}", (j // KST) & 1)
                    else:  # an earlier form: the NB-deep dq_full barriers of the TMEM buffers
                        ok = yield from wait(f"dqfull{j % NB}", (j // NB) & 1)
                    ok = ok and (yield from landed(f"full{st}"))
                step_tile[i] = wt
                if ok and (unguarded or not M.aborted):  # after its waits succeeded, never after an abort
                    if j >= 0:
                        for k in ("S", "dP", "dV", "dK"):
                            need((k, j) in done, f"stage {st} reloaded for step {i} before {k}{j} completed")
                    M.load(f"full{st}", 1, ("qdo", i))
                    last_par[f"full{st}"] = (i // KST) & 1
                i += 1
                yield None
            if not kv_issued:
                yield from issue_kv()
            wt += 1

    def issuer1():
        sn, wt, w = 0, 0, 0
        while True:
            t = yield from take_tile(w)
            w += 1
            if t >= ntiles:
                break
            n = tiles[t]
            if n == 0:
                continue
            yield from wait("kv", wt & 1)
            need(("kv", wt) in done, f"S issuer saw K/V of work tile {wt} before they landed")
            for _ in range(n):
                st, buf = sn % KST, sn % NB
                yield from wait(f"full{st}", (sn // KST) & 1)
                need(("qdo", sn) in done, f"S^T{sn} issued before its Q/dO landed")
                if sn >= NB:
                    yield from wait(f"sfree{buf}", ((sn - NB) // NB) & 1)
                    need(("dV", sn - NB) in done, f"S^T{sn} over P^T before dV{sn - NB} completed")
                mma(1, ("S", sn))
                if sn >= NB:
                    yield from wait(f"dqfree{buf}", ((sn - NB) // NB) & 1)
                    for k in ("dK", "dQ", "rdQ"):
                        need((k, sn - NB) in done, f"dP^T{sn} over dS^T/dQ^T before {k}{sn - NB}")
                mma(1, ("dP", sn))
                commit(1, f"sfull{buf}")
                sn += 1
                yield None
            wt += 1
        commit(1, "drain")

    def issuer2():
        g, wt, w = 0, 0, 0
        while True:
            t = yield from take_tile(w)
            w += 1
            if t >= ntiles:
                break
            n = tiles[t]
            if n == 0:
                continue
            if wt > 0:
                yield from wait("accfree", (wt - 1) & 1)
                need(("acc_ew", wt - 1) in done and ("acc_dq", wt - 1) in done,
                     f"accumulators of work tile {wt - 1} overwritten before their read-out")
            for _ in range(n):
                st, buf = g % KST, g % NB
                yield from wait(f"pready{buf}", (g // NB) & 1)
                need(("P", g) in done, f"dV{g} issued before P/dS of step {g} were written")
                mma(2, ("dV", g))
                commit(2, f"sfree{buf}")
                mma(2, ("dK", g))
                commit(2, f"empty{st}")
                mma(2, ("dQ", g))
                commit(2, f"dqfull{buf}")
                g += 1
                yield None
            commit(2, "done")
            wt += 1
        commit(2, "drain")

    def issuer_single():
        sn, wt, w = 0, 0, 0
        queued = set()  # operations already in this thread's in-order queue

        def mma1(rec):
            mma(1, rec)
            queued.add(rec)

        while True:
            t = yield from take_tile(w)
            w += 1
            if t >= ntiles:
                break
            n = tiles[t]
            if n == 0:
                continue
            yield from wait("kv", wt & 1)
            need(("kv", wt) in done, f"issuer saw K/V of work tile {wt} before they landed")
            for l in range(n):
                st = sn % KST
                yield from wait(f"full{st}", (sn // KST) & 1)
                need(("qdo", sn) in done, f"S^T{sn} issued before its Q/dO landed")
                if sn >= 1:
                    need(("dK", sn - 1) in queued, f"dP^T{sn} over dS^T ahead of dK{sn - 1} in the queue")
                mma1(("dP", sn))
                if sn >= 1:
                    yield from wait("dqfree0", (sn - 1) & 1)
                    need(("rdQ", sn - 1) in done, f"S^T{sn} over dQ^T{sn - 1} before its read-out")
                mma1(("S", sn))
                commit(1, "sfull0")
                if l == 0 and wt > 0:
                    yield from wait("accfree", (wt - 1) & 1)
                    need(("acc_ew", wt - 1) in done and ("acc_dq", wt - 1) in done,
                         f"accumulators of work tile {wt - 1} overwritten before their read-out")
                yield from wait("pready0", sn & 1)
                need(("P", sn) in done, f"dV{sn} issued before P/dS of step {sn} were written")
                mma1(("dV", sn))
                need(("dV", sn) in queued, f"dQ^T{sn} over P^T ahead of dV{sn} in the queue")
                mma1(("dQ", sn))
                commit(1, "dqfull0")
                mma1(("dK", sn))
                commit(1, f"empty{st}")
                sn += 1
                yield None
            commit(1, "done")
            wt += 1
        commit(1, "drain")

    def group_single():
        it, wt, w = 0, 0, 0
        while True:
            t = yield from take_tile(w)
            w += 1
            if t >= ntiles:
                break
            n = tiles[t]
            for _ in range(n):
                yield from wait("sfull0", it & 1)
                need(("S", it) in done and ("dP", it) in done, f"P/dS of step {it} before S/dP completed")
                if it >= 1:  # dS^T into the shared-memory tile read by dQ of step it - 1
                    need(("dQ", it - 1) in done, f"dS^T{it} written before dQ{it - 1} completed")
                done.add(("P", it))
                B["pready0"].arrive()
                yield None
                yield from wait("dqfull0", it & 1)
                need(("dQ", it) in done, f"dQ^T{it} read before it completed")
                done.add(("rdQ", it))
                B["dqfree0"].arrive()
                it += 1
                yield None
            if n > 0:
                yield from wait("done", wt & 1)
                for s in [s for s, tt in step_tile.items() if tt == wt]:
                    need(("dV", s) in done and ("dK", s) in done, f"read-out of work tile {wt} before dV/dK{s}")
                yield None
                done.add(("acc_ew", wt))
                done.add(("acc_dq", wt))
                B["accfree"].arrive()
                wt += 1

    def group(kind):
        it, wt, w = 0, 0, 0
        while True:
            t = yield from take_tile(w)
            w += 1
            if t >= ntiles:
                break
            n = tiles[t]
            for _ in range(n):
                buf = it % NB
                if kind == "ew":
                    yield from wait(f"sfull{buf}", (it // NB) & 1)
                    need(("S", it) in done and ("dP", it) in done, f"P/dS of step {it} before S/dP completed")
                    if it >= NB:  # dS^T into the shared-memory tile read by dQ of step it - NB
                        need(("dQ", it - NB) in done, f"dS^T{it} written before dQ{it - NB} completed")
                    done.add(("P", it))
                    B[f"pready{buf}"].arrive()
                else:
                    yield from wait(f"dqfull{buf}", (it // NB) & 1)
                    need(("dQ", it) in done, f"dQ^T{it} read before it completed")
                    done.add(("rdQ", it))
                    B[f"dqfree{buf}"].arrive()
                it += 1
                yield None
            if n > 0:
                yield from wait("done", wt & 1)
                last = [s for s, tt in step_tile.items() if tt == wt]
                for s in last:
                    need(("dV", s) in done and ("dK", s) in done, f"read-out of work tile {wt} before dV/dK{s}")
                yield None
                done.add(("acc_" + kind, wt))
                B["accfree"].arrive()
                wt += 1

    if single:
        roles = {"prod": producer(), "i": issuer_single(), "g": group_single()}
    else:
        roles = {"prod": producer(), "i1": issuer1(), "i2": issuer2(), "ew": group("ew"), "dr": group("dq")}
    return M.run(roles), M.errors


def _cases(n):
    for seed in range(n):
        r = random.Random(seed * 7919)
        yield [r.choice([0, 0, 1, 1, 2, 3, 4, 5, 7]) for _ in range(r.randint(1, 10))], seed


@pytest.mark.parametrize("single", [False, True])
def test_protocol_has_no_deadlock_or_hazard(single):
    for tiles, seed in _cases(3000):
        res, errs = run(tiles, seed, single=single)
        assert res == "ok" and not errs, (tiles, seed, res, errs[:3])


def test_model_finds_the_earlier_release_race():
    hangs = [seed for tiles, seed in _cases(3000) if run(tiles, seed, release="dq_full")[0] == "deadlock"]
    assert hangs, "the model no longer sees the aliasing deadlock of the earlier release"


@pytest.mark.parametrize("single", [False, True])
def test_abort_path_terminates(single):
    """Waits that run out at random points: every role still leaves its loops (the kernel's abort
    flag makes every later wait return at once; a tile-queue read that fails ends the role's tile
    loop), even when the roles no longer agree on how many tiles they saw; no barrier gets an
    arrival beyond its count (the mbarrier model raises); the drain leaves no copy in flight."""
    for tiles, seed in _cases(1500):
        res, errs = run(tiles, seed, abort_p=0.02, single=single)
        assert res == "ok" and not errs, (tiles, seed, res, errs[:3])


def test_abort_path_model_sees_the_unguarded_producer():
    """The earlier producer (reloading a stage on its release alone) must hit the second
    arrive.expect_tx on an open phase: the model can see that fault."""
    for tiles, seed in _cases(1500):
        try:
            run(tiles, seed, abort_p=0.02, unguarded=True)
        except AssertionError:
            return
    raise AssertionError("the model no longer sees the unguarded producer")
