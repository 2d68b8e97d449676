"""A model of the forward kernel's barrier protocol, checked over random interleavings.

The roles of fwd_tc_kernel (exact_io_aware_38_gb300/csrc/fa_fwd_sm103.cu) for one CTA (two query
tiles against the union of the key tiles they see) are modelled with the kernel's waits, arrivals
and commits (tests/mbarrier_model.py gives the machine and the mbarrier rule):
  producer   Q once; the first key tile's K alone into the K half of the last ring buffer; then
             stage t in buffer t % stages: V of union tile t and K of tile t + 1 under one
             arrive.expect_tx, after the buffer's previous use has been released (empty); when
             query tile 0 skips tile t it also arrives for tile 0's softmax (the stand-in);
  issuer     S_x(0); then per tile: wait stage t (its copies and tile 0's P_0(t)), PV_0(t),
             S_0(t+1), wait P_1(t), PV_1(t), S_1(t+1), release the buffer; O done at the end;
  softmax x  per visible tile: wait S_x, write P_x over S_x (reading O_x for the rescale), arrive
             on stage t's barrier (x = 0) or on p_ready (x = 1); at the end wait for O.
Checked: no deadlock, and no hazard: a buffer reloaded before the MMAs that read its V and K
completed; an MMA issued before its operands landed or its P was written; S_x overwritten before
its P_x was written; O_x rescaled while an earlier PV_x is unfinished; O read before all PV_x.
A planted mistake (the buffer's release committed before its last reader is issued) must be found.

sepp: the single mode at d = 64 (one query tile), where P has columns of its own: per tile the
issuer issues S(t+1) first (the softmax has read S(t) once P(t) is written), then PV(t) and a
commit on pv_done; the softmax waits for pv_done of the previous tile before it rescales O or
writes P. Checked as above, and a softmax that skips that wait must be found.
"""
import random

import pytest
from mbarrier_model import Machine


def run(union, has1, stages, seed, early_release=False, abort_p=0.0, unguarded=False, sepp=False,
        skip_pv_wait=False):
    """union: [(v0, v1)] per union key tile (at least one of the two set).
    unguarded: the earlier abort handling (the issuer and the softmax warpgroups carried on after a
    failed wait, and the producer did not check the abort flag before a copy)."""
    M = Machine(seed, abort_p)
    B, bar, need, done = M.B, M.bar, M.need, M.done

    def wait(name, parity):
        ok = yield from M.wait(name, parity)
        return ok or unguarded
    bar("q", 1)
    bar("k0", 1)
    for i in range(stages):
        bar(f"full{i}", 2)  # the producer's arrive.expect_tx + tile 0's softmax (or the stand-in)
        bar(f"empty{i}", 1)
    for x in (0, 1):
        bar(f"sfull{x}", 1)
        bar(f"odone{x}", 1)
    bar("pready1", 1)  # 128 softmax threads of tile 1, modelled as one arrival
    bar("pvdone", 1)   # sepp: the issuer's commit after each PV
    U = len(union)
    vis = lambda x, t: t < U and bool(union[t][x])

    last_stage = {}  # buffer -> (last stage issued into it, whether tile 0's softmax arrives on it)
    p0_last = [-1]   # the last stage tile 0's softmax arrived on

    def producer():
        M.load("q", 1, ("Q",))
        if U == 0:
            return
        M.load("k0", 1, ("K", 0))
        for t in range(U):
            b = t % stages
            uses = t // stages + (1 if b == stages - 1 else 0)
            ok = True
            if uses > 0:
                ok = yield from M.wait(f"empty{b}", (uses - 1) & 1)
            if ok and t >= stages and not unguarded:  # the buffer's previous stage phase has completed
                ok = yield from M.wait(f"full{b}", ((t - stages) // stages) & 1)
            if ok and (unguarded or not M.aborted):  # after a successful wait, never after an abort
                tv, tk = t - stages, t - stages + 1  # previous V and K of this buffer
                for x in (0, 1):
                    if uses > 0 and tv >= 0 and vis(x, tv):
                        need((f"PV{x}", tv) in done, f"buffer {b} reloaded before PV{x}({tv}) completed")
                    if uses > 0 and vis(x, tk):
                        need((f"S{x}", tk) in done, f"buffer {b} reloaded before S{x}({tk}) completed")
                M.expect(f"full{b}", 2 if t + 1 < U else 1)
                M.copy(f"full{b}", 1, ("V", t))
                if t + 1 < U:
                    M.copy(f"full{b}", 1, ("K", t + 1))
                if not vis(0, t):
                    B[f"full{b}"].arrive()  # stands in for tile 0's softmax
                last_stage[b] = (t, vis(0, t))
            yield None

    def exit_drain():
        """After the CTA-wide barrier at exit, when the CTA has aborted: every stage barrier has at
        most one phase in flight (the last issued); tile 0's softmax arrival on it is made up if it
        never came, then the phase completes once the copies have landed."""
        if not M.aborted:
            return
        for name in ("q", "k0") if U > 0 else ("q",):  # K0 is loaded only when a key tile is visited
            while not B[name].passes(0):
                yield (name, 0)
        for b, (t, needs_p0) in last_stage.items():
            par = (t // stages) & 1
            if B[f"full{b}"].passes(par):
                continue
            if needs_p0 and p0_last[0] < t:
                B[f"full{b}"].arrive()
            while not B[f"full{b}"].passes(par):
                yield (f"full{b}", par)
        need(not M.loads, "the CTA exits with copies in flight")
        yield None

    def issuer():
        last_p = {0: None, 1: None}  # the latest tile whose P_x the issuer has consumed

        def issue_s(x, t):
            need(("K", t) in done, f"S{x}({t}) issued before K({t}) landed")
            if sepp and t > 0:
                need((f"P{x}", t - 1) in done, f"S{x}({t}) over S{x} before the softmax read S{x}({t - 1})")
            if last_p[x] is not None:
                need((f"P{x}", last_p[x]) in done, f"S{x}({t}) over S{x} before P{x}({last_p[x]}) was written")
            M.mma("i", (f"S{x}", t))
            M.commit("i", f"sfull{x}")

        def issue_pv(x, t):
            need(("V", t) in done, f"PV{x}({t}) issued before V({t}) landed")
            need((f"P{x}", t) in done, f"PV{x}({t}) issued before P{x}({t}) was written")
            M.mma("i", (f"PV{x}", t))
            last_p[x] = t

        # After its first wait that fails the issuer issues no MMA and no commit.
        run = yield from wait("q", 0)
        if U == 0:
            return
        if run:
            run = yield from wait("k0", 0)
        if run:
            for x in (0, 1):
                if vis(x, 0):
                    issue_s(x, 0)
            M.commit("i", f"empty{stages - 1}")
        np1 = 0
        for t in range(U):
            if not run:
                break
            b = t % stages
            run = yield from wait(f"full{b}", (t // stages) & 1)
            if not run:
                break
            if early_release:
                M.commit("i", f"empty{b}")
            if sepp:
                if vis(0, t + 1):
                    issue_s(0, t + 1)
                if vis(0, t):
                    issue_pv(0, t)
                    M.commit("i", "pvdone")
            else:
                if vis(0, t):
                    issue_pv(0, t)
                if vis(0, t + 1):
                    issue_s(0, t + 1)
            if vis(1, t):
                run = yield from wait("pready1", np1 & 1)
                np1 += 1
                if not run:
                    break
                issue_pv(1, t)
            if vis(1, t + 1):
                issue_s(1, t + 1)
            if not early_release:
                M.commit("i", f"empty{b}")
            yield None
        for x in (0, 1):
            if run and any(vis(x, t) for t in range(U)):
                M.commit("i", f"odone{x}")

    def softmax(x):
        # After its first wait that fails the warpgroup makes no more arrivals.
        run = yield from wait("q", 0)
        cnt = 0
        for t in range(U):
            if not vis(x, t):
                continue
            if run:
                run = yield from wait(f"sfull{x}", cnt & 1)
            if run:
                need((f"S{x}", t) in done, f"softmax {x} read S({t}) before it completed")
            if run and sepp and cnt > 0 and not skip_pv_wait:  # before the rescale and the P write
                run = yield from wait("pvdone", (cnt - 1) & 1)
            if run:
                for tp in range(t):
                    if vis(x, tp):
                        need((f"PV{x}", tp) in done, f"softmax {x} rescaled O at {t} before PV{x}({tp}) completed")
            yield None
            if run:
                done.add((f"P{x}", t))
                B[f"full{t % stages}" if x == 0 else "pready1"].arrive()
                if x == 0:
                    p0_last[0] = t
            cnt += 1
        if cnt and run:
            run = yield from wait(f"odone{x}", 0)
            if run:
                for tp in range(U):
                    if vis(x, tp):
                        need((f"PV{x}", tp) in done, f"O{x} read before PV{x}({tp}) completed")

    roles = {"prod": producer(), "mma": issuer(), "sm0": softmax(0)}
    if has1:
        roles["sm1"] = softmax(1)
    return M.run(roles, final=exit_drain), M.errors


def _cases(n):
    for seed in range(n):
        r = random.Random(seed * 104729)
        has1 = r.random() < 0.8
        U = r.randint(0, 12)
        union = []
        for _ in range(U):
            v0 = r.random() < 0.7
            v1 = has1 and (not v0 or r.random() < 0.7)
            union.append((v0, v1 if has1 else False))
        union = [u for u in union if u[0] or u[1]]
        yield union, has1, r.choice([1, 2, 4]), seed


def _sepp_cases(n):
    for union, _, stages, seed in _cases(n):
        union = [(True, False) for u in union if u[0]]
        yield union, stages, seed


def test_single_mode_separate_p_has_no_deadlock_or_hazard():
    for union, stages, seed in _sepp_cases(3000):
        res, errs = run(union, False, stages, seed, sepp=True)
        assert res == "ok" and not errs, (union, stages, seed, res, errs[:3])
    for union, stages, seed in _sepp_cases(1500):
        res, errs = run(union, False, stages, seed, abort_p=0.02, sepp=True)
        assert res == "ok" and not errs, (union, stages, seed, res, errs[:3])


def test_model_finds_a_missing_pv_wait():
    found = [seed for union, stages, seed in _sepp_cases(3000)
             if run(union, False, stages, seed, sepp=True, skip_pv_wait=True)[1]]
    assert found, "the model no longer sees P or O written before the previous PV completed"


def test_protocol_has_no_deadlock_or_hazard():
    for union, has1, stages, seed in _cases(3000):
        res, errs = run(union, has1, stages, seed)
        assert res == "ok" and not errs, (union, has1, stages, seed, res, errs[:3])


def test_model_finds_an_early_buffer_release():
    found = [seed for union, has1, stages, seed in _cases(3000)
             if run(union, has1, stages, seed, early_release=True)[1]]
    assert found, "the model no longer sees a buffer released before its readers"


def test_abort_path_terminates():
    """Waits that run out at random points: every role still leaves its loops, no stage barrier
    gets an arrival beyond its count (a second arrive.expect_tx, or tile 0's softmax arriving for a
    later use of the buffer, while a phase is in flight), no hazard is issued, and the exit drain
    leaves no copy in flight."""
    for union, has1, stages, seed in _cases(1500):
        res, errs = run(union, has1, stages, seed, abort_p=0.02)
        assert res == "ok" and not errs, (union, has1, stages, seed, res, errs[:3])


def test_abort_path_model_sees_the_unguarded_release():
    """With the earlier abort handling the model must hit an arrival beyond a stage barrier's
    count (the undefined pending-count underflow): the model can see that fault."""
    for union, has1, stages, seed in _cases(1500):
        try:
            run(union, has1, stages, seed, abort_p=0.02, unguarded=True)
        except AssertionError:
            return
    raise AssertionError("the model no longer sees the unguarded abort path")
