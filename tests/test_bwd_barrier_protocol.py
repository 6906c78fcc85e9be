"""CPU model of the backward main kernel's mbarrier protocol (no GPU).

`fa2_bwd_kernel` runs a TMA producer, one MMA issuer, two P/dS warpgroups
and a dQ drain warpgroup (whose first lane also issues the TMA reduces)
over the query tiles of one key/value tile.  This model replays each
role's waits, arrivals, loads, MMA commits and bulk reduces with the
kernel's barrier counts (BwdBar enum) and stage counts (two Q stages, one
or two dO stages, dQ in 1, 2 or 4 pieces of at most 32 columns), lets loads
land and reduces finish reading in any order, and checks that no wait is
two phases away from its barrier and that every run ends
(`protocol_model.Engine`).  It also tracks the shared-memory buffers the
barriers guard and reports a hazard when a Q or dO stage is reloaded, or the
dS^T buffer rewritten, while an MMA that reads it may still run.  With one
dO stage the stage is free once dV(i) is done.  The dS^T buffer needs no
barrier of its own: its last reader dK(i-1) is issued before dP^T(i), and
the commit that completes dP-full tracks every earlier MMA of the issuing
thread (the model's in-order MMA queue), so the P/dS warps, which wait for
dP^T(i) before writing dS^T(i), find the buffer free.
"""
import random

import pytest

from protocol_model import Engine

SQ = 2  # Q stages


def backward_roles(e, n_iter, sd, pieces, early_release=False, planted=None):
    e.bar("KV", 1)
    for s in range(2):
        for name in ("QFull", "QEmpty", "DoFull", "DoEmpty"):
            e.bar((name, s), 1, f"{name}[{s}]")
        e.bar(("StageFull", s), 4, f"StageFull[{s}]")
        e.bar(("StageFree", s), 1, f"StageFree[{s}]")
    for name, count in (("SFull", 1), ("DpFull", 1), ("PFull", 8), ("DvDone", 1), ("DsFull", 8),
                        ("DqFull", 1), ("DqDrained", 4), ("AccFull", 1), ("Drain", 1)):
        e.bar(name, count)

    reading = {}  # buffer -> MMAs in flight that read it

    def hazard(msg):
        if e.error is None:
            e.error = "hazard: " + msg

    def load(key):
        e.unordered(lambda: e.arrive(key))

    def commit(*keys):
        for key in keys:
            if planted == "dp_full_not_ordered" and key == "DpFull":
                e.unordered(lambda key=key: e.arrive(key))  # arrives without waiting for earlier MMAs
            else:
                e.ordered("mma", lambda key=key: e.arrive(key))

    def mma(tag, *buffers):  # an MMA group reading shared-memory buffers
        for b in buffers:
            reading.setdefault(b, set()).add(tag)

        def done():
            for b in buffers:
                reading[b].discard(tag)

        e.ordered("mma", done)

    def overwrite(buffer, what):
        if reading.get(buffer):
            hazard(f"{what} while {sorted(reading[buffer])} may read it")

    def producer():
        load("KV")
        for it in range(n_iter):
            st, u = it % SQ, it // SQ
            if it >= SQ:
                yield ("QEmpty", st), u - 1
            overwrite(("Q", st), f"Q stage {st} reloaded for tile {it}")
            load(("QFull", st))
            st, u = it % sd, it // sd
            if it >= sd:
                if sd == 1:  # one stage: dV(it - 1), its last reader, done frees it
                    if planted != "dO_freed_by_dP":
                        yield "DvDone", it - 1
                    else:
                        yield "DpFull", it - 1
                else:
                    yield ("DoEmpty", st), u - 1
            overwrite(("dO", st), f"dO stage {st} reloaded for tile {it}")
            load(("DoFull", st))

    def issuer():
        yield "KV", 0
        yield ("QFull", 0), 0
        mma("S0", ("Q", 0))
        commit("SFull")
        for it in range(n_iter):
            qs, ds, du = it % SQ, it % sd, it // sd
            yield ("DoFull", ds), du
            if it >= 1:
                yield "DqDrained", it - 1
            mma(f"dP{it}", ("dO", ds))
            commit("DpFull")
            yield "PFull", it
            mma(f"dV{it}", ("dO", ds))
            commit(*([("DoEmpty", ds)] if sd > 1 else []), "DvDone")
            dq_done = False
            if it + 1 < n_iter:
                yield "DvDone", it
                yield ("QFull", (it + 1) % SQ), (it + 1) // SQ
                mma(f"S{it + 1}", ("Q", (it + 1) % SQ))
                # dQ(i) goes out before the last quarter of S(i+1) when dS(i)
                # is already there (a non-blocking test in the kernel)
                if e.bars["DsFull"].done >= it + 1:
                    mma(f"dQ{it}", "dS")
                    commit("DqFull")
                    dq_done = True
                commit("SFull")
            if not dq_done:
                yield "DsFull", it
                mma(f"dQ{it}", "dS")
                commit("DqFull")
            mma(f"dK{it}", "dS", ("Q", qs))
            commit(("QEmpty", qs))
        commit("AccFull", "Drain")
        yield "Drain", 0

    def p_ds():
        for it in range(n_iter):
            yield ("QFull", it % SQ), it // SQ
            yield "SFull", it
            e.arrive("PFull")
            yield "DpFull", it
            overwrite("dS", f"dS^T of tile {it} written")
            e.arrive("DsFull")

    read_done, issued = set(), []

    def drain(w):
        for it in range(n_iter):
            yield "DqFull", it
            if pieces <= 3 or early_release:
                e.arrive("DqDrained")
            for c in range(pieces):
                gi = it * pieces + c
                bsel, u = gi & 1, gi >> 1
                if gi >= 2:
                    yield ("StageFree", bsel), u - 1
                e.arrive(("StageFull", bsel))
                if pieces == 4 and c == 0:  # the fourth piece is read, then the columns released
                    e.arrive("DqDrained")
                if w == 0:  # lane 0 of the first drain warp issues the reduce
                    yield ("StageFull", bsel), u
                    issued.append(gi)
                    e.unordered(lambda gi=gi: read_done.add(gi))
                    if gi >= 1:
                        older = list(issued[:-1])
                        yield ("cond", lambda older=older: all(g in read_done for g in older),
                               "bulk reads of the older reduces")
                        e.arrive(("StageFree", bsel ^ 1))
        yield "AccFull", 0

    roles = {"producer": producer(), "issuer": issuer()}
    for w in range(8):
        roles[f"P/dS {w}"] = p_ds()
    for w in range(4):
        roles[f"drain {w}"] = drain(w)
    return roles


@pytest.mark.parametrize("sd,pieces", [(1, 4), (2, 2), (2, 1)], ids=["d128", "d64", "d32_d16"])
def test_backward_protocol_has_no_deadlock_or_parity_aliasing(sd, pieces):
    for seed in range(300):
        n_iter = random.Random(seed).randint(1, 12)
        e = Engine(seed)
        result = e.run(backward_roles(e, n_iter, sd, pieces))
        assert result is None, f"seed {seed}, {n_iter} query tiles: {result}"


def test_model_catches_the_ds_buffer_rewritten_if_dp_full_did_not_track_dk():
    # Without the commit's tracking of earlier MMAs, dS^T(i) could overwrite
    # the buffer while dK(i-1) still reads it.
    found = None
    for seed in range(300):
        e = Engine(seed)
        found = e.run(backward_roles(e, random.Random(seed).randint(2, 12), 1, 4, planted="dp_full_not_ordered"))
        if found:
            break
    assert found and "hazard" in found and "dS^T" in found


def test_model_catches_the_do_stage_reloaded_before_dv_is_done():
    # With one dO stage the stage must wait for dV(i-1), not just dP(i-1).
    found = None
    for seed in range(300):
        e = Engine(seed)
        found = e.run(backward_roles(e, random.Random(seed).randint(2, 12), 1, 4, planted="dO_freed_by_dP"))
        if found:
            break
    assert found and "hazard" in found and "dO stage" in found


def test_model_catches_a_second_release_of_the_dq_columns():
    # A drain that also released the dQ columns right after its first read
    # (as well as after the fourth piece) would run the barrier two phases
    # past the MMA issuer's wait.
    found = None
    for seed in range(300):
        e = Engine(seed)
        found = e.run(backward_roles(e, random.Random(seed).randint(2, 12), 1, 4, early_release=True))
        if found:
            break
    assert found and "DqDrained" in found
