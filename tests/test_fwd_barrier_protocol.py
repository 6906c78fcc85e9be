"""CPU model of the forward kernel's mbarrier protocol (no GPU).

`fa2_fwd_kernel` coordinates its roles (TMA producer, two MMA issuers, two
groups of four softmax warps) through mbarriers waited on by phase parity.
This model replays each role's sequence of waits, arrivals, TMA loads and
MMA commits (`protocol_model.Engine`: loads land in any order, one issuer's
commits in issue order) and checks that no wait is ever two phases away
from its barrier and that every run ends.  Barrier names and counts follow
the kernel's FwdBar enum; a unit is the pair (K/V tiles of query tile A,
K/V tiles of query tile B) that `fwd_unit` computes.  The scheduler
barriers (one response per unit, read by all eleven roles) are included.
"""
import random

import pytest

from protocol_model import Engine


def forward_roles(e, units, skip_full_waits=True, turns=True, dual=False, seed=0, one_p_full=False,
                  phantom_turns_a=False):
    """Roles of one CTA.  ``dual``: decoding (tile B never has rows), where
    tile A alternates its S / P / PV barriers between the two S buffers and
    issues S(j+1) before PV(j)."""
    rng = random.Random(seed + 7)

    def buf(x, k):  # S buffer (and barrier index) of a tile's k-th S, and its use count
        return (k & 1, k >> 1) if dual else (x, k)

    def p_full(x, k):  # P-full barrier and completion number of a tile's k-th P
        if one_p_full:  # (one barrier per tile even when S is double-buffered)
            return ("PFull", x), k
        b, i = buf(x, k)
        return ("PFull", b), i

    for s in range(2):
        for name, count in (("QFull", 1), ("QEmpty", 1), ("KFull", 1), ("KEmpty", 2), ("VFull", 1),
                            ("VEmpty", 2), ("SFull", 1), ("PFull", 4), ("PVDone", 1), ("SchedFull", 1),
                            ("SchedEmpty", 11)):
            e.bar((name, s), count, f"{name}[{s}]")
    for w in range(4):
        e.bar(("TokA", w), 1, f"TokA[{w}]")
        e.bar(("TokB", w), 1, f"TokB[{w}]")

    def load(key):
        e.unordered(lambda: e.arrive(key))

    def commit(x, *keys):
        for key in keys:
            e.ordered(("mma", x), lambda key=key: e.arrive(key))

    def producer():
        g, qn = 0, [0, 0]
        for n, (na, nb) in enumerate(units):
            def load_q(x):
                if qn[x] >= 1:
                    yield ("QEmpty", x), qn[x] - 1
                load(("QFull", x))
                qn[x] += 1

            if na > 0:
                yield from load_q(0)
            for j in range(max(na, nb)):
                st = g & 1
                if g >= 2:
                    yield ("KEmpty", st), (g >> 1) - 1
                load(("KFull", st))
                if g >= 2:
                    yield ("VEmpty", st), (g >> 1) - 1
                load(("VFull", st))
                if j == 0 and nb > 0:
                    yield from load_q(1)
                g += 1
            if n >= 2:
                yield ("SchedEmpty", n & 1), (n >> 1) - 1
            load(("SchedFull", n & 1))
            yield ("SchedFull", n & 1), n >> 1
            e.arrive(("SchedEmpty", n & 1))

    def issuer(x):
        g = k = qn = 0
        for n, cnt in enumerate(units):
            n_kv, nx = max(cnt), cnt[x]
            if n_kv > 0:
                def s_ready(kk):  # S number kk may overwrite its buffer
                    prev = kk - 2 if dual else kk - 1
                    if prev >= 0:
                        b, i = buf(x, prev)
                        yield ("PVDone", b), i

                def issue_s(kk, st, last):
                    b, _ = buf(x, kk)
                    commit(x, ("SFull", b), ("KEmpty", st), *([("QEmpty", x)] if last else []))

                if nx > 0:
                    yield ("QFull", x), qn
                    qn += 1
                    yield from s_ready(k)
                    yield ("KFull", g & 1), g >> 1
                    issue_s(k, g & 1, nx == 1)
                for j in range(nx):
                    gj = g + j
                    st = gj & 1
                    if dual and j + 1 < nx:
                        yield from s_ready(k + 1)
                        yield ("KFull", st ^ 1), (gj + 1) >> 1
                        issue_s(k + 1, st ^ 1, j + 2 == nx)
                    yield ("VFull", st), gj >> 1
                    yield p_full(x, k)
                    b, _ = buf(x, k)
                    commit(x, ("PVDone", b), ("VEmpty", st))
                    k += 1
                    if not dual and j + 1 < nx:
                        yield from s_ready(k)
                        yield ("KFull", st ^ 1), (gj + 1) >> 1
                        issue_s(k, st ^ 1, j + 2 == nx)
                for j in range(nx, n_kv):  # K/V tiles this issuer does not visit
                    gj = g + j
                    st = gj & 1
                    if skip_full_waits:
                        yield ("KFull", st), gj >> 1
                        yield ("VFull", st), gj >> 1
                    if gj >= 2:
                        yield ("KEmpty", st), (gj >> 1) - 1
                    e.arrive(("KEmpty", st))
                    if gj >= 2:
                        yield ("VEmpty", st), (gj >> 1) - 1
                    e.arrive(("VEmpty", st))
                g += n_kv
            yield ("SchedFull", n & 1), n >> 1
            e.arrive(("SchedEmpty", n & 1))

    def softmax(x, w):
        k = tn = 0
        tok_wait, tok_pass = (("TokB", w), ("TokA", w)) if x else (("TokA", w), ("TokB", w))
        for n, cnt in enumerate(units):
            nx = cnt[x]
            # turns only for the K/V tiles both query tiles visit
            n_turns = min(cnt) if (turns and not dual and min(cnt) > 0) else 0
            if phantom_turns_a and x == 0 and n_turns:  # planted: tile A also takes turns for B's extra tiles
                n_turns = max(cnt)
            for j in range(max(nx, n_turns)):
                if j < nx:
                    b, i = buf(x, k)
                    yield ("SFull", b), i
                if j < n_turns:
                    t = tn if x else tn - 1
                    if t >= 0:
                        yield tok_wait, t
                    e.arrive(tok_pass)
                    tn += 1
                if j < nx:
                    if dual and j >= 1 and rng.random() < 0.5:  # O rescale waits for PV(k - 1)
                        pb, pi = buf(x, k - 1)
                        yield ("PVDone", pb), pi
                    e.arrive(p_full(x, k)[0])
                    k += 1
            if nx > 0:
                pb, pi = buf(x, k - 1)
                yield ("PVDone", pb), pi
            yield ("SchedFull", n & 1), n >> 1
            e.arrive(("SchedEmpty", n & 1))

    roles = {"producer": producer(), "issuer A": issuer(0), "issuer B": issuer(1)}
    for x in range(2):
        for w in range(4):
            roles[f"softmax {'AB'[x]}{w}"] = softmax(x, w)
    return roles


def _units(rng, kind):
    out = []
    for _ in range(rng.randint(1, 5)):
        p = rng.randint(0, 6)
        r = rng.random()
        if kind == "causal" or r < 0.4:
            out.append((2 * p + 1, 2 * p + 2))   # square causal pair: tile B sees one more K/V tile
        elif r < 0.6:
            out.append((p + 1, 0))               # tile B past the last row
        elif r < 0.7:
            out.append((0, p + 1))               # tile A sees no key (N_q > N_k alignment)
        elif r < 0.85:
            out.append((p + 1, p + 3))           # general causal offsets
        else:
            out.append((p + 1, p + 1))           # non-causal
    return out


def _run(units, seed, **kw):
    e = Engine(seed)
    return e.run(forward_roles(e, units, seed=seed, **kw))


@pytest.mark.parametrize("kind", ["causal", "mixed"])
def test_forward_protocol_has_no_deadlock_or_parity_aliasing(kind):
    for seed in range(400):
        units = _units(random.Random(seed), kind)
        result = _run(units, seed)
        assert result is None, f"seed {seed}, units {units}: {result}"


def test_model_catches_a_release_without_the_full_waits():
    # Releasing a skipped K/V tile without first taking its full phases lets
    # the issuer's next wait on that stage pass on an older load's parity.
    found = None
    for seed in range(3000):
        units = _units(random.Random(seed), "mixed")
        found = _run(units, seed, skip_full_waits=False)
        if found:
            break
    assert found and "parity wait passes early" in found


def test_decode_protocol_has_no_deadlock_or_parity_aliasing():
    # Decoding: every unit is (K/V tiles of its split, 0).
    for seed in range(400):
        rng = random.Random(seed)
        units = [(rng.randint(1, 9), 0) for _ in range(rng.randint(1, 5))]
        result = _run(units, seed, dual=True)
        assert result is None, f"seed {seed}, units {units}: {result}"


def test_model_catches_a_single_p_full_barrier_in_decode():
    # One P-full barrier per tile while S is double-buffered lets a fast
    # softmax warp arrive for P(j+1) before a slow one has arrived for P(j):
    # the phase completes with arrivals of two tiles, PV(j) and S(j+2) go
    # out early, and the slow warp ends up two phases behind.
    found = None
    for seed in range(2000):
        rng = random.Random(seed)
        units = [(rng.randint(2, 9), 0) for _ in range(rng.randint(1, 3))]
        e = Engine(seed)
        found = e.run(forward_roles(e, units, dual=True, seed=seed, one_p_full=True))
        if found:
            break
    assert found and "two phases" in found


def test_model_catches_turns_taken_by_one_tile_only():
    # Tile A taking turns for the K/V tiles only tile B visits (while B
    # takes turns only for the shared ones) puts the two token barriers out
    # of step: a waiter ends up two phases behind or waits forever.
    found = None
    for seed in range(2000):
        units = _units(random.Random(seed), "causal")
        found = _run(units, seed, phantom_turns_a=True)
        if found:
            break
    assert found
