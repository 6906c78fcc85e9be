"""CPU model of the forward kernel's mbarrier protocol (no GPU).

`fa2_fwd_kernel` coordinates its roles (TMA producer, two MMA issuers, two
groups of four softmax warps) through mbarriers waited on by phase parity.
This model replays each role's sequence of waits, arrivals, TMA loads and
MMA commits (`protocol_model.Engine`: loads land in any order, one issuer's
MMAs and commits complete in issue order) and checks that no wait is ever
two phases away from its barrier and that every run ends.  Barrier names and
counts follow the kernel's FwdBar enum; a unit is the pair (K/V tiles of
query tile A, K/V tiles of query tile B) that `fwd_unit` computes.  K and V
tiles share one ring of three slots, loaded in the order K_0, (K_j, V_{j-1})
for j = 1 .. n-1, V_{n-1}.  The scheduler barriers (one response per unit,
read by all eleven roles) are included.  (The softmax warps of the two
tiles no longer take turns at the exponentials, so the model has no token
barriers.)

Besides the barrier phases, the model tracks the data the barriers protect
and reports a hazard when a protocol step would let one side overwrite what
the other still reads: a ring slot reloaded while an MMA reads it, S_x
computed again before every softmax warp has read the previous S_x, P_x
written while the P V MMA that reads the previous P_x may still run.
"""
import random

import pytest

from protocol_model import Engine

RING = 3


def ring_pos_k(j):
    return 0 if j == 0 else 2 * j - 1


def ring_pos_v(j, n):
    return 2 * j + 2 if j + 1 < n else 2 * n - 1


def forward_roles(e, units, planted=None):
    """Roles of one CTA.  ``planted`` names one deliberate protocol mistake
    (for the tests that check the model catches it)."""
    for s in range(2):
        for name, count in (("QFull", 1), ("QEmpty", 1), ("SFull", 1), ("SRead", 4), ("PFull", 4), ("PVDone", 1),
                            ("SchedFull", 1), ("SchedEmpty", 11)):
            e.bar((name, s), count, f"{name}[{s}]")
    for s in range(RING):
        e.bar(("KVFull", s), 1, f"KVFull[{s}]")
        e.bar(("KVEmpty", s), 2, f"KVEmpty[{s}]")

    reading = {sl: set() for sl in range(RING)}  # MMAs in flight that read a ring slot
    s_read = [[0] * 4 for _ in range(2)]  # S tiles each softmax warp has read, per tile
    pv_done = [0, 0]  # P V MMAs completed, per tile

    def hazard(msg):
        if e.error is None:
            e.error = "hazard: " + msg

    def load(key):
        e.unordered(lambda: e.arrive(key))

    def commit(x, *keys):
        for key in keys:
            e.ordered(("mma", x), lambda key=key: e.arrive(key))

    def mma_reads(x, slot, use, tag, pv=False):
        item = (use, x, tag)
        reading[slot].add(item)

        def done():
            reading[slot].discard(item)
            if pv:
                pv_done[x] += 1

        e.ordered(("mma", x), done)

    def producer():
        g, qn = 0, [0, 0]
        for n, (na, nb) in enumerate(units):
            n_kv = max(na, nb)

            def load_q(x):
                if qn[x] >= 1:
                    yield ("QEmpty", x), qn[x] - 1
                load(("QFull", x))
                qn[x] += 1

            def load_kv():
                nonlocal g
                slot, use = g % RING, g // RING
                if use >= 1:
                    yield ("KVEmpty", slot), use - 1
                if reading[slot]:
                    hazard(f"slot {slot} reloaded (use {use}) while MMAs read it: {sorted(reading[slot])}")
                load(("KVFull", slot))
                g += 1

            if n_kv > 0:
                if na > 0:
                    yield from load_q(0)
                yield from load_kv()
                if nb > 0:
                    yield from load_q(1)
                for _ in range(1, n_kv):
                    yield from load_kv()  # K_j
                    yield from load_kv()  # V_{j-1}
                yield from load_kv()  # V_{n-1}
            if n >= 2:
                yield ("SchedEmpty", n & 1), (n >> 1) - 1
            load(("SchedFull", n & 1))
            yield ("SchedFull", n & 1), n >> 1
            e.arrive(("SchedEmpty", n & 1))

    def issuer(x):
        g = k = qn = 0

        def full(pos):
            return ("KVFull", pos % RING), pos // RING

        def issue_s(pos, kk, last_q):
            if min(s_read[x]) < kk:
                hazard(f"S_{'AB'[x]} #{kk} computed before every warp read S #{kk - 1}")
            mma_reads(x, pos % RING, pos // RING, f"S{kk}")
            commit(x, ("SFull", x), ("KVEmpty", pos % RING), *([("QEmpty", x)] if last_q else []))

        for n, cnt in enumerate(units):
            n_kv, nx = max(cnt), cnt[x]
            if n_kv > 0:
                if nx > 0:
                    yield ("QFull", x), qn
                    qn += 1
                    if k >= 1:
                        yield ("SRead", x), k - 1
                    yield full(g)
                    issue_s(g, k, nx == 1)
                for j in range(nx):
                    if j + 1 < nx:
                        pk = g + ring_pos_k(j + 1)
                        if planted != "s_before_read":
                            yield ("SRead", x), k
                        yield full(pk)
                        issue_s(pk, k + 1, j + 2 == nx)
                    pv = g + ring_pos_v(j, n_kv)
                    yield full(pv)
                    yield ("PFull", x), k
                    mma_reads(x, pv % RING, pv // RING, f"PV{k}", pv=True)
                    commit(x, ("PVDone", x), ("KVEmpty", pv % RING))
                    k += 1
                # ring positions of the tiles this query tile does not visit
                start = g + (0 if nx == 0 else ring_pos_k(nx))
                for pos in range(start, g + 2 * n_kv):
                    rel = pos - g
                    if rel == 0:
                        mine = nx > 0
                    elif rel == 2 * n_kv - 1:
                        mine = nx == n_kv
                    elif rel & 1:
                        mine = (rel + 1) // 2 < nx
                    else:
                        mine = (rel - 2) // 2 < nx
                    if mine:
                        continue
                    slot, use = pos % RING, pos // RING
                    if planted != "release_without_full":
                        yield full(pos)
                    if use >= 1:
                        yield ("KVEmpty", slot), use - 1
                    e.arrive(("KVEmpty", slot))
                g += 2 * n_kv
            yield ("SchedFull", n & 1), n >> 1
            e.arrive(("SchedEmpty", n & 1))

    def softmax(x, w):
        k = 0
        for n, cnt in enumerate(units):
            nx = cnt[x]
            for j in range(nx):
                yield ("SFull", x), k
                s_read[x][w] += 1
                e.arrive(("SRead", x))
                if k >= 1 and planted != "p_before_pv_done":
                    yield ("PVDone", x), k - 1
                if pv_done[x] < k:
                    hazard(f"P_{'AB'[x]} #{k} written while P V #{k - 1} may still read P")
                e.arrive(("PFull", x))
                k += 1
            if nx > 0:
                yield ("PVDone", x), k - 1
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
        elif r < 0.55:
            out.append((p + 1, 0))               # tile B past the last row
        elif r < 0.65:
            out.append((0, p + 1))               # tile A sees no key (N_q > N_k alignment)
        elif r < 0.8:
            out.append((p + 1, p + 3))           # general causal offsets
        elif r < 0.9:
            out.append((p + 3, p + 1))           # tile A sees more (key splits)
        else:
            out.append((p + 1, p + 1))           # non-causal
    return out


def _run(units, seed, **kw):
    e = Engine(seed)
    return e.run(forward_roles(e, units, **kw))


@pytest.mark.parametrize("kind", ["causal", "mixed"])
def test_forward_protocol_has_no_deadlock_parity_aliasing_or_hazard(kind):
    for seed in range(400):
        units = _units(random.Random(seed), kind)
        result = _run(units, seed)
        assert result is None, f"seed {seed}, units {units}: {result}"


def test_decode_protocol_has_no_deadlock_parity_aliasing_or_hazard():
    # Decoding: every unit is (K/V tiles of its split, 0).
    for seed in range(300):
        rng = random.Random(seed)
        units = [(rng.randint(1, 9), 0) for _ in range(rng.randint(1, 5))]
        result = _run(units, seed)
        assert result is None, f"seed {seed}, units {units}: {result}"


def _first_failure(planted, kind="mixed", seeds=3000):
    for seed in range(seeds):
        found = _run(_units(random.Random(seed), kind), seed, planted=planted)
        if found:
            return found
    return None


def test_model_catches_a_release_without_the_full_wait():
    # Releasing a skipped K/V tile without first taking its full phase lets
    # the issuer's next wait on that slot pass on an older load's parity.
    found = _first_failure("release_without_full")
    assert found and "parity wait passes early" in found


def test_model_catches_s_computed_before_the_softmax_read_it():
    found = _first_failure("s_before_read")
    assert found and "computed before every warp read" in found


def test_model_catches_p_written_while_the_previous_p_v_may_run():
    found = _first_failure("p_before_pv_done")
    assert found and "may still read P" in found

