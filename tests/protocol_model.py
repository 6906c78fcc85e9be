"""A small engine for CPU models of the kernels' mbarrier protocols.

Roles are Python generators that yield what they wait for:

* ``(key, t)``: completion number t (0-based) of the mbarrier ``key``, waited
  on by phase parity, as the kernels do;
* ``("cond", fn, text)``: any other condition (``fn()`` true), e.g. a bulk
  async-group wait.

Between waits a role arrives on barriers and enqueues asynchronous work:
``engine.ordered(q, fn)`` appends to queue q, whose items complete in order
(the MMAs and commits of one issuing thread); ``engine.unordered(fn)`` adds
an item that may complete at any time (a TMA load landing).  The run picks
one possible step at random until every role has finished.

On every wait the engine checks the parity hazard both ways: a barrier two
phases past the waited completion (the waiter would block forever) and a
barrier still two phases short of it (the parity test would pass on an
older phase).  Either, or a state where nothing can move, ends the run with
a message.
"""
import random


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.done = name, count, 0, 0

    def arrive(self):
        self.pending += 1
        assert self.pending <= self.count, f"{self.name}: more arrivals than its count"
        if self.pending == self.count:
            self.pending, self.done = 0, self.done + 1


class Engine:
    def __init__(self, seed):
        self.rng = random.Random(seed)
        self.bars = {}
        self.queues = {}
        self.loose = []
        self.error = None

    def bar(self, key, count, name=None):
        self.bars[key] = Bar(name or str(key), count)

    def arrive(self, key):
        self.bars[key].arrive()

    def ordered(self, queue, fn):
        self.queues.setdefault(queue, []).append(fn)

    def unordered(self, fn):
        self.loose.append(fn)

    def _ready(self, wait):
        if wait[0] == "cond":
            return wait[1]()
        key, t = wait
        b = self.bars[key]
        if b.done >= t + 2:
            self.error = f"{b.name}: waiter two phases behind (done {b.done}, waits #{t})"
        elif b.done <= t - 1 and (t - b.done) % 2 == 1:
            self.error = f"{b.name}: parity wait passes early (done {b.done}, waits #{t})"
        return b.done >= t + 1

    def _describe(self, wait):
        if wait[0] == "cond":
            return wait[2]
        return f"{self.bars[wait[0]].name} #{wait[1]}"

    def run(self, roles, max_steps=1_000_000):
        waiting = dict.fromkeys(roles)
        for _ in range(max_steps):
            moves = [("role", r) for r, w in waiting.items() if w is None or self._ready(w)]
            moves += [("queue", q) for q, items in self.queues.items() if items]
            moves += [("loose", None)] if self.loose else []
            if self.error:
                return self.error
            if not moves:
                if not waiting:
                    return None
                return "deadlock: " + "; ".join(f"{r} waits {self._describe(w)}" for r, w in waiting.items() if w)
            kind, who = self.rng.choice(moves)
            if kind == "queue":
                self.queues[who].pop(0)()
            elif kind == "loose":
                self.loose.pop(self.rng.randrange(len(self.loose)))()
            else:
                waiting[who] = None
                try:
                    while True:
                        w = next(roles[who])
                        if not self._ready(w):
                            waiting[who] = w
                            break
                        if self.error:
                            return self.error
                except StopIteration:
                    del waiting[who]
                    del roles[who]
        return "step limit"
