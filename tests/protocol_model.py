"""mbarrier and scheduler model shared by the CPU protocol tests of the persistent kernels.

An mbarrier has an arrival count, pending arrivals, a transaction count and a phase; a wait
on parity p is satisfied once the phase of parity p has completed (at once on a fresh
barrier for p = 1), as PTX's mbarrier.try_wait.parity.  Agents are generators that yield
(barrier, parity) to wait; asynchronous copies are events that complete in any order, and
ordered queues hold completions that land in issue order (one CTA's MMAs)."""
import random


class Violation(Exception):
    pass


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.tx, self.phase = count, count, 0, 0

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def arrive(self):
        if self.pending == 0:  # the phase still waits for bytes: the count would underflow
            raise Violation("arrival beyond the barrier's count")
        self.pending -= 1
        self._check()

    def expect_tx(self, n):  # mbarrier.arrive.expect_tx
        self.tx += n
        self.arrive()

    def complete_tx(self, n):
        self.tx -= n
        self._check()

    def ready(self, parity):
        return (self.phase & 1) != parity


def run(agents, events, queues, seed):
    """Run the agents under a random schedule until all have finished; events (callables)
    fire in any order, the head of each queue in `queues` in order.  Raises Violation on a
    deadlock.  Returns the number of steps."""
    rnd = random.Random(seed)
    waits = [None] * len(agents)
    alive = [True] * len(agents)
    steps = 0
    while True:
        steps += 1
        cands = [("a", k) for k in range(len(agents))
                 if alive[k] and (waits[k] is None or waits[k][0].ready(waits[k][1]))]
        cands += [("e", k) for k in range(len(events))]
        cands += [("q", k) for k in range(len(queues)) if queues[k]]
        if not cands:
            if any(alive) or events:
                raise Violation("deadlock")
            return steps
        kind, k = rnd.choice(cands)
        if kind == "e":
            events.pop(k)()
        elif kind == "q":
            queues[k].pop(0)()
        else:
            try:
                waits[k] = next(agents[k])
            except StopIteration:
                alive[k] = False
                waits[k] = None
