"""A CPU model of a persistent kernel's mbarrier protocol, for the pipeline tests.

Each role of a kernel is a generator of the operations it performs on its barriers, in the
order the kernel performs them:
- ("wait", bar, parity, target): a parity wait that the kernel means to pass once `bar` has
  completed `target` phases (`wait_full`);
- ("arrive", bar, phase): an arrival meant for phase `phase` of `bar`;
- ("async", key, bar, phase): an arrival that completes later, as a copy or an MMA commit does;
  those with the same key (one thread's commits) complete in order, the others in any order.

`run` plays the roles under a random schedule in which each role gets a random speed, so that
some run far ahead of the others. A wait passes as the hardware lets it, when the barrier's
count of completed phases has the other parity; the model then records an error if the count is
not the one the wait means (a waiter that began a phase early and passed at once: phase
aliasing). It also records arrivals that land in another phase than the one they are meant for,
and schedules that stop with roles unfinished (deadlock)."""

import random


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.arrived, self.done = name, count, 0, 0

    def arrive(self, phase, errors):
        if phase != self.done:
            errors.append(f"{self.name}: arrival meant for phase {phase} landed in phase {self.done}")
        self.arrived += 1
        if self.arrived == self.count:
            self.arrived = 0
            self.done += 1


def ring(name, depth, count):
    return [Barrier(f"{name}{s}", count) for s in range(depth)]


def wait_full(bar, q):
    """Wait for phase q of `bar` to complete (parity q & 1; q = -1 passes at once)."""
    return ("wait", bar, q & 1, q + 1)


def run(gens, seed):
    rng = random.Random(seed)
    speed = [rng.choice((0.05, 0.3, 1.0, 3.0)) for _ in gens]
    ops = [next(g, None) for g in gens]
    fifo = {}
    loose = []
    errors = []
    while True:
        cand = []
        for i, op in enumerate(ops):
            if op is None:
                continue
            if op[0] != "wait" or (op[1].done & 1) != op[2]:
                cand.append(("role", i))
        cand += [("fifo", k) for k, v in fifo.items() if v]
        cand += [("loose", k) for k in range(len(loose))]
        if not cand:
            if any(op is not None for op in ops) or loose or any(fifo.values()):
                errors.append("deadlock")
            return errors
        weights = [speed[x[1]] if x[0] == "role" else 0.5 for x in cand]
        kind, i = rng.choices(cand, weights)[0]
        if kind == "fifo":
            bar, phase = fifo[i].pop(0)
            bar.arrive(phase, errors)
            continue
        if kind == "loose":
            bar, phase = loose.pop(i)
            bar.arrive(phase, errors)
            continue
        op = ops[i]
        if op[0] == "wait":
            _, bar, _, target = op
            if bar.done != target:
                errors.append(f"{bar.name}: a wait for completion {target} passed at {bar.done}")
        elif op[0] == "arrive":
            op[1].arrive(op[2], errors)
        else:
            _, key, bar, phase = op
            if key is None:
                loose.append((bar, phase))
            else:
                fifo.setdefault(key, []).append((bar, phase))
        ops[i] = next(gens[i], None)
