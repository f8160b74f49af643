"""Model check of the mbarrier protocols of the tcgen05 kernels (CPU).

An mbarrier completes a phase when its expected arrivals are in; a wait
names the parity of the phase it wants finished and passes while the
barrier's current phase has the other parity.  So a waiter that falls two
phases behind the barrier waits on a phase that has come round again and
never returns.  These tests run each kernel's roles (copy threads, MMA
threads, softmax or consumer warps, and the asynchronous completions of
bulk copies and MMA commits, which arrive in the issuing thread's order)
under many random interleavings and check that every wait is released by
the phase it names (never by a later one, never after the barrier has moved
two phases on) and that every run finishes.  The protocols are the
kernels' own; a variant of the prefill protocol with a single "P written"
barrier, which the per-buffer design replaced, must be caught aliasing.
"""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count = count
        self.pending = 0
        self.phase = 0  # completed phases

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.phase += 1


class Alias(Exception):
    pass


def wait(bar, k):
    """('wait', bar, k): block until phase k of bar has completed."""
    return ("wait", bar, k)


def run(actors, rng, max_steps=200000):
    """actors: dict name -> generator yielding ops; ops are
    ('wait', bar, k), ('arrive', bar), ('async', queue, bar) (an arrival on
    bar fired later by the named in-order completion queue).  Returns the
    number of steps; raises Alias or RuntimeError (deadlock)."""
    state = {n: [g, next(g, None)] for n, g in actors.items()}
    queues = {}
    for step in range(max_steps):
        ready = []
        for n, (g, op) in state.items():
            if op is None:
                continue
            if op[0] == "wait":
                bar, k = op[1], op[2]
                if bar.phase >= k + 2:
                    raise Alias(f"{n} waits for phase {k}, barrier already completed {bar.phase}")
                if bar.phase == k + 1:
                    ready.append(("actor", n))
            else:
                ready.append(("actor", n))
        ready += [("queue", q) for q, items in queues.items() if items]
        if not ready:
            if all(op is None for _, op in state.values()):
                return step
            raise RuntimeError("deadlock: " + ", ".join(f"{n}: {op[0]}" for n, (_, op) in state.items() if op))
        kind, name = rng.choice(ready)
        if kind == "queue":
            queues[name].pop(0).arrive()
            continue
        g, op = state[name]
        if op[0] == "arrive":
            op[1].arrive()
        elif op[0] == "async":
            queues.setdefault(op[1], []).append(op[2])
        state[name][1] = next(g, None)
    raise RuntimeError("step limit")


# ---------------------------------------------------------------------------
# prefill_kernel: key ring (3 stages), value ring (2), S single-buffered in
# TMEM, P double-buffered with one "P written" and one "P.V done" barrier
# per buffer; a softmax warp that rescales O waits for the previous tile's
# P.V, else for the one two tiles back.

def prefill_actors(nt, warps, rng, per_buffer=True, ks=3, vs=2):
    kfull = [Barrier(1) for _ in range(ks)]
    kempty = [Barrier(1) for _ in range(ks)]
    vfull = [Barrier(1) for _ in range(vs)]
    vempty = [Barrier(1) for _ in range(vs)]
    sfull, sfree = Barrier(1), Barrier(warps)
    pfull = [Barrier(warps), Barrier(warps)] if per_buffer else [Barrier(warps)]
    pvdone = [Barrier(1), Barrier(1)]

    def pf(i):  # (barrier, phase) of "P of tile i written"
        return (pfull[i & 1], i >> 1) if per_buffer else (pfull[0], i)

    def copier(full, empty, stages, tag):
        for j in range(nt):
            s = j % stages
            if j >= stages:
                yield wait(empty[s], j // stages - 1)
            yield ("async", tag, full[s])

    def qk():
        for j in range(nt):
            yield wait(kfull[j % ks], j // ks)
            if j >= 1:
                yield wait(sfree, j - 1)
            yield ("async", "mma_qk", sfull)
            yield ("async", "mma_qk", kempty[j % ks])

    def pv():
        for i in range(nt):
            yield wait(vfull[i % vs], i // vs)
            b, k = pf(i)
            yield wait(b, k)
            yield ("async", "mma_pv", pvdone[i & 1])
            yield ("async", "mma_pv", vempty[i % vs])

    def softmax(w):
        r = random.Random(rng.random())
        for j in range(nt):
            yield wait(sfull, j)
            yield ("arrive", sfree)
            resc = j > 0 and r.random() < 0.3
            if per_buffer:
                if resc or j > 1:
                    jw = j - 1 if resc else j - 2
                    yield wait(pvdone[jw & 1], jw >> 1)
            elif j > 1:  # the single-barrier variant with the same waits
                jw = j - 1 if resc else j - 2
                yield wait(pvdone[jw & 1], jw >> 1)
            b, _ = pf(j)
            yield ("arrive", b)
        if nt:
            yield wait(pvdone[(nt - 1) & 1], (nt - 1) >> 1)

    actors = {"kcopy": copier(kfull, kempty, ks, "tma_k"), "vcopy": copier(vfull, vempty, vs, "tma_v"),
              "qk": qk(), "pv": pv()}
    for w in range(warps):
        actors[f"softmax{w}"] = softmax(w)
    return actors


@pytest.mark.parametrize("nt", [0, 1, 2, 3, 5, 9])
def test_prefill_protocol_never_aliases(nt):
    for seed in range(300):
        rng = random.Random(seed)
        run(prefill_actors(nt, warps=3, rng=rng), rng)


def test_prefill_single_p_barrier_aliases():
    """With one "P written" barrier, softmax warps that no longer wait for
    the previous tile's P.V can finish two of its phases before the P.V
    thread looks: the checker must find it."""
    found = 0
    for seed in range(300):
        rng = random.Random(seed)
        try:
            run(prefill_actors(9, warps=2, rng=rng, per_buffer=False), rng)
        except Alias:
            found += 1
    assert found > 0


# ---------------------------------------------------------------------------
# mass_stats_kernel / mass_colsum_kernel: the query by TMA (one barrier),
# a 4-stage key ring, two TMEM buffers released by every consumer thread.

def mass_actors(n, consumers, stages=4, q_tma=True):
    kfull = [Barrier(1) for _ in range(stages)]
    kempty = [Barrier(1) for _ in range(stages)]
    dfull = [Barrier(1), Barrier(1)]
    dfree = [Barrier(consumers), Barrier(consumers)]
    qfull = Barrier(1)

    def loader():
        if q_tma and n > 0:
            yield ("async", "tma", qfull)
        for i in range(n):
            s = i % stages
            if i >= stages:
                yield wait(kempty[s], i // stages - 1)
            yield ("async", "tma", kfull[s])
        if q_tma and n > 0:
            yield wait(qfull, 0)

    def mma():
        if q_tma and n > 0:
            yield wait(qfull, 0)
        for i in range(n):
            yield wait(kfull[i % stages], i // stages)
            if i >= 2:
                yield wait(dfree[i & 1], (i >> 1) - 1)
            yield ("async", "mma", dfull[i & 1])
            yield ("async", "mma", kempty[i % stages])

    def consumer():
        for i in range(n):
            yield wait(dfull[i & 1], i >> 1)
            yield ("arrive", dfree[i & 1])

    actors = {"loader": loader(), "mma": mma()}
    for c in range(consumers):
        actors[f"consumer{c}"] = consumer()
    return actors


@pytest.mark.parametrize("q_tma", [True, False])
@pytest.mark.parametrize("n", [0, 1, 2, 4, 7, 13])
def test_mass_protocol_never_aliases(n, q_tma):
    for seed in range(200):
        rng = random.Random(seed)
        run(mass_actors(n, consumers=3, q_tma=q_tma), rng)
