"""Randomised model of the routed-rows colwise kernel's ring and unit queue.

The kernel (csrc/colwise_jagged.cu) has one producer thread that takes units
in order, publishes each in a 32-entry shared-memory queue (entry, first
fill) and issues its boxes into a 12-slot ring, and consumer groups that take
queue entries in rotation (group g: entries g, g + G, ...).  A unit of at
most 12 boxes is waited on box by box, then released box by box after its
cast; a longer one is streamed twice (its first pass released right after
the maxima, its second pass waited on and released by the cast).  mbarriers
know phases only by parity, so a waiter that is a whole phase behind would
pass at once: consumers first wait until the producer has published that it
issued the fill they want (the "issued" gate).

This model runs the protocol's steps in random interleavings (copies of
different slots landing in any order) and checks at every parity wait that
the barrier is not a whole phase behind, that no queue entry is overwritten
before its group took it, and that every run ends with all units consumed.
It also checks that without the issued gate the same interleavings do alias,
which is what the gate is for.
"""
import random

import pytest

NS, UQ = 12, 32   # ring slots, queue entries (as in the kernel)


def run(nboxes, groups, seed, gate=True):
    rnd = random.Random(seed)
    U = len(nboxes)
    # producer: room for entry n, publish it, then its fills (two passes when long)
    prod, f0s, f = [], [], 0
    for n, nb in enumerate(nboxes):
        prod += [("room", n), ("pub", n)]
        f0s.append(f)
        for _ in range(nb if nb <= NS else 2 * nb):
            prod.append(("fill", f))
            f += 1
    for e in range(groups):           # one end entry per group
        prod += [("room", U + e), ("pub", U + e)]
    progs = {g: [] for g in range(groups)}
    for n, nb in enumerate(nboxes):
        res, f0, ops = nb <= NS, f0s[n], [("take", n)]
        for b in range(nb):
            ops.append(("wait", f0 + b))
            if not res:
                ops.append(("rel", f0 + b))
        for b in range(nb):
            fb = f0 + b if res else f0 + nb + b
            if not res:
                ops.append(("wait", fb))
            ops.append(("rel", fb))
        progs[n % groups] += ops
    for e in range(groups):
        progs[(U + e) % groups].append(("take", U + e))
    full_c, empty_c = [0] * NS, [0] * NS
    inflight, issued, nq, read = [], 0, 0, [0] * groups
    qent = [None] * UQ
    pp, pc = 0, [0] * groups
    for _ in range(10 ** 6):
        acts = []
        if pp < len(prod):
            op, x = prod[pp]
            if op == "room":
                if x < UQ or read[(x - UQ) % groups] > x - UQ:
                    acts.append(("p",))
            elif op == "pub":
                acts.append(("p",))
            else:
                s, ph = x % NS, x // NS - 1
                if x < NS or empty_c[s] > ph:
                    acts.append(("p",))
                elif empty_c[s] % 2 != ph % 2:
                    return "producer alias"
        if inflight:
            acts.append(("tma",))
        for g in range(groups):
            if pc[g] == len(progs[g]):
                continue
            op, x = progs[g][pc[g]]
            if op == "rel":
                acts.append(("c", g))
            elif op == "take":
                if nq > x:
                    acts.append(("c", g))
            else:
                s, ph = x % NS, x // NS
                if gate and issued <= x:
                    continue
                if full_c[s] > ph:
                    acts.append(("c", g))
                elif full_c[s] % 2 != ph % 2:
                    return "consumer alias"
        if not acts:
            done = pp == len(prod) and not inflight and all(pc[g] == len(progs[g]) for g in range(groups))
            return "ok" if done else "deadlock"
        a = rnd.choice(acts)
        if a[0] == "p":
            op, x = prod[pp]
            if op == "pub":
                if qent[x % UQ] is not None and not qent[x % UQ][1]:
                    return "queue overwrite"
                qent[x % UQ] = [x, False]
                nq = x + 1
            elif op == "fill":
                inflight.append(x)
                issued = x + 1
            pp += 1
        elif a[0] == "tma":
            full_c[inflight.pop(rnd.randrange(len(inflight))) % NS] += 1
        else:
            g = a[1]
            op, x = progs[g][pc[g]]
            if op == "rel":
                empty_c[x % NS] += 1
            elif op == "take":
                if qent[x % UQ] is None or qent[x % UQ][0] != x:
                    return "wrong entry"
                qent[x % UQ][1] = True
                read[g] = x + 1
            pc[g] += 1
    return "stuck"


def _cases():
    rng = random.Random(7)
    cases = [[55, 3, 12, 13, 1, 6, 2, 40, 7, 9, 12, 12, 5], [5], [], [0, 0, 3, 0, 0, 0, 1], [13, 14]]
    for _ in range(3):
        cases.append([rng.choice([0, 1, 2, 3, 6, 12, 13, 20, 55]) for _ in range(rng.randint(35, 60))])
    return cases


@pytest.mark.parametrize("groups", [2, 3])
def test_ring_and_queue_never_alias_or_deadlock(groups):
    for nb in _cases():
        for seed in range(12):
            assert run(nb, groups, seed) == "ok", (groups, nb, seed)


def test_without_the_issued_gate_the_ring_aliases():
    # full-ring units alternating between the groups: one group can fall a
    # whole phase behind on a slot the other keeps refilling
    bad = [run([12] * 20, 2, seed, gate=False) for seed in range(40)]
    assert any(r == "consumer alias" for r in bad)
    assert all(run([12] * 20, 2, seed) == "ok" for seed in range(40))
