"""Discrete-event model of the attention kernel's mbarrier protocol (host
logic only; no attention arithmetic).

Roles, as in the kernel: the TMA producer, the QK^T issuer, the softmax warps
(one actor) and the P.V issuer.  TMA loads land after random delays, in any
order; the MMAs of one issuer complete in order after random delays, and a
tcgen05.commit arrival fires when every earlier MMA of its issuer completed.
A wait follows the hardware rule for a parity wait, passing iff the parity
of the number of completed phases differs from the one asked for, and the
model checks it against the phase the waiter means: a wait that passes on an
older phase of the same parity (aliasing) or a deadlock fails the run, as
does an issuer reading a ring slot that does not hold the tile it wants.

K/V ring: position pos holds K (pos even) or V (pos odd) in slot pos % slots.
``per_kind`` selects one full barrier per (slot, kind), waited on with the
use index of the fill among the fills of its kind in its slot; otherwise one
full barrier per slot, waited on with pos // slots.
"""

import random


class Bar:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.completed = 0
        self.arrived = 0
        self.tx = 0

    def arrive(self, tx=0):
        if self.arrived >= self.count:
            raise AssertionError(f"{self.name}: arrival past count in phase {self.completed}")
        self.arrived += 1
        self.tx += tx
        self._check()

    def complete_tx(self, tx):
        self.tx -= tx
        if self.tx < 0:
            raise AssertionError(f"{self.name}: tx underflow")
        self._check()

    def _check(self):
        if self.arrived == self.count and self.tx == 0:
            self.completed += 1
            self.arrived = 0

    def try_wait(self, parity, meant):
        ok = (self.completed & 1) != parity
        if ok and self.completed <= meant:
            raise AssertionError(f"{self.name}: parity wait for phase {meant} passed with only "
                                 f"{self.completed} phases complete (aliasing)")
        return ok


def run(units, slots, per_kind, seed, rescale_p=0.3):
    rng = random.Random(seed)
    B = {}

    def bar(name, count=1):
        if name not in B:
            B[name] = Bar(name, count)
        return B[name]

    for b in (0, 1):
        bar(f"s_full{b}"); bar(f"s_free{b}"); bar(f"p_full{b}"); bar(f"p_free{b}")
    bar("q_full"); bar("q_empty"); bar("o_full")

    def full_bar(pos):
        slot = pos % slots
        if per_kind:
            return bar(f"{'v' if pos & 1 else 'k'}_full{slot}")
        return bar(f"kv_full{slot}")

    def full_use(pos):
        if per_kind:
            return ((pos // slots) >> 1) if (slots & 1) else pos // slots
        return pos // slots

    slot_data = {}      # slot -> ring position whose data is in it (None while a load is in flight)
    events = []         # (time, seq, fn)
    now = [0.0]
    seq = [0]

    def later(delay, fn):
        seq[0] += 1
        events.append((now[0] + delay, seq[0], fn))

    mma_tail = {"qk": 0.0, "pv": 0.0}

    def mma(issuer, check, commits):
        t = max(now[0], mma_tail[issuer]) + rng.uniform(0.1, 2.0)
        mma_tail[issuer] = t

        def done():
            check()
            for c in commits:
                c.arrive()
        seq[0] += 1
        events.append((t, seq[0], done))

    def producer():
        ring = qcount = 0
        for n in units:
            yield lambda: bar("q_empty").try_wait((qcount & 1) ^ 1, qcount - 1)
            bar("q_full").arrive(tx=1)
            later(rng.expovariate(1.0), lambda: bar("q_full").complete_tx(1))
            qcount += 1
            for j in range(n):
                for sel in (0, 1):
                    slot, use = ring % slots, ring // slots
                    yield lambda: bar(f"kv_empty{slot}").try_wait((use & 1) ^ 1, use - 1)
                    f = full_bar(ring)
                    f.arrive(tx=1)
                    slot_data[slot] = None
                    pos = ring

                    def land(slot=slot, pos=pos, f=f):
                        slot_data[slot] = pos
                        f.complete_tx(1)
                    later(rng.expovariate(0.5) if rng.random() < 0.9 else rng.uniform(5, 30), land)
                    ring += 1

    def qk():
        ring = qcount = tcount = 0
        for n in units:
            yield lambda: bar("q_full").try_wait(qcount & 1, qcount)
            qcount += 1
            for j in range(n):
                b, use = tcount & 1, tcount >> 1
                if tcount >= 2:
                    yield lambda: bar(f"s_free{b}").try_wait((use - 1) & 1, use - 1)
                pos = ring + 2 * j
                slot = pos % slots
                yield lambda: full_bar(pos).try_wait(full_use(pos) & 1, full_use(pos))
                assert slot_data.get(slot) == pos, f"QK read slot {slot}: has {slot_data.get(slot)}, wants {pos}"

                def chk(slot=slot, pos=pos):
                    assert slot_data.get(slot) == pos, f"K slot {slot} overwritten under the MMA"
                mma("qk", chk, [bar(f"s_full{b}"), bar(f"kv_empty{slot}")])
                tcount += 1
            ring += 2 * n
            mma("qk", lambda: None, [bar("q_empty")])

    def softmax():
        tcount = ocount = 0
        for n in units:
            for j in range(n):
                b, use = tcount & 1, tcount >> 1
                yield lambda: bar(f"s_full{b}").try_wait(use & 1, use)
                bar(f"s_free{b}").arrive()
                if tcount >= 2:
                    yield lambda: bar(f"p_free{b}").try_wait((use - 1) & 1, use - 1)
                if j > 0 and rng.random() < rescale_p:
                    tp = tcount - 1
                    yield lambda: bar(f"p_free{tp & 1}").try_wait((tp >> 1) & 1, tp >> 1)
                bar(f"p_full{b}").arrive()
                tcount += 1
            yield lambda: bar("o_full").try_wait(ocount & 1, ocount)
            ocount += 1

    def pv():
        ring = tcount = 0
        for n in units:
            for j in range(n):
                b, use = tcount & 1, tcount >> 1
                yield lambda: bar(f"p_full{b}").try_wait(use & 1, use)
                pos = ring + 2 * j + 1
                slot = pos % slots
                yield lambda: full_bar(pos).try_wait(full_use(pos) & 1, full_use(pos))
                assert slot_data.get(slot) == pos, f"PV read slot {slot}: has {slot_data.get(slot)}, wants {pos}"

                def chk(slot=slot, pos=pos):
                    assert slot_data.get(slot) == pos, f"V slot {slot} overwritten under the MMA"
                commits = [bar(f"p_free{b}"), bar(f"kv_empty{slot}")]
                if j == n - 1:
                    commits.append(bar("o_full"))
                mma("pv", chk, commits)
                tcount += 1
            ring += 2 * n

    for s in range(slots):
        bar(f"kv_empty{s}")
        if per_kind:
            bar(f"k_full{s}"); bar(f"v_full{s}")
        else:
            bar(f"kv_full{s}")
    actors = {"prod": producer(), "qk": qk(), "sm": softmax(), "pv": pv()}
    waiting = {k: next(g, None) for k, g in actors.items()}
    while True:
        ready = [k for k, w in waiting.items() if w is not None and w()]
        if ready:
            k = rng.choice(ready)
            waiting[k] = next(actors[k], None)
            continue
        if all(w is None for w in waiting.values()) and not events:
            return
        if not events:
            raise AssertionError(f"deadlock: {[k for k, w in waiting.items() if w is not None]}")
        events.sort()
        t, _, fn = events.pop(0)
        now[0] = t
        fn()


