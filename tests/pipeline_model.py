"""Discrete-event model of the attention kernel's mbarrier protocol (host
logic only; no attention arithmetic).

Roles, as in the kernel: the TMA producer, the QK^T issuer, the softmax warps
(one actor) and the P.V issuer; the QK^T issuer starts a unit's products only
once the P.V issuer has issued the last product of the unit before.  Tensor memory as in the kernel, in both of
its protocols: (bf16) two S buffers released by the softmax once read, two
P buffers, one O buffer; (E4M3) two S buffers with P_b written over S_b and
released by the P V commit, and two O buffers that consecutive units
alternate between.  The model checks that no S or P buffer is overwritten
before it has been consumed, that P V reads the P of its own tile, that a
rescale or an epilogue sees O holding exactly the products issued so far,
and that an O buffer is reused only after its epilogue.  TMA loads land after random delays, in any
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


def run(units, slots, per_kind, seed, rescale_p=0.3, mistake=None, p_in_s=False, rings=None):
    """``p_in_s`` selects the E4M3 kernel's protocol (P written over S, two O
    buffers, S released by the P V commit) instead of the bf16 kernel's
    (separate P buffers, S released by the softmax, one O buffer).
    ``rings`` = (slots_k, slots_v) selects the kernel's ring layout: K_t in
    slot t % slots_k, V_t in slot slots_k + t % slots_v, one full and one empty
    barrier per slot, and two producers (Q and K; V), each filling its ring in
    order (``slots`` and ``per_kind`` are then unused); without it the single
    ring of positions described above, filled by one producer.
    ``mistake`` plants one protocol error, for the tests that show the model
    catches it: "qk_skips_buffer_wait", "pv_skips_o_free",
    "rescale_skips_p_free", "p_store_skips_p_free", "producer_skips_kv_empty"."""
    rng = random.Random(seed)
    B = {}

    def bar(name, count=1):
        if name not in B:
            B[name] = Bar(name, count)
        return B[name]

    for b in (0, 1):
        bar(f"s_full{b}"); bar(f"s_free{b}"); bar(f"p_full{b}"); bar(f"p_free{b}"); bar(f"o_full{b}")
        bar(f"o_free{b}")
    bar("q_full"); bar("q_empty"); bar("pv_issued")

    def slot_of(pos):
        if rings:
            t, sel = pos >> 1, pos & 1
            return rings[0] + t % rings[1] if sel else t % rings[0]
        return pos % slots

    def empty_use(pos):   # fills of the slot before this one
        if rings:
            t, sel = pos >> 1, pos & 1
            return t // rings[sel]
        return pos // slots

    def full_bar(pos):
        slot = slot_of(pos)
        if per_kind and not rings:
            return bar(f"{'v' if pos & 1 else 'k'}_full{slot}")
        return bar(f"kv_full{slot}")

    def full_use(pos):
        if rings:
            return empty_use(pos)
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

    def producer(kinds=(0, 1)):
        # kinds: (0, 1) one producer for Q, K and V in order; (0,) the split
        # layout's producer of Q and the K ring; (1,) its producer of the V ring
        ring = qcount = 0
        for n in units:
            if 0 in kinds:
                yield lambda: bar("q_empty").try_wait((qcount & 1) ^ 1, qcount - 1)
                bar("q_full").arrive(tx=1)
                later(rng.expovariate(1.0), lambda: bar("q_full").complete_tx(1))
                qcount += 1
            for j in range(n):
                for sel in (0, 1):
                    if sel not in kinds:
                        ring += 1
                        continue
                    slot, use = slot_of(ring), empty_use(ring)
                    if mistake != "producer_skips_kv_empty":
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

    # TMEM state.  S_b: ("S", t) after QK_t, then ("S", t, "read") once the
    # softmax has read it (separate-P protocol) or ("P", t) once P_t is written
    # over it (P-over-S protocol), ("P", t, "done") after P V_t.  P_b (separate
    # P buffers): ("P", t), then ("P", t, "done").  O buffers: ("busy", unit,
    # last tile issued) or ("free", unit whose epilogue read it).
    tmem_s = {0: None, 1: None}
    tmem_p = {0: None, 1: None}
    n_obuf = 2 if p_in_s else 1
    o_state = {0: ("free", -2 if p_in_s else -1), 1: ("free", -1)}

    def qk():
        ring = qcount = tcount = 0
        for n in units:
            yield lambda: bar("q_full").try_wait(qcount & 1, qcount)
            if qcount > 0:   # the unit before has issued its last P V
                yield lambda: bar("pv_issued").try_wait((qcount - 1) & 1, qcount - 1)
            qcount += 1
            for j in range(n):
                b, use = tcount & 1, tcount >> 1
                if tcount >= 2 and mistake != "qk_skips_buffer_wait":
                    if p_in_s:   # the P V of tile tcount-2 has consumed P_b, which overlays S_b
                        yield lambda: bar(f"p_free{b}").try_wait((use - 1) & 1, use - 1)
                    else:        # the softmax has read S of tile tcount-2
                        yield lambda: bar(f"s_free{b}").try_wait((use - 1) & 1, use - 1)
                pos = ring + 2 * j
                slot = slot_of(pos)
                yield lambda: full_bar(pos).try_wait(full_use(pos) & 1, full_use(pos))
                assert slot_data.get(slot) == pos, f"QK read slot {slot}: has {slot_data.get(slot)}, wants {pos}"
                st = tmem_s[b]
                ok_prev = ("P", tcount - 2, "done") if p_in_s else ("S", tcount - 2, "read")
                assert st is None or st == ok_prev, f"S{b} overwritten while holding {st}"

                def chk(slot=slot, pos=pos, b=b, t=tcount):
                    assert slot_data.get(slot) == pos, f"K slot {slot} overwritten under the MMA"
                    tmem_s[b] = ("S", t)
                mma("qk", chk, [bar(f"s_full{b}"), bar(f"kv_empty{slot}")])
                tcount += 1
            ring += 2 * n
            mma("qk", lambda: None, [bar("q_empty")])

    def softmax():
        tcount = ocount = 0
        for n in units:
            ob = ocount % n_obuf
            for j in range(n):
                b, use = tcount & 1, tcount >> 1
                yield lambda: bar(f"s_full{b}").try_wait(use & 1, use)
                assert tmem_s[b] == ("S", tcount), f"softmax read S{b} holding {tmem_s[b]}, wants tile {tcount}"
                if not p_in_s:
                    tmem_s[b] = ("S", tcount, "read")
                    bar(f"s_free{b}").arrive()
                    if tcount >= 2 and mistake != "p_store_skips_p_free":   # P_b consumed by P V tcount-2
                        yield lambda: bar(f"p_free{b}").try_wait((use - 1) & 1, use - 1)
                if j > 0 and rng.random() < rescale_p:   # O (this unit's buffer) is rescaled in place
                    tp = tcount - 1
                    if mistake != "rescale_skips_p_free":
                        yield lambda: bar(f"p_free{tp & 1}").try_wait((tp >> 1) & 1, tp >> 1)
                    assert o_state[ob] == ("busy", ocount, tp), f"rescale of O{ob} while {o_state[ob]}"
                if p_in_s:
                    tmem_s[b] = ("P", tcount)
                else:
                    pb = tmem_p[b]
                    assert pb is None or pb == ("P", tcount - 2, "done"), f"P{b} overwritten while holding {pb}"
                    tmem_p[b] = ("P", tcount)
                bar(f"p_full{b}").arrive()
                tcount += 1
            phase = ocount // n_obuf
            yield lambda: bar(f"o_full{ob}").try_wait(phase & 1, phase)
            assert o_state[ob] == ("busy", ocount, tcount - 1), f"epilogue read O{ob} while {o_state[ob]}"
            o_state[ob] = ("free", ocount)
            if p_in_s:
                bar(f"o_free{ob}").arrive()
            ocount += 1

    def pv():
        ring = tcount = ucount = 0
        for n in units:
            ob = ucount % n_obuf
            for j in range(n):
                b, use = tcount & 1, tcount >> 1
                yield lambda: bar(f"p_full{b}").try_wait(use & 1, use)
                if p_in_s and j == 0 and ucount >= 2 and mistake != "pv_skips_o_free":
                    yield lambda: bar(f"o_free{ob}").try_wait(((ucount >> 1) - 1) & 1, (ucount >> 1) - 1)
                if j == 0:
                    assert o_state[ob] == ("free", ucount - n_obuf), f"O{ob} reused while {o_state[ob]}"
                pos = ring + 2 * j + 1
                slot = slot_of(pos)
                yield lambda: full_bar(pos).try_wait(full_use(pos) & 1, full_use(pos))
                assert slot_data.get(slot) == pos, f"PV read slot {slot}: has {slot_data.get(slot)}, wants {pos}"

                def chk(slot=slot, pos=pos, b=b, t=tcount, u=ucount, ob=ob):
                    assert slot_data.get(slot) == pos, f"V slot {slot} overwritten under the MMA"
                    buf = tmem_s if p_in_s else tmem_p
                    assert buf[b] == ("P", t), f"PV read P{b} holding {buf[b]}, wants tile {t}"
                    buf[b] = ("P", t, "done")
                    o_state[ob] = ("busy", u, t)
                commits = [bar(f"p_free{b}"), bar(f"kv_empty{slot}")]
                if j == n - 1:
                    commits.append(bar(f"o_full{ob}"))
                mma("pv", chk, commits)
                if j == n - 1:
                    bar("pv_issued").arrive()   # a plain arrive right after the issue
                tcount += 1
            ring += 2 * n
            ucount += 1

    for s in range(sum(rings) if rings else slots):
        bar(f"kv_empty{s}")
        if rings:
            bar(f"kv_full{s}")
        elif per_kind:
            bar(f"k_full{s}"); bar(f"v_full{s}")
        else:
            bar(f"kv_full{s}")
    actors = {"qk": qk(), "sm": softmax(), "pv": pv()}
    if rings:
        actors["prod_k"], actors["prod_v"] = producer((0,)), producer((1,))
    else:
        actors["prod"] = producer()
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




def run_pair(units, slots, seed, mistake=None):
    """The barrier protocol of the padded forward with two query tiles per
    unit (attn_fwd_pair_kernel).  ``units`` is a list of (n_A, n_B): the K
    tiles each query tile processes (a unit loads max(n_A, n_B) K/V tiles;
    tile x takes part in K tile j iff j < n_x).  One ring of alternating K
    and V positions with one full barrier per (slot, kind); S_x written by
    the QK^T issuer after the P V of the previous S_x completed (P_x is
    written over S_x); the softmax of x reads S_x, writes P_x and, after the
    unit's last tile, reads O_x, which the next unit's first P V of x
    overwrites only after the softmax's p_full for it.  The P V issuer issues
    P_B V_j only after S_A of tile j + 1 has been issued (when tile A has
    one).  ``mistake``:
    "qk_skips_p_free", "producer_skips_kv_empty", "pv_skips_p_full"."""
    rng = random.Random(seed)
    B = {}

    def bar(name, count=1):
        if name not in B:
            B[name] = Bar(name, count)
        return B[name]

    for x in (0, 1):
        bar(f"s_full{x}"); bar(f"p_free{x}"); bar(f"o_full{x}"); bar(f"p_full{x}")
    bar("q_full"); bar("q_empty"); bar("qk_issued_a")
    for s in range(slots):
        bar(f"k_full{s}"); bar(f"v_full{s}"); bar(f"kv_empty{s}")

    def fill(pos):   # slot, full-barrier use, empty-barrier use of ring position pos
        return pos % slots, ((pos // slots) >> 1) if (slots & 1) else pos // slots, pos // slots

    slot_data = {}
    events = []
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

    # TMEM: s[x] = ("S", x, k) after QK_x #k, ("P", x, k) once the softmax
    # wrote P over it, ("P", x, k, "done") after its P V; o[x] = (unit, products)
    s_state = {0: None, 1: None}
    o_state = {0: None, 1: None}

    def producer():
        pos = qcount = 0
        for nA, nB in units:
            n = max(nA, nB)
            if n == 0:
                continue
            yield lambda: bar("q_empty").try_wait((qcount & 1) ^ 1, qcount - 1)
            bar("q_full").arrive(tx=1)
            later(rng.expovariate(1.0), lambda: bar("q_full").complete_tx(1))
            qcount += 1
            for j in range(n):
                for sel in (0, 1):
                    slot, fuse, euse = fill(pos)
                    if mistake != "producer_skips_kv_empty":
                        yield lambda: bar(f"kv_empty{slot}").try_wait((euse & 1) ^ 1, euse - 1)
                    f = bar(f"{'v' if sel else 'k'}_full{slot}")
                    f.arrive(tx=1)
                    slot_data[slot] = None

                    def land(slot=slot, p=pos, f=f):
                        slot_data[slot] = p
                        f.complete_tx(1)
                    later(rng.expovariate(0.5) if rng.random() < 0.9 else rng.uniform(5, 30), land)
                    pos += 1

    def qk():
        pos = qcount = 0
        sc = [0, 0]
        for nA, nB in units:
            n, nx = max(nA, nB), (nA, nB)
            if n == 0:
                continue
            yield lambda: bar("q_full").try_wait(qcount & 1, qcount)
            qcount += 1
            for j in range(n):
                slot, fuse, _ = fill(pos)
                yield lambda: bar(f"k_full{slot}").try_wait(fuse & 1, fuse)
                assert slot_data.get(slot) == pos, f"QK read slot {slot}: has {slot_data.get(slot)}, wants {pos}"
                for x in (0, 1):
                    if j >= nx[x]:
                        continue
                    k = sc[x]
                    if k > 0 and mistake != "qk_skips_p_free":
                        yield lambda: bar(f"p_free{x}").try_wait((k - 1) & 1, k - 1)
                    st = s_state[x]
                    assert st is None or st == ("P", x, k - 1, "done"), f"S{x} overwritten while holding {st}"

                    def chk(x=x, k=k, slot=slot, p=pos):
                        assert slot_data.get(slot) == p, f"K slot {slot} overwritten under the MMA"
                        s_state[x] = ("S", x, k)
                    mma("qk", chk, [bar(f"s_full{x}")])
                    if x == 0:
                        bar("qk_issued_a").arrive()   # a plain arrive right after the issue
                    sc[x] += 1
                mma("qk", lambda: None, [bar(f"kv_empty{slot}")])
                pos += 2
            mma("qk", lambda: None, [bar("q_empty")])

    def pv():
        pos = 0
        pc = [0, 0]
        unit_no = 0
        for nA, nB in units:
            n, nx = max(nA, nB), (nA, nB)
            if n == 0:
                continue
            for j in range(n):
                slot, fuse, _ = fill(pos + 1)
                v_ready = False
                for x in (0, 1):
                    if j >= nx[x]:
                        continue
                    k = pc[x]
                    if mistake != "pv_skips_p_full":
                        yield lambda: bar(f"p_full{x}").try_wait(k & 1, k)
                    if x == 1 and j + 1 < nA:   # P_B V_j queued after S_A of tile j + 1
                        ka = pc[0]
                        yield lambda: bar("qk_issued_a").try_wait(ka & 1, ka)
                    if not v_ready:
                        yield lambda: bar(f"v_full{slot}").try_wait(fuse & 1, fuse)
                        v_ready = True
                    assert slot_data.get(slot) == pos + 1, f"PV read slot {slot}: has {slot_data.get(slot)}"

                    def chk(x=x, k=k, j=j, u=unit_no, slot=slot, p=pos + 1):
                        assert slot_data.get(slot) == p, f"V slot {slot} overwritten under the MMA"
                        assert s_state[x] == ("P", x, k), f"PV read P{x} holding {s_state[x]}, wants {k}"
                        s_state[x] = ("P", x, k, "done")
                        if j == 0:
                            assert o_state[x] in (None, ("read",)), f"O{x} overwritten while {o_state[x]}"
                            o_state[x] = (u, 1)
                        else:
                            assert o_state[x] == (u, j), f"O{x} holds {o_state[x]}, wants ({u}, {j})"
                            o_state[x] = (u, j + 1)
                    commits = [bar(f"p_free{x}")]
                    if j == nx[x] - 1:
                        commits.append(bar(f"o_full{x}"))
                    mma("pv", chk, commits)
                    pc[x] += 1
                mma("pv", lambda: None, [bar(f"kv_empty{slot}")])
                pos += 2
            unit_no += 1

    def softmax(x):
        sc = oc = 0
        unit_no = 0
        for nA, nB in units:
            n, nx = max(nA, nB), (nA, nB)
            if n == 0:
                continue
            for j in range(nx[x]):
                k = sc
                yield lambda: bar(f"s_full{x}").try_wait(k & 1, k)
                assert s_state[x] == ("S", x, k), f"softmax read S{x} holding {s_state[x]}, wants {k}"
                if j > 0 and rng.random() < 0.3:   # a rescale reads and writes O_x in place
                    assert o_state[x] == (unit_no, j), f"rescale of O{x} while {o_state[x]}"
                s_state[x] = ("P", x, k)
                bar(f"p_full{x}").arrive()
                sc += 1
            if nx[x] > 0:
                o = oc
                yield lambda: bar(f"o_full{x}").try_wait(o & 1, o)
                assert o_state[x] == (unit_no, nx[x]), f"epilogue read O{x} while {o_state[x]}"
                o_state[x] = ("read",)
                oc += 1
            unit_no += 1

    actors = {"prod": producer(), "qk": qk(), "pv": pv(), "smA": softmax(0), "smB": softmax(1)}
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
