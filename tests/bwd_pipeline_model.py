"""Discrete-event model of the dK/dV backward kernel's mbarrier protocol (host
logic only; no attention arithmetic).

Roles, as in the kernel: the TMA producer (K and V once per unit, then a ring
of (Q_t, dO_t) pairs, one per 64-query step), the warp that issues S^T and
dP^T, the warp that issues the dV and dK products, and the elementwise warps
(one actor).  Tensor memory as in the kernel: two step
buffers b = t % 2 (the dQ kernel: three, b = t % 3), each with an S^T half and a dP^T half; the elementwise
warps read both and write P^T and dS^T over them; the dV product reads P^T
(its commit releases the S^T half) and the dK product reads dS^T (its commit
releases the dP^T half and the ring slot).  Per step t the first issuer
issues S^T_t after the release of the S^T half by step t-2 and dP^T_t after
the release of the dP^T half, with one commit for both; the second issues the
products of step t once the elementwise warps are done with it, and after a
unit's last step the commits that publish the accumulators and free K/V.

The model checks that no buffer half is overwritten before its product has
consumed it, that every MMA reads the step (and ring slot, and K/V unit) it
means, that a unit's first products find the accumulators already read by
the previous unit's epilogue, and that the epilogue reads them complete.
TMA loads land after random delays; MMAs start and complete in issue order
but overlap one another in the pipe, a commit arrives once every earlier MMA
has completed, and the elementwise warps take time over each step and over
the epilogue.
A parity wait passes iff the parity of the completed phases differs from the
one asked for; passing on an older phase (aliasing) or a deadlock fails the
run.
"""

import random

from pipeline_model import Bar


def run(units, slots, seed, mistake=None, kernel="dkdv"):
    """``units``: steps per unit (0 = a unit without gradient work).
    ``kernel`` "dkdv" models the dK/dV kernel as described above; "dq" the
    dQ kernel, which differs in three ways: one product per step (dQ += dS
    K_t) reads only the S half, where dS was written, and its commit frees the
    whole step buffer and the ring slot; S and dP both wait for that one
    release; and the unit-resident operands (Q and dO there) are freed by the
    score issuer's commit after the unit's last S and dP.
    ``mistake`` plants one protocol error: "s_skips_s_free",
    "dp_skips_d_free", "products_skip_pd_full", "producer_skips_qd_empty",
    "epilogue_skips_out_full", "kv_load_skips_kv_empty"."""
    dq = kernel == "dq"
    rng = random.Random(seed)
    B = {}

    def bar(name, count=1):
        if name not in B:
            B[name] = Bar(name, count)
        return B[name]

    nbuf = 3 if dq else 2
    for b in range(nbuf):
        for n in ("st_full", "pd_full", "s_free", "d_free"):
            bar(f"{n}{b}")
    for s in range(slots):
        bar(f"qd_full{s}"); bar(f"qd_empty{s}")
    for n in ("kv_full", "kv_empty", "out_full"):
        bar(n)

    events, now, seq = [], [0.0], [0]

    def later(delay, fn):
        seq[0] += 1
        events.append((now[0] + delay, seq[0], fn))

    tails = {w: {"start": 0.0, "end": 0.0} for w in ("st", "pd")}

    def mma(check_start, check_end, commits=(), issuer="st"):
        # The MMAs of one issuer start and complete in issue order, but the
        # pipe overlaps them (one may start before the previous one has
        # completed); the two issuers' streams are not ordered against each
        # other at all.  An MMA reads and writes from its start to its
        # completion, and both ends are checked.  A commit tracks the earlier
        # MMAs of its own issuer only.
        tail = tails[issuer]
        start = max(now[0], tail["start"]) + rng.uniform(0.0, 0.3)
        end = max(start + rng.uniform(0.1, 2.0), tail["end"] + rng.uniform(0.0, 0.2))
        tail["start"], tail["end"] = start, end
        seq[0] += 1
        events.append((start, seq[0], check_start))
        seq[0] += 1

        def done():
            check_end()
            for c in commits:
                c.arrive()
        events.append((end, seq[0], done))

    def commit(*bars, issuer="st"):
        mma(lambda: None, lambda: None, bars, issuer)

    work = [u for u in units if u > 0]
    slot_data = {}                    # ring slot -> step whose Q/dO it holds
    kv_data = [None]                  # unit whose K/V is resident
    half_s = {b: None for b in range(nbuf)}   # ("S", t) -> ("P", t) -> ("P", t, "done")
    half_d = {b: None for b in range(nbuf)}   # ("dP", t) -> ("dS", t) -> ("dS", t, "done")
    acc = {"dv": ("free", -1), "dk": ("free", -1)}   # ("busy", unit, last step) / ("free", unit)

    def producer():
        ring = 0
        for u, n in enumerate(work):
            if mistake != "kv_load_skips_kv_empty":
                yield lambda: bar("kv_empty").try_wait((u & 1) ^ 1, u - 1)
            bar("kv_full").arrive(tx=1)
            kv_data[0] = None

            def land_kv(u=u):
                kv_data[0] = u
                bar("kv_full").complete_tx(1)
            later(rng.expovariate(0.5), land_kv)
            for _ in range(n):
                slot, use = ring % slots, ring // slots
                if mistake != "producer_skips_qd_empty":
                    yield lambda: bar(f"qd_empty{slot}").try_wait((use & 1) ^ 1, use - 1)
                bar(f"qd_full{slot}").arrive(tx=1)
                slot_data[slot] = None

                def land(slot=slot, t=ring):
                    slot_data[slot] = t
                    bar(f"qd_full{slot}").complete_tx(1)
                later(rng.expovariate(1.0) if rng.random() < 0.9 else rng.uniform(5, 20), land)
                ring += 1

    def products_issuer():
        # the dV and dK products of every step, in step order
        tcount = 0

        def products(t, u, first):
            b, slot = t % nbuf, t % slots
            if mistake != "products_skip_pd_full":
                yield lambda: bar(f"pd_full{b}").try_wait((t // nbuf) & 1, t // nbuf)

            def dv_start(t=t, b=b, slot=slot, u=u, first=first):
                assert half_s[b] == ("P", t), f"dV of step {t} reads S half {b} holding {half_s[b]}"
                assert slot_data.get(slot) == t, f"dV of step {t} reads slot {slot} holding {slot_data.get(slot)}"
                if first:
                    assert acc["dv"] == ("free", u - 1), f"dV accumulator reused while {acc['dv']}"

            def dv_end(t=t, b=b, u=u):
                assert half_s[b] == ("P", t), f"S half {b} changed under the dV of step {t}"
                assert acc["dv"][0] != "reading", f"dV of step {t} lands while the epilogue reads"
                half_s[b] = ("P", t, "done")
                acc["dv"] = ("busy", u, t)

            def dk_start(t=t, b=b, slot=slot, u=u, first=first):
                assert half_d[b] == ("dS", t), f"dK of step {t} reads dP half {b} holding {half_d[b]}"
                assert slot_data.get(slot) == t, f"dK of step {t} reads slot {slot} holding {slot_data.get(slot)}"
                if first:
                    assert acc["dk"] == ("free", u - 1), f"dK accumulator reused while {acc['dk']}"

            def dk_end(t=t, b=b, slot=slot, u=u):
                assert half_d[b] == ("dS", t) and slot_data.get(slot) == t, f"operands of dK {t} changed"
                assert acc["dk"][0] != "reading", f"dK of step {t} lands while the epilogue reads"
                half_d[b] = ("dS", t, "done")
                acc["dk"] = ("busy", u, t)
            def dq_end(t=t, b=b, slot=slot, u=u):
                assert half_s[b] == ("P", t) and slot_data.get(slot) == t, f"operands of dQ {t} changed"
                assert acc["dv"][0] != "reading", f"dQ of step {t} lands while the epilogue reads"
                half_s[b] = ("P", t, "done")
                half_d[b] = ("dS", t, "done")   # the dP half was only read
                acc["dv"] = acc["dk"] = ("busy", u, t)
            if dq:
                mma(dv_start, dq_end, [bar(f"s_free{b}"), bar(f"qd_empty{slot}")], "pd")
            else:
                mma(dv_start, dv_end, [bar(f"s_free{b}")], "pd")
                mma(dk_start, dk_end, [bar(f"d_free{b}"), bar(f"qd_empty{slot}")], "pd")

        for u, n in enumerate(work):
            for i in range(n):
                yield from products(tcount + i, u, i == 0)
            if dq:
                commit(bar("out_full"), issuer="pd")
            else:
                commit(bar("out_full"), bar("kv_empty"), issuer="pd")
            tcount += n

    def scores_issuer():
        # S^T and dP^T of every step
        tcount = 0
        for u, n in enumerate(work):
            yield lambda: bar("kv_full").try_wait(u & 1, u)
            for i in range(n):
                tt = tcount + i
                b, slot, use = tt % nbuf, tt % slots, tt // nbuf
                yield lambda: bar(f"qd_full{slot}").try_wait((tt // slots) & 1, tt // slots)
                if tt >= nbuf and mistake != "s_skips_s_free":
                    yield lambda: bar(f"s_free{b}").try_wait((use - 1) & 1, use - 1)

                def s_start(tt=tt, b=b, slot=slot, u=u):
                    assert half_s[b] in (None, ("P", tt - nbuf, "done")), f"S^T {tt} overwrites {half_s[b]}"
                    assert slot_data.get(slot) == tt and kv_data[0] == u, f"S^T {tt} reads the wrong Q or K"

                def s_end(tt=tt, b=b, slot=slot, u=u):
                    assert slot_data.get(slot) == tt and kv_data[0] == u, f"Q or K changed under S^T {tt}"
                    assert half_s[b] in (None, ("P", tt - nbuf, "done")), f"S^T {tt} lands on {half_s[b]}"
                    half_s[b] = ("S", tt)
                mma(s_start, s_end)
                if tt >= nbuf and mistake != "dp_skips_d_free" and not dq:
                    yield lambda: bar(f"d_free{b}").try_wait((use - 1) & 1, use - 1)

                def d_start(tt=tt, b=b, slot=slot, u=u):
                    assert half_d[b] in (None, ("dS", tt - nbuf, "done")), f"dP^T {tt} overwrites {half_d[b]}"
                    assert slot_data.get(slot) == tt and kv_data[0] == u, f"dP^T {tt} reads the wrong dO or V"

                def d_end(tt=tt, b=b, slot=slot, u=u):
                    assert slot_data.get(slot) == tt and kv_data[0] == u, f"dO or V changed under dP^T {tt}"
                    assert half_d[b] in (None, ("dS", tt - nbuf, "done")), f"dP^T {tt} lands on {half_d[b]}"
                    half_d[b] = ("dP", tt)
                mma(d_start, d_end, [bar(f"st_full{b}")])
            if dq:   # Q and dO are done after the unit's last S and dP
                commit(bar("kv_empty"))
            tcount += n

    def elementwise():
        # reading, computing and writing a step takes time; so does the epilogue
        tcount = 0
        for u, n in enumerate(work):
            for i in range(n):
                tt = tcount + i
                b = tt % nbuf
                yield lambda: bar(f"st_full{b}").try_wait((tt // nbuf) & 1, tt // nbuf)
                assert half_s[b] == ("S", tt) and half_d[b] == ("dP", tt), \
                    f"step {tt} reads {half_s[b]}, {half_d[b]}"
                half_s[b] = ("reading", tt)
                half_d[b] = ("reading", tt)
                done = [False]

                def write(tt=tt, b=b, done=done):
                    assert half_s[b] == ("reading", tt) and half_d[b] == ("reading", tt), \
                        f"step {tt}: buffer {b} changed while the elementwise warps worked on it"
                    half_s[b] = ("P", tt)
                    half_d[b] = ("dS", tt)
                    done[0] = True
                later(rng.uniform(0.1, 3.0), write)
                yield lambda: done[0]
                bar(f"pd_full{b}").arrive()
            tcount += n
            if mistake != "epilogue_skips_out_full":
                yield lambda: bar("out_full").try_wait(u & 1, u)
            last = tcount - 1
            assert acc["dv"] == ("busy", u, last) and acc["dk"] == ("busy", u, last), \
                f"epilogue of unit {u} reads {acc}"
            acc["dv"] = acc["dk"] = ("reading", u)
            done = [False]

            def read_out(u=u, done=done):
                assert acc["dv"] == ("reading", u) and acc["dk"] == ("reading", u), \
                    f"accumulators changed under the epilogue of unit {u}: {acc}"
                acc["dv"] = acc["dk"] = ("free", u)
                done[0] = True
            later(rng.uniform(0.1, 3.0), read_out)
            yield lambda: done[0]

    actors = {"prod": producer(), "st": scores_issuer(), "pd": products_issuer(), "ew": elementwise()}
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
