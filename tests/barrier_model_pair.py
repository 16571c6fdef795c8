"""A random-schedule model of the two-CTA cluster decode kernel's hand-offs.

Each CTA of the pair runs the roles of the single-CTA model
(tests/barrier_model.py):
- one TMA producer;
- the S issuer;
- the softmax group;
- two PV issuers, on one ring of R pair slots and RR rope slots.
The two CTAs also exchange data. Every tile, each sends the other its
partial scores with a bulk copy into the peer's exchange buffer; that copy
lands on the peer's `xfull`, and the peer hands the buffer back through a
remote arrive on `xfree`. With split softmax columns, each CTA also pushes
its P block into the peer's P buffer. That copy lands on the peer's `pin`,
and it is sent only after the peer's `rp_free` has said that its PV of the
buffer's previous tile is done. With 32 query rows the score staging is
the tile's own P buffer. With an fp8 pool, the TMA lands codes and scales
and the expand warps widen them in place before S may read the slots.

A bulk copy reads its source and writes its destination at one random later
moment. The model reports:
- a source changed before the copy read it;
- a destination still in use when the copy wrote it;
- a reader that finds the wrong tile's data;
- a deadlock.
Parity waits follow the hardware rule; see tests/barrier_model.py."""
from __future__ import annotations

import random

from barrier_model import Bar


def run_pair(seed: int, *, R: int, RR: int, PB: int, split: bool, send_in_p: bool, N: int = 30,
             weights: dict | None = None, skip_xfree_before_p: bool = False, fp8: bool = False,
             raw_slots: int = 3) -> list[str]:
    """fp8: the TMA lands a tile's codes and scales in its two pair slots and
    completes raw_full[i % raw_slots]; the expand warps (one actor: four warps
    that meet at a named barrier every tile) wait for it, widen the codes in
    place and then arrive on both slots' pair_full."""
    rnd = random.Random(seed)
    errors: list[str] = []
    asyncs = []                                 # (name, fn): fire at a random later moment
    commits = {}                                # per (cta, thread) in-order tcgen05 commits

    class CTA:
        def __init__(self, c):
            self.c = c
            self.pair_full = [Bar(1) for _ in range(R)]
            self.raw_full = [Bar(1) for _ in range(raw_slots)]
            self.raw_data = [None] * raw_slots
            self.pair_empty = [Bar(1) for _ in range(R)]
            self.rope_full = [Bar(1) for _ in range(RR)]
            self.rope_empty = [Bar(1) for _ in range(RR)]
            self.s_full, self.s_free = [Bar(1), Bar(1)], [Bar(1), Bar(1)]
            self.o_done = [Bar(2), Bar(2)]
            self.p_full = [Bar(1), Bar(1)]
            self.xfull, self.xfree = Bar(1), Bar(1)
            self.pin = [Bar(1) for _ in range(PB)]
            self.rp_free = [Bar(1) for _ in range(PB)]
            self.slot_data, self.slot_held = [None] * R, [None] * R
            self.rope_data = [None] * RR
            self.s_buf = [None, None]
            self.xbuf = None                        # the peer's partial scores: tile
            self.xbuf_unread = False
            self.send = None                        # the staging of this CTA's partial scores (no P-buffer staging)
            # P buffer b: [own block, peer block, staged scores (32 rows)], and PV reads done of its tile
            self.pbuf = [{"own": None, "peer": None, "stage": None, "tile": None, "reads": 2} for _ in range(PB)]
            for k in ("S", "PV0", "PV1"):
                commits[(c, k)] = []

    ctas = [CTA(0), CTA(1)]

    def bulk(name, src_check, dst_write):
        def fire():
            if not src_check():
                errors.append(f"{name}: source changed before the copy read it")
            dst_write()
        asyncs.append((name, fire))

    def producer(me):
        for i in range(N):
            for pp in range(2):
                u = 2 * i + pp
                s, f = u % R, u // R
                if f > 0:
                    yield lambda s=s, f=f: me.pair_empty[s].passes((f - 1) & 1)
                if me.slot_held[s] is not None:
                    errors.append(f"CTA{me.c}: load of tile {i} pair {pp} over unfreed {me.slot_held[s]}")
                me.slot_held[s] = (i, pp)
                if not fp8:
                    me.pair_full[s].arrive_expect(1, 1)

                    def land(s=s, i=i, pp=pp):
                        me.slot_data[s] = (i, pp)
                        me.pair_full[s].complete_tx(1)
                    asyncs.append(("tma", land))
                yield None
            if fp8:
                # codes into the first slot, scales into the second, one barrier
                rs = i % raw_slots
                me.raw_full[rs].arrive_expect(1, 1)

                def land_raw(rs=rs, i=i):
                    me.slot_data[(2 * i) % R] = ("raw", i)
                    me.slot_data[(2 * i + 1) % R] = ("raw", i)
                    me.raw_data[rs] = i
                    me.raw_full[rs].complete_tx(1)
                asyncs.append(("tma", land_raw))
                yield None
            rr = i % RR
            if i >= RR:
                yield lambda rr=rr, i=i: me.rope_empty[rr].passes(((i // RR) - 1) & 1)
            me.rope_full[rr].arrive_expect(1, 1)

            def land_r(rr=rr, i=i):
                me.rope_data[rr] = i
                me.rope_full[rr].complete_tx(1)
            asyncs.append(("tma", land_r))
            yield None

    def expand(me):
        for i in range(N):
            rs = i % raw_slots
            yield lambda rs=rs, i=i: me.raw_full[rs].passes((i // raw_slots) & 1)
            s0, s1 = (2 * i) % R, (2 * i + 1) % R
            if me.raw_data[rs] != i or me.slot_data[s0] != ("raw", i) or me.slot_data[s1] != ("raw", i):
                errors.append(f"CTA{me.c} expand({i}) found {me.raw_data[rs]} / {me.slot_data[s0]} / {me.slot_data[s1]}")
            yield None
            me.slot_data[s0], me.slot_data[s1] = (i, 0), (i, 1)
            me.pair_full[s0].arrive_expect()
            me.pair_full[s1].arrive_expect()
            yield None

    def s_issuer(me):
        for i in range(N):
            if i >= 2:
                yield lambda i=i: me.s_free[i & 1].passes(((i - 2) >> 1) & 1)
            for pp in range(2):
                u = 2 * i + pp
                yield lambda s=u % R, f=u // R: me.pair_full[s].passes(f & 1)
                if me.slot_data[u % R] != (i, pp):
                    errors.append(f"CTA{me.c} S({i}) pair {pp} read {me.slot_data[u % R]}")
            rr = i % RR
            yield lambda rr=rr, i=i: me.rope_full[rr].passes((i // RR) & 1)

            def done(i=i, rr=rr):
                me.s_buf[i & 1] = i
                me.s_full[i & 1].arrive_expect()
                me.rope_empty[rr].arrive_expect()
            commits[(me.c, "S")].append(done)
            yield None

    def softmax(me, peer):
        for i in range(N):
            b = i % PB
            buf = me.pbuf[b]
            yield lambda i=i: me.s_full[i & 1].passes((i >> 1) & 1)
            if me.s_buf[i & 1] != i:
                errors.append(f"CTA{me.c} softmax({i}) read S of {me.s_buf[i & 1]}")
            if send_in_p and i >= PB:
                yield lambda i=i: me.o_done[(i - PB) & 1].passes(((i - PB) >> 1) & 1)
            if i > 0:
                yield lambda i=i: me.xfree.passes((i - 1) & 1)
            # stage this CTA's partial scores and push them to the peer
            if send_in_p:
                if buf["reads"] != 2:
                    errors.append(f"CTA{me.c} tile {i}: score staging over P of {buf['tile']} still read")
                buf["stage"] = i
                src_ok = (lambda buf=buf, i=i: buf["stage"] == i)
            else:
                me.send = i
                src_ok = (lambda i=i: me.send == i)

            def xland(i=i):
                if peer.xbuf_unread:
                    errors.append(f"CTA{peer.c}: scores of tile {i} landed over unread {peer.xbuf}")
                peer.xbuf = i
                peer.xbuf_unread = True
                peer.xfull.complete_tx(1)
            me.xfull.arrive_expect(1, 1)
            bulk(f"CTA{me.c} scores({i})", src_ok, xland)
            yield None
            yield lambda i=i: me.xfull.passes(i & 1)
            if me.xbuf != i:
                errors.append(f"CTA{me.c} softmax({i}) read the peer's scores of {me.xbuf}")
            me.xbuf_unread = False
            me.s_free[i & 1].arrive_expect()
            peer.xfree.arrive_expect()
            yield None
            if i > 0 and rnd.random() < 0.3:
                yield lambda i=i: me.o_done[(i - 1) & 1].passes(((i - 1) >> 1) & 1)
            if i >= PB:
                yield lambda i=i: me.o_done[(i - PB) & 1].passes(((i - PB) >> 1) & 1)
            if send_in_p and not skip_xfree_before_p:
                yield lambda i=i: me.xfree.passes(i & 1)
            if split:
                if i >= PB:
                    peer.rp_free[b].arrive_expect()
                me.pin[b].arrive_expect(1, 1)
            # this CTA's P block (and, unsplit, the whole P)
            if buf["reads"] != 2 and buf["tile"] is not None and buf["tile"] != i:
                errors.append(f"CTA{me.c} P({i}) over P of {buf['tile']} still read")
            if buf["tile"] != i:
                buf["tile"], buf["reads"] = i, 0
            buf["own"] = i
            if send_in_p:
                buf["stage"] = None
            if not split:
                buf["peer"] = i
            yield None
            if split:
                if i >= PB:
                    yield lambda b=b, i=i: me.rp_free[b].passes(((i // PB) - 1) & 1)

                def pland(b=b, i=i):
                    pb = peer.pbuf[b]
                    if pb["tile"] is not None and pb["tile"] != i and pb["reads"] != 2:
                        errors.append(f"CTA{peer.c}: P block of tile {i} landed over P of {pb['tile']} still read")
                    if pb["tile"] != i:
                        pb["tile"], pb["reads"] = i, 0
                    pb["peer"] = i
                    peer.pin[b].complete_tx(1)
                bulk(f"CTA{me.c} P({i})", lambda buf=buf, i=i: buf["own"] == i, pland)
                yield None
                yield lambda b=b, i=i: me.pin[b].passes((i // PB) & 1)
            if buf["own"] != i or buf["peer"] != i:
                errors.append(f"CTA{me.c} hands over P({i}) holding {buf['own']}/{buf['peer']}")
            me.p_full[i & 1].arrive_expect()
            yield None
        yield lambda: me.o_done[(N - 1) & 1].passes(((N - 1) >> 1) & 1)

    def pv(me, mt):
        for i in range(N):
            yield lambda i=i: me.p_full[i & 1].passes((i >> 1) & 1)
            buf = me.pbuf[i % PB]
            if buf["own"] != i or buf["peer"] != i:
                errors.append(f"CTA{me.c} PV{mt}({i}) read P {buf['own']}/{buf['peer']}")
            s = (2 * i + mt) % R
            if me.slot_data[s] != (i, mt):
                errors.append(f"CTA{me.c} PV{mt}({i}) read slot {s} = {me.slot_data[s]}")

            def free(s=s, i=i, mt=mt):
                if me.slot_held[s] == (i, mt):
                    me.slot_held[s] = None
                me.pair_empty[s].arrive_expect()

            def finished(i=i, buf=buf):
                if buf["tile"] == i:
                    buf["reads"] += 1
                me.o_done[i & 1].arrive_expect()
            commits[(me.c, f"PV{mt}")] += [free, finished]
            yield None

    actors = {}
    for c in (0, 1):
        me, peer = ctas[c], ctas[1 - c]
        actors[f"LD{c}"] = producer(me)
        if fp8:
            actors[f"EX{c}"] = expand(me)
        actors[f"S{c}"] = s_issuer(me)
        actors[f"SM{c}"] = softmax(me, peer)
        actors[f"PV0_{c}"] = pv(me, 0)
        actors[f"PV1_{c}"] = pv(me, 1)
    weight = {k: (weights or {}).get(k, 1.0) for k in actors}
    waiting = {k: None for k in actors}
    done = set()
    for _ in range(600000):
        if len(done) == len(actors) and not asyncs and not any(commits.values()):
            return errors
        movers = [k for k in actors if k not in done and (waiting[k] is None or waiting[k]())]
        pend = [("async", j) for j in range(len(asyncs))] + [("commit", k) for k, v in commits.items() if v]
        if not movers and not pend:
            return errors + [f"deadlock: {sorted(k for k in actors if k not in done)}"]
        opts = [(weight[k], ("actor", k)) for k in movers] + [(0.5, a) for a in pend]
        x = rnd.random() * sum(w for w, _ in opts)
        for w, o in opts:
            x -= w
            if x <= 0:
                break
        if o[0] == "actor":
            try:
                waiting[o[1]] = next(actors[o[1]])
            except StopIteration:
                done.add(o[1])
                waiting[o[1]] = None
        elif o[0] == "async":
            asyncs.pop(o[1])[1]()
        else:
            commits[o[1]].pop(0)()
        if errors:
            return errors
    return errors + ["step limit"]
