"""A random-schedule model of the 65..128-row decode: the two 64-row groups
of a worker run as two CTAs of a cluster that share every tile through
multicast copies.

Each CTA runs the roles of the single-CTA model (tests/barrier_model.py) at
64 rows: two producers (K-blocks [0, KB/2) and [KB/2, KB)), the S issuer
(rope first, one score buffer), the softmax (one actor), two PV issuers.
What the pair adds:
- producer pp of CTA c issues, for its K-blocks, only the half of the tile
  rows that belongs to rank c, multicast into both CTAs' slot; each CTA arms
  its own full barrier for both halves, so a slot's barrier in one CTA may
  see the peer's bytes before its own producer has armed it;
- the rope halves: producer pp of CTA pp issues half pp into both CTAs, and
  both producers of each CTA arm half of its rope barrier;
- a K-block slot is released by the value products of both CTAs (the PV
  issuers commit to both CTAs' empty barriers, count 2), the rope slot by
  both CTAs' score products.

The model reports a copy that lands in a CTA's slot while that CTA still
needs the slot's previous contents, a reader that finds the wrong tile, and
a deadlock. Parity waits follow the hardware rule (tests/barrier_model.py)."""
from __future__ import annotations

import random

from barrier_model import Bar


def run_mc(seed: int, *, KB: int = 4, R: int = 11, RR: int = 2, PB: int = 1, N: int = 30,
           weights: dict | None = None, empty_count: int = 2, rope_count: int = 2) -> list[str]:
    """One random schedule; returns the problems found (empty when none).
    empty_count 1 (a control) releases a K-block slot on the value products of
    the barrier's own CTA only; rope_count 1 does the same for a rope slot and
    the score products."""
    rnd = random.Random(seed)
    errors: list[str] = []
    landings = []                                  # copy completions, any order
    commits = {}                                   # (cta, thread) -> in-order tcgen05 commits
    half = KB // 2

    class CTA:
        def __init__(self):
            self.blk_full = [Bar(1) for _ in range(R)]
            self.blk_empty = [Bar(empty_count) for _ in range(R)]
            self.rope_full = [Bar(2) for _ in range(RR)]
            self.rope_empty = [Bar(rope_count) for _ in range(RR)]
            self.s_full, self.s_free = Bar(1), Bar(1)
            self.o_done = [Bar(2), Bar(2)]
            self.p_full = [Bar(1), Bar(1)]
            self.slot_halves = [[None, None] for _ in range(R)]   # (tile, block) per half
            self.freed = [-1] * R                                  # last fill this CTA's PV released
            self.rope_halves = [[None, None] for _ in range(RR)]
            self.rope_freed = [-1] * RR
            self.s_buf = None
            self.pbuf, self.pbuf_reads = [None] * PB, [None] * PB

    ctas = [CTA(), CTA()]

    def producer(c, pp):
        me = ctas[c]
        mine = range(0, half) if pp == 0 else range(half, KB)
        for i in range(N):
            rr, rf = i % RR, i // RR
            if i >= RR:
                yield lambda rr=rr, rf=rf: me.rope_empty[rr].passes((rf - 1) & 1)
            me.rope_full[rr].arrive_expect(1, 1)
            if pp == c:
                # rope half pp, into both CTAs
                for x in (0, 1):
                    if ctas[x].rope_freed[rr] < rf - 1:
                        errors.append(f"rope of tile {i} into CTA {x} over an unconsumed rope slot {rr}")

                def land_rope(rr=rr, i=i, h=pp):
                    for x in (0, 1):
                        ctas[x].rope_halves[rr][h] = i
                        ctas[x].rope_full[rr].complete_tx(1)
                landings.append(land_rope)
            yield None
            for kb in mine:
                u = KB * i + kb
                s, f = u % R, u // R
                if f > 0:
                    yield lambda s=s, f=f: me.blk_empty[s].passes((f - 1) & 1)
                for x in (0, 1):
                    if ctas[x].freed[s] < f - 1:
                        errors.append(f"CTA {c} loads tile {i} block {kb} into CTA {x}'s slot {s}, "
                                      f"still in use there")
                me.blk_full[s].arrive_expect(1, 2)   # both halves, own and peer's

                def land(s=s, i=i, kb=kb, h=c):
                    for x in (0, 1):
                        ctas[x].slot_halves[s][h] = (i, kb)
                        ctas[x].blk_full[s].complete_tx(1)
                landings.append(land)
                yield None

    def s_issuer(c):
        me = ctas[c]
        key = (c, "S")
        commits[key] = []
        for i in range(N):
            if i >= 1:
                yield lambda i=i: me.s_free.passes((i - 1) & 1)
            rr, rf = i % RR, i // RR
            yield lambda rr=rr, rf=rf: me.rope_full[rr].passes(rf & 1)
            if me.rope_halves[rr] != [i, i]:
                errors.append(f"CTA {c} S({i}) read rope halves of tiles {me.rope_halves[rr]}")

            def rope_done(rr=rr, rf=rf):
                me.rope_freed[rr] = rf
                for x in ((0, 1) if rope_count == 2 else (c,)):
                    ctas[x].rope_empty[rr].arrive_expect()
            commits[key].append(rope_done)
            for kb in range(KB):
                u = KB * i + kb
                s, f = u % R, u // R
                yield lambda s=s, f=f: me.blk_full[s].passes(f & 1)
                if me.slot_halves[s] != [(i, kb), (i, kb)]:
                    errors.append(f"CTA {c} S({i}) block {kb} read {me.slot_halves[s]}")

            def done(i=i):
                me.s_buf = i
                me.s_full.arrive_expect()
            commits[key].append(done)
            yield None

    def softmax(c):
        me = ctas[c]
        for i in range(N):
            yield lambda i=i: me.s_full.passes(i & 1)
            if me.s_buf != i:
                errors.append(f"CTA {c} softmax({i}) read S of tile {me.s_buf}")
            me.s_free.arrive_expect()
            yield None
            if i >= PB:
                yield lambda i=i: me.o_done[(i - PB) & 1].passes(((i - PB) >> 1) & 1)
            b = i % PB
            if me.pbuf_reads[b] is not None and me.pbuf_reads[b][0] != 2:
                errors.append(f"CTA {c} softmax({i}) overwrote P of tile {me.pbuf[b]}")
            me.pbuf[b], me.pbuf_reads[b] = i, [0]
            me.p_full[i & 1].arrive_expect()
            yield None
        yield lambda: me.o_done[(N - 1) & 1].passes(((N - 1) >> 1) & 1)

    def pv(c, m):
        me = ctas[c]
        key = (c, f"PV{m}")
        commits[key] = []
        mine = range(0, half) if m == 0 else range(half, KB)
        for i in range(N):
            yield lambda i=i: me.p_full[i & 1].passes((i >> 1) & 1)
            if me.pbuf[i % PB] != i:
                errors.append(f"CTA {c} PV{m}({i}) read P of tile {me.pbuf[i % PB]}")
            reads = me.pbuf_reads[i % PB]
            for kb in mine:
                u = KB * i + kb
                s, f = u % R, u // R
                if me.slot_halves[s] != [(i, kb), (i, kb)]:
                    errors.append(f"CTA {c} PV{m}({i}) block {kb} read {me.slot_halves[s]}")

                def free(s=s, f=f):
                    me.freed[s] = f
                    # a multicast commit: both CTAs' empty barriers
                    for x in ((0, 1) if empty_count == 2 else (c,)):
                        ctas[x].blk_empty[s].arrive_expect()
                commits[key].append(free)

            def finished(i=i, reads=reads):
                reads[0] += 1
                me.o_done[i & 1].arrive_expect()
            commits[key].append(finished)
            yield None

    actors = {}
    for c in (0, 1):
        actors[f"LD{c}0"] = producer(c, 0)
        actors[f"LD{c}1"] = producer(c, 1)
        actors[f"S{c}"] = s_issuer(c)
        actors[f"SM{c}"] = softmax(c)
        actors[f"PV{c}0"] = pv(c, 0)
        actors[f"PV{c}1"] = pv(c, 1)
    weight = {k: (weights or {}).get(k, 1.0) for k in actors}
    waiting = {k: None for k in actors}
    done_actors = set()
    for _ in range(600000):
        if len(done_actors) == len(actors) and not landings and not any(commits.values()):
            return errors
        movers = [k for k in actors if k not in done_actors and (waiting[k] is None or waiting[k]())]
        asyncs = [("land", j) for j in range(len(landings))] + [("commit", k) for k, v in commits.items() if v]
        if not movers and not asyncs:
            stuck = sorted(k for k in actors if k not in done_actors)
            return errors + [f"deadlock: {stuck} all waiting"]
        opts = [(weight[k], ("actor", k)) for k in movers] + [(0.5, a) for a in asyncs]
        x = rnd.random() * sum(w for w, _ in opts)
        for w, o in opts:
            x -= w
            if x <= 0:
                break
        if o[0] == "actor":
            try:
                waiting[o[1]] = next(actors[o[1]])
            except StopIteration:
                done_actors.add(o[1])
                waiting[o[1]] = None
        elif o[0] == "land":
            landings.pop(o[1])()
        else:
            commits[o[1]].pop(0)()
        if errors:
            return errors
    return errors + ["step limit"]
