"""A random-schedule model of the decode kernels' mbarrier hand-offs.

The actors are the roles of one CTA:
- the load producers, one warp, or two that split each tile's blocks;
- the S (score) issuer, into SB score buffers (one with the transposed
  64-row product);
- the softmax warps, as one actor because named barriers keep them in step;
- the two PV issuers.
Each actor takes one step at a time, in a random order weighted per actor,
so that chosen roles run far behind. Asynchronous completions fire at random
too: TMA landings in any order, and tcgen05 commits in order per issuing
thread.

An mbarrier completes a phase once it has its arrivals and its transaction
bytes. A parity wait passes iff the number of completed phases has the other
parity; this is the hardware's rule, so a waiter two phases behind is fooled.

The model reports:
- a load into a ring slot whose last contents no PV has freed;
- a read of the wrong tile's data (S, rope, P);
- a P buffer overwritten before both PVs read it;
- a deadlock, where nothing can move (on the GPU, the bounded wait gives up).

Ring layout: tile i has KB blocks; block kb is the u = KB * i + kb-th use of
the ring, slot u % R. With two producers, producer 0 loads blocks
[0, ceil(KB/2)) and producer 1 the rest (an odd KB gives producer 0 one
more). PV issuer m frees the blocks producer m loads (with one producer,
the same split). The rope ring has RR
slots, one per tile, and every producer loads a part of each; the S issuer
reads it last and frees it with its final commit, or (rope_first) reads it
first and frees it with a commit of its own before the tile's blocks, and
then the producers load each tile's rope before its blocks. With expand (fp8
rows) one producer lands each block's codes behind a raw barrier and each
tile's scales in one of two scale slots; expander e widens block e of every
tile in place once both have landed, then marks the block full, and the
producer reloads a scale slot once every expander is done with it. The softmax
waits for PV(i - PB) before it writes P(i) into buffer i % PB. It waits for
PV(i - 1) as well on a random 30% of tiles, standing for an O rescale. It
hands tile i to the PV issuers through hand-off barrier i % H."""
from __future__ import annotations

import random


class Bar:
    def __init__(self, count: int):
        self.count = count
        self.pending = 0
        self.tx = 0
        self.phases = 0

    def arrive_expect(self, n: int = 1, tx: int = 0):
        self.tx += tx
        self.pending += n
        self._check()

    def complete_tx(self, b: int):
        self.tx -= b
        self._check()

    def _check(self):
        if self.pending >= self.count and self.tx == 0:
            self.pending -= self.count
            self.phases += 1

    def passes(self, parity: int) -> bool:
        return (self.phases & 1) != parity


def run(seed: int, *, KB: int, R: int, RR: int, producers: int, PB: int, H: int, N: int = 40,
        weights: dict | None = None, rope_first: bool = False, expand: bool = False, SB: int = 2) -> list[str]:
    """One random schedule; returns the problems found (empty when none)."""
    rnd = random.Random(seed)
    blk_full = [Bar(1) for _ in range(R)]
    raw_full = [Bar(1) for _ in range(R)]
    # every expander releases a scale slot (a control may count fewer)
    scale_full, scale_empty = [Bar(1), Bar(1)], [Bar(KB), Bar(KB)]
    scale_data = [None, None]
    raw_data = [None] * R
    blk_empty = [Bar(1) for _ in range(R)]
    rope_full = [Bar(producers) for _ in range(RR)]
    rope_empty = [Bar(1) for _ in range(RR)]
    s_full, s_free = [Bar(1) for _ in range(SB)], [Bar(1) for _ in range(SB)]
    o_done = [Bar(2), Bar(2)]
    handoff = [Bar(1) for _ in range(H)]
    slot_data, slot_held = [None] * R, [None] * R
    rope_data = [None] * RR
    s_buf = [None, None]
    pbuf, pbuf_reads = [None] * PB, [None] * PB
    errors: list[str] = []
    landings = []                                  # TMA completions, any order
    commits = {"S": [], "PV0": [], "PV1": []}     # tcgen05 commits, in order per thread
    half = (KB + 1) // 2

    def blocks(m):
        # the blocks of producer / PV issuer m: [0, half) and [half, KB)
        return range(0, half) if m == 0 else range(half, KB)

    def load_rope(i):
        rr = i % RR
        if i >= RR:
            yield lambda rr=rr, i=i: rope_empty[rr].passes(((i // RR) - 1) & 1)
        rope_full[rr].arrive_expect(1, 1)

        def land_rope(rr=rr, i=i):
            rope_data[rr] = i
            rope_full[rr].complete_tx(1)
        landings.append(land_rope)
        yield None

    def producer(pp):
        mine = range(KB) if producers == 1 else blocks(pp)
        for i in range(N):
            if rope_first:
                yield from load_rope(i)
            for kb in mine:
                u = KB * i + kb
                s, f = u % R, u // R
                if f > 0:
                    yield lambda s=s, f=f: blk_empty[s].passes((f - 1) & 1)
                if slot_held[s] is not None:
                    errors.append(f"load of tile {i} block {kb} over unfreed {slot_held[s]} in slot {s}")
                slot_held[s] = (i, kb)
                bar = raw_full[s] if expand else blk_full[s]
                bar.arrive_expect(1, 1)

                def land(s=s, i=i, kb=kb, bar=bar):
                    if expand:
                        raw_data[s] = (i, kb)
                    else:
                        slot_data[s] = (i, kb)
                    bar.complete_tx(1)
                landings.append(land)
                yield None
            if expand:
                sb = i & 1
                if i >= 2:
                    yield lambda sb=sb, i=i: scale_empty[sb].passes(((i >> 1) - 1) & 1)
                scale_full[sb].arrive_expect(1, 1)

                def land_scales(sb=sb, i=i):
                    scale_data[sb] = i
                    scale_full[sb].complete_tx(1)
                landings.append(land_scales)
                yield None
            if not rope_first:
                yield from load_rope(i)

    def expander(e):
        for i in range(N):
            sb = i & 1
            yield lambda sb=sb, i=i: scale_full[sb].passes((i >> 1) & 1)
            u = KB * i + e
            s, f = u % R, u // R
            yield lambda s=s, f=f: raw_full[s].passes(f & 1)
            if raw_data[s] != (i, e):
                errors.append(f"expander {e} tile {i} widened codes of {raw_data[s]}")
            if scale_data[sb] != i:
                errors.append(f"expander {e} tile {i} used the scales of tile {scale_data[sb]}")
            slot_data[s] = (i, e)
            blk_full[s].arrive_expect()
            yield None
            scale_empty[sb].arrive_expect()
            yield None

    def s_issuer():
        for i in range(N):
            if i >= SB:
                yield lambda i=i: s_free[i % SB].passes(((i // SB) - 1) & 1)
            rr = i % RR
            if rope_first:
                # the rope's products first; its slot is released once they are done
                yield lambda rr=rr, i=i: rope_full[rr].passes((i // RR) & 1)
                if rope_data[rr] != i:
                    errors.append(f"S({i}) rope read tile {rope_data[rr]}")
                commits["S"].append(lambda rr=rr: rope_empty[rr].arrive_expect())
                yield None
            for kb in range(KB):
                u = KB * i + kb
                yield lambda s=u % R, f=u // R: blk_full[s].passes(f & 1)
                if slot_data[u % R] != (i, kb):
                    errors.append(f"S({i}) block {kb} read {slot_data[u % R]}")
            if not rope_first:
                yield lambda rr=rr, i=i: rope_full[rr].passes((i // RR) & 1)
                if rope_data[rr] != i:
                    errors.append(f"S({i}) rope read tile {rope_data[rr]}")

            def done(i=i, rr=rr):
                s_buf[i % SB] = i
                s_full[i % SB].arrive_expect()
                if not rope_first:
                    rope_empty[rr].arrive_expect()
            commits["S"].append(done)
            yield None

    def softmax():
        for i in range(N):
            yield lambda i=i: s_full[i % SB].passes((i // SB) & 1)
            if s_buf[i % SB] != i:
                errors.append(f"softmax({i}) read S of tile {s_buf[i % SB]}")
            s_free[i % SB].arrive_expect()
            yield None
            if i > 0 and rnd.random() < 0.3:
                yield lambda i=i: o_done[(i - 1) & 1].passes(((i - 1) >> 1) & 1)
            if i >= PB:
                yield lambda i=i: o_done[(i - PB) & 1].passes(((i - PB) >> 1) & 1)
            b = i % PB
            if pbuf_reads[b] is not None and pbuf_reads[b][0] != 2:
                errors.append(f"softmax({i}) overwrote P of tile {pbuf[b]} before both PVs read it")
            pbuf[b], pbuf_reads[b] = i, [0]
            handoff[i % H].arrive_expect()
            yield None
        yield lambda: o_done[(N - 1) & 1].passes(((N - 1) >> 1) & 1)

    def pv(mt):
        for i in range(N):
            yield lambda i=i: handoff[i % H].passes((i // H) & 1)
            if pbuf[i % PB] != i:
                errors.append(f"PV{mt}({i}) read P of tile {pbuf[i % PB]}")
            reads = pbuf_reads[i % PB]
            for kb in blocks(mt):
                s = (KB * i + kb) % R
                if slot_data[s] != (i, kb):
                    errors.append(f"PV{mt}({i}) block {kb} read {slot_data[s]}")

                def free(s=s, i=i, kb=kb):
                    if slot_held[s] == (i, kb):
                        slot_held[s] = None
                    blk_empty[s].arrive_expect()
                commits[f"PV{mt}"].append(free)

            def finished(i=i, reads=reads):
                reads[0] += 1
                o_done[i & 1].arrive_expect()
            commits[f"PV{mt}"].append(finished)
            yield None

    actors = {"S": s_issuer(), "SM": softmax(), "PV0": pv(0), "PV1": pv(1)}
    for pp in range(producers):
        actors[f"LD{pp}"] = producer(pp)
    if expand:
        for e in range(KB):
            actors[f"EX{e}"] = expander(e)
    weight = {k: (weights or {}).get(k, 1.0) for k in actors}
    waiting = {k: None for k in actors}
    finished_actors = set()
    for _ in range(400000):
        if len(finished_actors) == len(actors) and not landings and not any(commits.values()):
            return errors
        movers = [k for k in actors if k not in finished_actors and (waiting[k] is None or waiting[k]())]
        asyncs = [("land", j) for j in range(len(landings))] + [("commit", k) for k, v in commits.items() if v]
        if not movers and not asyncs:
            stuck = sorted(k for k in actors if k not in finished_actors)
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
                finished_actors.add(o[1])
                waiting[o[1]] = None
        elif o[0] == "land":
            landings.pop(o[1])()
        else:
            commits[o[1]].pop(0)()
        if errors:
            return errors
    return errors + ["step limit"]
