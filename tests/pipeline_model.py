"""A discrete-event model of one CTA of attn_fwd_kernel: its synchronisation protocol, run under
random timing on the CPU.

The model mirrors the control flow of each role of the kernel (csrc/attn_fwd.cu): the TMA
producer, the two MMA-issuing warps, the eight softmax warps (4 per Q tile) and the four
correction warps, over a CTA's list of work items (each given by its number of K/V tiles).
It models the hardware objects the roles meet on:

- mbarriers: an arrival count, a transaction count and a phase; try_wait.parity(P) succeeds
  when the current phase's parity differs from P, exactly as in PTX, so a wait that runs two
  phases ahead of (or behind) a barrier is modelled as the hardware would run it;
- named barriers (bar.arrive / bar.sync with a thread count), which have no generations;
- the tensor pipe: MMAs execute one after another in issue order, each reading its shared
  memory operands and tensor-memory columns; tcgen05.commit arrives once all earlier MMAs of
  the issuing warp are done;
- TMA loads (random latency, then the bytes land and complete the transaction count) and TMA
  stores (the staging buffer is read for a random time).

A roles' wake-up after a barrier completes is delayed at random, and optional random stalls
(up to microseconds) are added between the steps of every role. The checks raise ModelError:
a load into a shared-memory buffer whose previous contents an issued MMA still has to read; an
MMA reading an operand that has not landed or has been replaced; a QK overwriting S before every
softmax warp has read it; a PV reading a P part that is not the current tile's, or accumulating
into O before its rescale or after the next item's first PV should have started; an epilogue
reading an O that is not the item's; an arrival on an mbarrier whose arrival count is already
used up; a named barrier completing without its waiting warp or seeing a warp arrive twice; a
hang (every role waiting with no timer left); and, at exit, TMA loads or MMAs still in flight or
named barriers with pending arrivals. Bounded waits give up after their limits (2 s; the
softmax's wait for S after 10 s or once its issuing warp has stopped), set the abort flag and
the status, as the kernel does.

The producer's slot and Q-buffer waits exist in two forms: `count` (the kernel's: monotonic
counts of the S tiles the softmax warps have taken) and `parity` (an earlier form that waited on
the parity of the S-full barriers, kept so that the tests show the model catching its failure).
"""
from __future__ import annotations

import heapq
import itertools
import random

K_STAGES = 4          # K/V ring slots
N_PARTS = 3           # parts of P per tile (early PV)
WAIT_LIMIT = 2_000_000_000
DRAIN_LIMIT = 200_000_000
S_WAIT_LIMIT = 10_000_000_000


class ModelError(Exception):
    pass


class MBar:
    def __init__(self, name: str, count: int):
        self.name, self.count, self.pending, self.phase, self.tx = name, count, count, 0, 0

    def _maybe_complete(self, sim):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count
            sim.changed()

    def arrive(self, sim):
        if self.pending <= 0:
            raise ModelError(f"{self.name}: arrival with the arrival count used up")
        self.pending -= 1
        self._maybe_complete(sim)

    def arrive_expect_tx(self, sim, n: int):
        self.tx += n
        self.arrive(sim)

    def complete_tx(self, sim, n: int):
        self.tx -= n
        self._maybe_complete(sim)

    def try_wait(self, parity: int) -> bool:
        return (self.phase & 1) != parity


class CTA:
    """One CTA running its items; `items` lists the K/V tile count of each item."""

    def __init__(self, items, seed, withhold=-1, producer="count", stalls=False):
        self.items = list(items)
        self.rng = random.Random(seed)
        self.withhold = withhold
        self.producer_form = producer
        self.stalls = stalls
        self.t = 0
        self.events = []
        self.seq = itertools.count()
        self.waiters = []
        self.actors = 0
        self.finished = 0
        self.abort = False
        self.status = None
        self.stopped = [False, False]
        self.seen = [0, 0]
        self.bars = {}
        for q in range(2):
            for name, count in (("QFull", 1), ("SFull", 1), ("OSafe", 4), ("OFull", 1), ("Stats", 4),
                                ("MmaDone", 1), ("Turn", 1)):
                self.bars[f"{name}{q}"] = MBar(f"{name}{q}", count)
        for s in range(K_STAGES):
            self.bars[f"KV{s}"] = MBar(f"KV{s}", 1)
        self.nbar = {}
        self.smem = {"Q0": None, "Q1": None, **{f"KV{s}": None for s in range(K_STAGES)}}
        self.loads_in_flight = 0
        self.pipe = []
        self.pipe_free_at = 0
        self.last_op = {}
        self.done_ops = set()
        self.op_ids = itertools.count()
        self.S = [None, None]
        self.S_read = [[None] * 4 for _ in range(2)]
        self.P = [[[None] * N_PARTS for _ in range(4)] for _ in range(2)]
        self.O_acc = [[None] * 4 for _ in range(2)]
        self.O_rescaled = [[None] * 4 for _ in range(2)]
        self.O_read = [[None] * 4 for _ in range(2)]
        self.alpha = [[None] * 4 for _ in range(2)]
        self.alpha_read = [[None] * 4 for _ in range(2)]
        self.staging_busy = {}
        self.item_base = list(itertools.accumulate([0] + self.items[:-1]))

    # ------------------------------------------------------------------ event loop
    def at(self, dt, fn):
        heapq.heappush(self.events, (self.t + dt, next(self.seq), fn))

    def changed(self):
        self.at(0, self._wake)

    def _wake(self):
        keep = []
        for w in self.waiters:
            if w["ready"]():
                self.at(self.rng.choice((0, 5, 20, 50, 100, 200, 400)), lambda w=w: self._recheck(w))
            else:
                keep.append(w)
        self.waiters = keep

    def _recheck(self, w):
        if w["pred"]():
            self._resume(w["actor"], "ok")
        elif w.get("giveup") and w["giveup"]():
            self._resume(w["actor"], "abort")
        else:
            self.waiters.append(w)

    def _resume(self, actor, value):
        try:
            req = actor.send(value)
        except StopIteration:
            self.finished += 1
            return
        kind = req[0]
        if kind == "delay":
            self.at(req[1], lambda: self._resume(actor, None))
        elif kind == "wait":
            _, pred, giveup, deadline = req
            w = {"actor": actor, "pred": pred, "giveup": giveup, "deadline": deadline,
                 "ready": (lambda: pred() or (giveup is not None and giveup()))}
            if w["ready"]():
                self.at(0, lambda: self._recheck(w))
            else:
                self.waiters.append(w)
        else:
            raise ModelError(f"unknown request {kind}")

    def start(self, gen):
        self.actors += 1
        self.at(0, lambda: self._resume(gen, None))

    def run(self):
        while True:
            if self.events:
                self.t, _, fn = heapq.heappop(self.events)
                fn()
                continue
            if self.finished == self.actors:
                return
            timed = [w for w in self.waiters if w["deadline"] is not None]
            if not timed:
                raise ModelError("hang: every role waits with no timer left")
            w = min(timed, key=lambda x: x["deadline"])
            self.waiters.remove(w)
            self.t = max(self.t, w["deadline"])
            self._resume(w["actor"], "timeout")

    # ------------------------------------------------------------------ waits (generators)
    def stall(self):
        if self.stalls:
            d = self.rng.choice((0, 0, 0, 0, 0, 20, 3000))
            if d:
                yield ("delay", d)

    def wait_bar(self, bar, parity, role, watch_abort=True, limit=WAIT_LIMIT):
        b = self.bars[bar]
        if b.try_wait(parity):
            return True
        res = yield ("wait", lambda: b.try_wait(parity), (lambda: self.abort) if watch_abort else None,
                     self.t + limit)
        if res == "ok":
            return True
        if res == "timeout" and watch_abort:
            self.fail(role, bar)
        return False

    def wait_s_full(self, q, parity):
        b = self.bars[f"SFull{q}"]
        if b.try_wait(parity):
            return True
        res = yield ("wait", lambda: b.try_wait(parity), lambda: self.stopped[q], self.t + S_WAIT_LIMIT)
        if res == "ok":
            return True
        if res == "timeout":
            self.fail(3, f"SFull{q}")
        return False

    def wait_count(self, q, target):
        if self.seen[q] >= target:
            return True
        res = yield ("wait", lambda: self.seen[q] >= target, lambda: self.abort, self.t + WAIT_LIMIT)
        if res == "ok":
            return True
        if res == "timeout":
            self.fail(1, f"seen{q}")
        return False

    def wait_until(self, pred):
        if not pred():
            yield ("wait", pred, None, None)

    def fail(self, role, what):
        self.abort = True
        if self.status is None:
            self.status = (role, what)
        self.changed()

    # ------------------------------------------------------------------ asynchronous units
    def tma_load(self, buf, bar, content):
        old = self.smem[buf]
        for op in self.pipe:
            if buf in op["reads"] and op["reads"][buf] == old:
                raise ModelError(f"t={self.t}: load into {buf} while {op['name']} still has to read {old}")
        self.smem[buf] = ("in flight", content)
        self.loads_in_flight += 1
        self.bars[bar].arrive_expect_tx(self, 1)

        def land():
            self.smem[buf] = content
            self.loads_in_flight -= 1
            self.bars[bar].complete_tx(self, 1)
        self.at(self.rng.choice((600, 900, 1200, 2000, 3500)), land)

    def mma(self, issuer, name, reads, check, apply):
        op = {"id": next(self.op_ids), "name": name, "reads": reads, "check": check, "apply": apply}
        self.pipe.append(op)
        self.last_op[issuer] = op["id"]
        if len(self.pipe) == 1:
            self._start_next_mma()

    def _start_next_mma(self):
        if not self.pipe:
            return
        op = self.pipe[0]

        def operands_ok():
            for buf, want in op["reads"].items():
                if self.smem[buf] != want:
                    raise ModelError(f"t={self.t}: {op['name']} reads {buf} = {self.smem[buf]}, wants {want}")

        def go():
            operands_ok()
            op["check"]()
            dur = self.rng.choice((60, 100, 150, 300))
            self.pipe_free_at = self.t + dur

            def done():
                operands_ok()
                op["apply"]()
                self.done_ops.add(op["id"])
                self.pipe.pop(0)
                self.changed()
                self._start_next_mma()
            self.at(dur, done)
        self.at(max(0, self.pipe_free_at - self.t), go)

    def commit(self, issuer, bar):
        last = self.last_op.get(issuer)

        def fire():
            self.bars[bar].arrive(self)

        def poll():
            if last is None or last in self.done_ops:
                fire()
            else:
                self.at(10, poll)
        self.at(self.rng.choice((0, 30)), poll)

    # ------------------------------------------------------------------ named barriers
    def _nbar(self, bid):
        return self.nbar.setdefault(bid, {"arrived": [], "waiting": [], "gen": 0})

    def nb_arrive(self, bid, who):
        nb = self._nbar(bid)
        if who in nb["arrived"]:
            raise ModelError(f"t={self.t}: named barrier {bid}: {who} arrives twice in one generation")
        nb["arrived"].append(who)
        self._nb_check(bid)

    def nb_sync(self, bid, who):
        nb = self._nbar(bid)
        gen = nb["gen"]
        nb["arrived"].append(who)
        nb["waiting"].append(who)
        self._nb_check(bid)
        yield from self.wait_until(lambda: nb["gen"] > gen)

    def _nb_check(self, bid):
        nb = self.nbar[bid]
        if len(nb["arrived"]) == 5:  # 4 softmax warps arrive, 1 issuing warp waits (160 threads)
            if len(nb["waiting"]) != 1:
                raise ModelError(f"t={self.t}: named barrier {bid} completed with waiting warps {nb['waiting']}")
            nb["arrived"], nb["waiting"] = [], []
            nb["gen"] += 1
            self.changed()

    # ------------------------------------------------------------------ item geometry
    def item_of_tile(self, gt):
        for k, base in enumerate(self.item_base):
            if base <= gt < base + self.items[k]:
                return k
        raise ModelError(f"tile {gt} outside the CTA's items")


def token_bar(t):
    return f"KV{t % K_STAGES}"


def token_parity(t):
    return (t // K_STAGES) & 1


# ====================================================================== roles
def set_up(c: CTA):
    c.tma_load("Q0", "QFull0", ("Q", 0, 0))
    if c.withhold != 0:
        c.tma_load("KV0", "KV0", ("T", 0))
    c.tma_load("Q1", "QFull1", ("Q", 1, 0))


def producer(c: CTA):
    ok, issued, gbase, q_loads = True, 1, 0, [1, 1]

    def need_q(q, k_item):
        # Q tile q of item k may be replaced once QK_q of the previous item's last tile is done.
        if c.producer_form == "count":
            return (yield from c.wait_count(q, gbase))
        return (yield from c.wait_bar(f"SFull{q}", (gbase - 1) & 1, 1))

    for k, n in enumerate(c.items):
        if not ok:
            break
        for u in range(2 * n):
            T = 2 * gbase + u
            if T == 0:
                continue
            yield from c.stall()
            if k > 0 and u == 0:
                if not (yield from need_q(0, k)):
                    ok = False
                    break
                c.tma_load("Q0", "QFull0", ("Q", 0, k))
                q_loads[0] += 1
            if T >= K_STAGES:
                prev = T - K_STAGES
                if c.producer_form == "count":
                    r = yield from c.wait_count(1, prev // 2 + 1 + (prev & 1))
                else:
                    ph = (prev - 1) // 2 + 1 if prev & 1 else prev // 2
                    r = yield from c.wait_bar("SFull1", ph & 1, 1)
                if not r:
                    ok = False
                    break
            if T != c.withhold:
                c.tma_load(f"KV{T % K_STAGES}", token_bar(T), ("T", T))
            issued = T + 1
            yield from c.stall()
            if k > 0 and u == 0:
                if not (yield from need_q(1, k)):
                    ok = False
                    break
                c.tma_load("Q1", "QFull1", ("Q", 1, k))
                q_loads[1] += 1
        gbase += n
    if not ok:
        for q in range(2):
            par = (q_loads[q] - 1) & 1 if c.producer_form == "count" else 0
            yield from c.wait_bar(f"QFull{q}", par, 1, False, DRAIN_LIMIT)
        for t in range(max(issued - K_STAGES, 0), issued):
            if t != c.withhold:
                yield from c.wait_bar(token_bar(t), token_parity(t), 1, False, DRAIN_LIMIT)


def issuer(c: CTA, q: int):
    name = f"issuer{q}"

    def issue_qk(gt, hand_over):
        k = c.item_of_tile(gt)

        def check():
            for w in range(4):
                if gt > 0 and c.S_read[q][w] != gt - 1:
                    raise ModelError(f"t={c.t}: QK_{q}({gt}) overwrites S before softmax warp {w} read it")

        def apply():
            c.S[q] = gt
        c.mma(name, f"QK{q}({gt})", {f"Q{q}": ("Q", q, k), f"KV{(2 * gt) % K_STAGES}": ("T", 2 * gt)}, check, apply)
        if hand_over:
            c.bars[f"Turn{q ^ 1}"].arrive(c)

    def issue_pv(gt, pi, first):
        def check():
            for w in range(4):
                if c.P[q][w][pi] != gt:
                    raise ModelError(f"t={c.t}: PV_{q}({gt}) part {pi} reads P of tile {c.P[q][w][pi]}")
                k = c.item_of_tile(gt)
                if first and k > 0 and c.O_read[q][w] != k - 1:
                    raise ModelError(f"t={c.t}: first PV_{q}({gt}) overwrites O before the epilogue read it")
                if not first and pi == 0:
                    if c.O_acc[q][w] != gt - 1 or c.O_rescaled[q][w] != gt:
                        raise ModelError(f"t={c.t}: PV_{q}({gt}) accumulates onto O before its rescale")

        def apply():
            if pi == N_PARTS - 1:
                for w in range(4):
                    c.O_acc[q][w] = gt
        tv = 2 * gt + 1
        c.mma(name, f"PV{q}({gt}).{pi}", {f"KV{tv % K_STAGES}": ("T", tv)}, check, apply)

    ok = yield from c.wait_bar(f"QFull{q}", 0, 2)
    ok = ok and (yield from c.wait_bar(token_bar(0), 0, 2))
    ok = ok and (q == 0 or (yield from c.wait_bar("Turn1", 0, 2)))
    if ok:
        issue_qk(0, False)
        c.commit(name, f"SFull{q}")
        c.bars[f"Turn{q ^ 1}"].arrive(c)
    k, n, next_item, gt, i = 0, c.items[0], len(c.items) > 1, 0, 0
    while ok:
        tv, tk = 2 * gt + 1, 2 * gt + 2
        more = i + 1 < n
        for pi in range(N_PARTS):
            yield from c.stall()
            yield from c.nb_sync(2 + 2 * pi + q, name)
            if not ok:
                continue
            if pi == 0:
                ok = yield from c.wait_bar(token_bar(tv), token_parity(tv), 2)
                ok = ok and (gt == 0 or (yield from c.wait_bar(f"OSafe{q}", (gt - 1) & 1, 2)))
                ok = ok and (yield from c.wait_bar(f"Turn{q}", (gt if q == 0 else gt + 1) & 1, 2))
            if pi == N_PARTS - 1 and ok and more:
                ok = yield from c.wait_bar(token_bar(tk), token_parity(tk), 2)
            if not ok:
                continue
            issue_pv(gt, pi, pi == 0 and i == 0)
            if pi == N_PARTS - 1:
                if more:
                    issue_qk(gt + 1, True)
                    c.commit(name, f"SFull{q}")
                else:
                    c.commit(name, f"OFull{q}")
                    if next_item:
                        ok = yield from c.wait_bar(token_bar(tk), token_parity(tk), 2)
                        ok = ok and (yield from c.wait_bar(f"QFull{q}", (k + 1) & 1, 2))
                        if ok:
                            issue_qk(gt + 1, True)
                            c.commit(name, f"SFull{q}")
                    elif q == 0:
                        c.bars["Turn1"].arrive(c)
        if more:
            i += 1
        else:
            k += 1
            if not next_item:
                break
            i, n, next_item = 0, c.items[k], k + 1 < len(c.items)
        gt += 1
    if not ok:
        c.stopped[q] = True
        c.changed()
    fin = ok and (yield from c.wait_bar(f"OFull{q}", (k - 1) & 1, 2))
    if not fin:
        c.commit(name, f"MmaDone{q}")
        yield from c.wait_bar(f"MmaDone{q}", 0, 2, False, DRAIN_LIMIT)


def softmax(c: CTA, q: int, w: int):
    who = f"softmax{q}.{w}"
    ok, gbase = True, 0
    for k, n in enumerate(c.items):
        if not ok:
            break
        next_item = k + 1 < len(c.items)
        for i in range(n):
            gt = gbase + i
            yield from c.stall()
            if not (yield from c.wait_s_full(q, gt & 1)):
                ok = False
                break
            if w == 0:
                c.seen[q] = gt + 1
                c.changed()
            if c.S[q] != gt:
                raise ModelError(f"t={c.t}: {who} reads S of tile {c.S[q]}, wants {gt}")
            c.S_read[q][w] = gt
            yield ("delay", c.rng.choice((50, 200, 400)))
            if i > 0:
                if c.alpha[q][w] is not None and c.alpha_read[q][w] != c.alpha[q][w]:
                    raise ModelError(f"t={c.t}: {who} overwrites rescale factors before they were read")
                c.alpha[q][w] = gt
                c.bars[f"Stats{q}"].arrive(c)
            for pi in range(N_PARTS):
                yield ("delay", c.rng.choice((30, 100, 250)))
                c.P[q][w][pi] = gt
                c.nb_arrive(2 + 2 * pi + q, who)
        if not ok:
            break
        if not (yield from c.wait_bar(f"OFull{q}", k & 1, 3)):
            ok = False
            break
        last = gbase + n - 1
        if c.O_acc[q][w] != last:
            raise ModelError(f"t={c.t}: {who} epilogue reads O of tile {c.O_acc[q][w]}, wants {last}")
        c.O_read[q][w] = k
        if next_item:
            c.bars[f"OSafe{q}"].arrive(c)
        for half in range(2):
            if half == 1 or k > 0:
                yield from c.wait_until(lambda: c.staging_busy.get((q, w), 0) == 0)
            yield ("delay", 50)
            c.staging_busy[(q, w)] = 1

            def store_read(key=(q, w)):
                c.staging_busy[key] = 0
                c.changed()
            c.at(c.rng.choice((200, 800, 1500)), store_read)
        gbase += n
    yield from c.wait_until(lambda: c.staging_busy.get((q, w), 0) == 0)


def correction(c: CTA, w: int):
    ok, sbase = True, 0
    for r, n in enumerate(c.items):
        if not ok:
            break
        i = 1
        while i < n and ok:
            for q in range(2):
                yield from c.stall()
                if not (yield from c.wait_bar(f"Stats{q}", (sbase + i - 1) & 1, 4)):
                    ok = False
                    break
                gt = c.item_base[r] + i
                if c.alpha[q][w] != gt:
                    raise ModelError(f"t={c.t}: correction {w} reads rescale factors of tile {c.alpha[q][w]}")
                c.alpha_read[q][w] = gt
                if c.rng.random() < 0.5:  # some row of this warp rebased: rescale O in tensor memory
                    if c.O_acc[q][w] != gt - 1:
                        raise ModelError(f"t={c.t}: correction {w} rescales O_{q} of tile {c.O_acc[q][w]}")
                    yield ("delay", c.rng.choice((100, 300)))
                    if c.O_acc[q][w] != gt - 1:
                        raise ModelError(f"t={c.t}: O_{q} changed under correction {w}")
                c.O_rescaled[q][w] = gt
                c.bars[f"OSafe{q}"].arrive(c)
            i += 1
        sbase += n - 1


def run(items, seed, withhold=-1, producer_form="count", stalls=False) -> CTA:
    """Runs one CTA to its end; returns it (status None: no wait gave up). Raises ModelError."""
    c = CTA(items, seed, withhold, producer_form, stalls)
    set_up(c)
    c.start(producer(c))
    for q in range(2):
        c.start(issuer(c, q))
    for q in range(2):
        for w in range(4):
            c.start(softmax(c, q, w))
    for w in range(4):
        c.start(correction(c, w))
    c.run()
    if c.loads_in_flight:
        raise ModelError(f"exit with {c.loads_in_flight} TMA loads in flight (status {c.status})")
    if c.pipe:
        raise ModelError(f"exit with {len(c.pipe)} MMAs in the tensor pipe")
    for bid, nb in c.nbar.items():
        if nb["arrived"]:
            raise ModelError(f"exit with named barrier {bid} holding arrivals {nb['arrived']}")
    return c
