"""A model of K1's barrier protocol at head_dim 128, checked by random schedules.

The attention kernel at d = 128 runs five kinds of agents per CTA:
- the TMA producer (K, V and Q copies);
- two S issuers, one per query tile;
- one PV issuer for both tiles;
- two softmax groups.
They synchronise only through mbarriers waited on by phase parity. Each
MMA-issuing thread's products complete in its own issue order, and a commit
arrives once all earlier products of its thread have completed.

This test replays that protocol, as the kernel source states it, under
random interleavings. Each thread's products complete in issue order, but
different threads' products interleave freely, which allows more orders
than the hardware does. The test checks three things:

- every parity wait is exact: when it is evaluated, the barrier has
  completed either the phase before the awaited one or the awaited one
  itself, never two phases more or one fewer;
- no agent touches a buffer before the product or copy that feeds it has
  completed, or overwrites one that an outstanding product still reads;
- every agent finishes (no deadlock).

It needs no GPU. Like the kernel's header, it covers a CTA's range of
(item, key tile) units, which may start and end inside items.
"""
import random

import pytest

ST = 2  # K/V stages at d = 128 (one Q buffer)


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arr, self.done = name, count, 0, 0

    def arrive(self):
        self.arr += 1
        assert self.arr <= self.count, self.name
        if self.arr == self.count:
            self.arr = 0
            self.done += 1


class Sim:
    def __init__(self, seed, u_lo, u_hi, nkt, p_rescale=0.3):
        self.rng = random.Random(seed)
        self.u_lo, self.u_hi, self.nkt = u_lo, u_hi, nkt
        self.p_rescale = p_rescale
        B = {}
        B["q_full"] = Bar("q_full", 1)
        B["q_empty"] = Bar("q_empty", 2)
        for t in range(2):
            B[f"q_ready{t}"] = Bar(f"q_ready{t}", 1)
        for s in range(ST):
            B[f"k_full{s}"] = Bar(f"k_full{s}", 1)
            B[f"v_full{s}"] = Bar(f"v_full{s}", 1)
            B[f"k_empty{s}"] = Bar(f"k_empty{s}", 2)
            B[f"v_empty{s}"] = Bar(f"v_empty{s}", 1)
        for b in range(4):  # [tile][buffer]
            B[f"s_full{b}"] = Bar(f"s_full{b}", 1)
            B[f"p_full{b}"] = Bar(f"p_full{b}", 1)
            B[f"o_done{b}"] = Bar(f"o_done{b}", 1)
        self.B = B
        # segments of the range: (first unit, end unit)
        self.segs = []
        u = u_lo
        while u < u_hi:
            hi = min(u_hi, (u // nkt + 1) * nkt)
            self.segs.append((u, hi))
            u = hi
        # state for the hazard checks
        self.loaded_k = {}    # tile L -> stage copy landed
        self.loaded_v = {}
        self.stage_k = {}     # stage -> tile held
        self.stage_v = {}
        self.q_loaded = -1    # segment whose Q copy landed
        self.q_rot = {0: -1, 1: -1}  # segment whose tile-t queries are rotated
        self.done_ops = set()        # completed products ("S"|"PV", t, L, h)
        self.issued = set()
        self.p_written = set()       # (t, L, h)
        self.epilogue_done = {0: -1, 1: -1}  # last segment whose O was read
        self.queues = {}             # issuing thread -> list of pending items
        self.tma = []                # pending copies
        self.agents = []

    # ---------------------------------------------------------------- helpers
    def wait_ok(self, bar, n):
        """Parity wait for phase n (n = -1: the phase before the first)."""
        c = self.B[bar].done
        assert c in (n, n + 1), f"inexact parity wait on {bar}: phase {n} awaited, {c} completed"
        return c == n + 1

    def issue(self, thread, op):
        self.issued.add(op)
        self.queues.setdefault(thread, []).append(("op", op))

    def commit(self, thread, bar):
        self.queues.setdefault(thread, []).append(("commit", bar))

    def seg_of(self, L):
        u = self.u_lo + L
        for i, (lo, hi) in enumerate(self.segs):
            if lo <= u < hi:
                return i
        raise AssertionError

    # ---------------------------------------------------------------- agents
    # Each agent is a generator; it yields ("wait", bar, phase) and resumes
    # once the wait has returned true.
    def producer(self):
        for L in range(self.u_hi - self.u_lo):
            st = L % ST
            yield ("wait", f"k_empty{st}", L // ST - 1)
            old = self.stage_k.get(st)
            if old is not None:  # every S product that read the old K has completed
                assert all(("S", t, old, h) in self.done_ops for t in range(2) for h in range(2)), ("K", L)
            self.stage_k[st] = L
            self.loaded_k.pop(old, None)
            self.tma.append(("k", L, st))
            yield ("wait", f"v_empty{st}", L // ST - 1)
            old = self.stage_v.get(st)
            if old is not None:
                assert all(("PV", t, old, h) in self.done_ops for t in range(2) for h in range(2)), ("V", L)
            self.stage_v[st] = L
            self.loaded_v.pop(old, None)
            self.tma.append(("v", L, st))
            sg = self.seg_of(L)
            if self.u_lo + L == self.segs[sg][0]:
                if sg >= 1:
                    yield ("wait", "q_empty", sg - 1)
                    prev = [L2 for L2 in range(self.u_hi - self.u_lo) if self.seg_of(L2) == sg - 1]
                    assert all(("S", t, L2, h) in self.done_ops for t in range(2) for h in range(2)
                               for L2 in prev), ("Q", sg)
                self.tma.append(("q", sg, 0))

    def s_issuer(self, t):
        th = f"S{t}"

        def check_and_issue(L, h):
            assert L in self.loaded_k, ("S before K", t, L)
            assert self.q_rot[t] == self.seg_of(L), ("S before the queries", t, L)
            if L >= 1:  # P_t(L - 1, h) lies over this buffer
                assert ("PV", t, L - 1, h) in self.done_ops, ("S over unread P", t, L, h)
            self.issue(th, ("S", t, L, h))

        yield ("wait", f"q_ready{t}", 0)
        yield ("wait", "k_full0", 0)
        for h in range(2):
            check_and_issue(0, h)
            self.commit(th, f"s_full{2 * t + h}")
        self.commit(th, "k_empty0")
        if self.segs[0][1] - self.segs[0][0] == 1:
            self.commit(th, "q_empty")
        L = 0
        for sg, (lo, hi) in enumerate(self.segs):
            n_here = hi - lo
            final = sg == len(self.segs) - 1
            n_next = 0 if final else self.segs[sg + 1][1] - self.segs[sg + 1][0]
            for i in range(n_here):
                boundary = i + 1 == n_here
                if not (boundary and final):
                    st1 = (L + 1) % ST
                    next_last = n_next == 1 if boundary else i + 2 == n_here
                    yield ("wait", f"k_full{st1}", (L + 1) // ST)
                    if boundary:
                        yield ("wait", f"q_ready{t}", sg + 1)
                    for h in range(2):
                        yield ("wait", f"o_done{2 * t + h}", L)
                        check_and_issue(L + 1, h)
                        self.commit(th, f"s_full{2 * t + h}")
                    self.commit(th, f"k_empty{st1}")
                    if next_last:
                        self.commit(th, "q_empty")
                L += 1

    def pv_issuer(self):
        th = "PV"
        L = 0
        for sg, (lo, hi) in enumerate(self.segs):
            for i in range(hi - lo):
                st = L % ST
                yield ("wait", f"v_full{st}", L // ST)
                for h in range(2):
                    for t in range(2):
                        yield ("wait", f"p_full{2 * t + h}", L)
                        assert (t, L, h) in self.p_written, ("PV before P", t, L, h)
                        assert L in self.loaded_v, ("PV before V", t, L)
                        if i == 0 and h == 0:  # overwrites O_t: the last segment's O was read
                            assert self.epilogue_done[t] == sg - 1, ("O overwritten", t, sg)
                        self.issue(th, ("PV", t, L, h))
                        self.commit(th, f"o_done{2 * t + h}")
                self.commit(th, f"v_empty{st}")
                L += 1

    def softmax(self, t):
        g = 0
        L = 0
        for sg, (lo, hi) in enumerate(self.segs):
            yield ("wait", "q_full", sg)
            assert self.q_loaded == sg
            self.q_rot[t] = sg
            self.B[f"q_ready{t}"].arrive()
            for i in range(hi - lo):
                for h in range(2):
                    yield ("wait", f"s_full{2 * t + h}", g >> 1)
                    assert ("S", t, L, h) in self.done_ops, ("scores read early", t, L, h)
                    if not (i == 0 and h == 0) and self.rng.random() < self.p_rescale:
                        # O rescaled: PV(g - 1) must have landed, PV(g) not issued
                        gp = g - 1
                        yield ("wait", f"o_done{2 * t + (gp & 1)}", gp >> 1)
                        assert ("PV", t, gp >> 1, gp & 1) in self.done_ops, ("rescale early", t, g)
                        assert ("PV", t, L, h) not in self.issued
                    self.p_written.add((t, L, h))
                    self.B[f"p_full{2 * t + h}"].arrive()
                    g += 1
                L += 1
            gl = g - 1
            yield ("wait", f"o_done{2 * t + ((gl - 1) & 1)}", (gl - 1) >> 1)
            yield ("wait", f"o_done{2 * t + (gl & 1)}", gl >> 1)
            Ll = L - 1
            assert all(("PV", t, L2, h) in self.done_ops for L2 in range(Ll + 1) for h in range(2)
                       if self.seg_of(L2) == sg), ("O read early", t, sg)
            self.epilogue_done[t] = sg

    # ---------------------------------------------------------------- scheduler
    def run(self, max_steps=200000):
        agents = [self.producer(), self.s_issuer(0), self.s_issuer(1), self.pv_issuer(),
                  self.softmax(0), self.softmax(1)]
        pending = {i: None for i in range(len(agents))}  # the wait each agent sits in

        def advance(i):
            try:
                pending[i] = next(agents[i])
            except StopIteration:
                pending[i] = "done"

        for i in range(len(agents)):
            advance(i)
        for _ in range(max_steps):
            choices = []
            for i, w in pending.items():
                if w == "done":
                    continue
                _, bar, n = w
                if self.wait_ok(bar, n):
                    choices.append(("agent", i))
            for th, q in self.queues.items():
                if q:
                    choices.append(("thread", th))
            if self.tma:
                choices.append(("tma", None))
            if not choices:
                break
            kind, x = self.rng.choice(choices)
            if kind == "agent":
                advance(x)
            elif kind == "thread":
                what, item = self.queues[x].pop(0)
                if what == "op":
                    self.done_ops.add(item)
                else:  # a commit arrives once the thread's earlier products are done
                    self.B[item].arrive()
            else:
                j = self.rng.randrange(len(self.tma))
                kind2, L, st = self.tma.pop(j)
                if kind2 == "k":
                    self.loaded_k[L] = st
                    self.B[f"k_full{st}"].arrive()
                elif kind2 == "v":
                    self.loaded_v[L] = st
                    self.B[f"v_full{st}"].arrive()
                else:
                    self.q_loaded = L
                    self.B["q_full"].arrive()
        stuck = {i: w for i, w in pending.items() if w != "done"}
        assert not stuck, f"deadlock: {stuck}"
        assert not any(self.queues.values()) and not self.tma


@pytest.mark.parametrize("seed", range(120))
def test_d128_protocol_random_schedules(seed):
    rng = random.Random(1000 + seed)
    nkt = rng.choice([1, 2, 3, 5, 8])
    u_lo = rng.randrange(0, 3 * nkt)
    u_hi = u_lo + rng.randint(1, 14)
    Sim(seed, u_lo, u_hi, nkt, p_rescale=rng.choice([0.0, 0.3, 1.0])).run()


def test_model_catches_a_missing_wait():
    """Take out the waits on o_done (PV(L, h) landed): the checks for scores
    written over unread P, or O read before its last PV, fire in some
    schedules, so the model sees the hazards those waits prevent."""

    class NoPvWait(Sim):
        def wait_ok(self, bar, n):
            return True if bar.startswith("o_done") else super().wait_ok(bar, n)

    hits = 0
    for seed in range(60):
        try:
            NoPvWait(seed, 0, 8, 4).run()
        except AssertionError:
            hits += 1
    assert hits > 0


def test_model_catches_a_missing_query_wait():
    """Take out the S issuer's wait for the next item's rotated queries:
    the model reports S products issued before the queries are ready."""

    class NoQueryWait(Sim):
        def wait_ok(self, bar, n):
            return True if bar.startswith("q_ready") else super().wait_ok(bar, n)

    hits = 0
    for seed in range(60):
        try:
            NoQueryWait(seed, 1, 9, 3).run()
        except AssertionError:
            hits += 1
    assert hits > 0


# --------------------------------------------------------------------------
# head_dim 64: one issuing thread per tile (S and PV), P in its own columns,
# four K/V stages released together after PV, two Q buffers, and the
# softmax's rare recomputation of a tile's scores from Q and K in shared
# memory (the overflow case of the running reference).

ST64, QB64 = 4, 2


class Sim64(Sim):
    def __init__(self, seed, u_lo, u_hi, nkt, p_redo=0.3, softmax_frees_q=None):
        # as the kernel: the softmax arrives on q_empty for items of at most ST - 2 tiles
        if softmax_frees_q is None:
            softmax_frees_q = nkt <= ST64 - 2
        self.rng = random.Random(seed)
        self.u_lo, self.u_hi, self.nkt = u_lo, u_hi, nkt
        self.p_redo = p_redo
        self.softmax_frees_q = softmax_frees_q
        B = {}
        for qb in range(QB64):
            B[f"q_full{qb}"] = Bar(f"q_full{qb}", 1)
            B[f"q_empty{qb}"] = Bar(f"q_empty{qb}", 2 + (2 if softmax_frees_q else 0))
            for t in range(2):
                B[f"q_ready{2 * qb + t}"] = Bar(f"q_ready{2 * qb + t}", 1)
        for s in range(ST64):
            B[f"k_full{s}"] = Bar(f"k_full{s}", 1)
            B[f"v_full{s}"] = Bar(f"v_full{s}", 1)
            B[f"k_empty{s}"] = Bar(f"k_empty{s}", 2)
        for t in range(2):
            for name in ("s_full", "s_free", "p_full", "o_done"):
                B[f"{name}{t}"] = Bar(f"{name}{t}", 1)
        self.B = B
        self.segs = []
        u = u_lo
        while u < u_hi:
            hi = min(u_hi, (u // nkt + 1) * nkt)
            self.segs.append((u, hi))
            u = hi
        self.loaded_k, self.loaded_v, self.stage_k, self.stage_v = {}, {}, {}, {}
        self.q_buf = {0: -1, 1: -1}      # segment whose queries the buffer holds (from the copy's issue)
        self.q_landed = set()
        self.q_rot = {0: -1, 1: -1}
        self.s_read = set()              # (t, g): the softmax holds S_t(g) in registers
        self.tile_done = set()           # (t, g): the softmax has finished tile g (P stored, p_full)
        self.done_ops, self.issued, self.p_written = set(), set(), set()
        self.epilogue_done = {0: -1, 1: -1}
        self.queues, self.tma = {}, []

    def producer(self):
        n = self.u_hi - self.u_lo
        for g in range(n):
            st = g % ST64
            for kind in ("k", "v"):
                yield ("wait", f"k_empty{st}", g // ST64 - 1)
                stage = self.stage_k if kind == "k" else self.stage_v
                old = stage.get(st)
                if old is not None:
                    if kind == "k":  # read by the S products and by a recomputation of tile old
                        assert all(("S", t, old, ) in self.done_ops for t in range(2)), ("K", g)
                        assert all((t, old) in self.tile_done for t in range(2)), ("K reused", g)
                        self.loaded_k.pop(old, None)
                    else:
                        assert all(("PV", t, old) in self.done_ops for t in range(2)), ("V", g)
                        self.loaded_v.pop(old, None)
                stage[st] = g
                self.tma.append((kind, g, st))
            sg = self.seg_of(g)
            if self.u_lo + g == self.segs[sg][0]:
                qb = sg % QB64
                if sg >= QB64:
                    yield ("wait", f"q_empty{qb}", sg // QB64 - 1)
                    old = sg - QB64
                    tiles = [g2 for g2 in range(n) if self.seg_of(g2) == old]
                    assert all(("S", t, g2) in self.done_ops for t in range(2) for g2 in tiles), ("Q", sg)
                    # a recomputation in segment `old` reads these queries
                    assert all((t, g2) in self.tile_done for t in range(2) for g2 in tiles), ("Q reused", sg)
                self.q_buf[qb] = sg
                self.tma.append(("q", sg, qb))

    def issuer(self, t):
        th = f"I{t}"

        def issue_s(g, qb):
            assert g in self.loaded_k, ("S before K", t, g)
            assert self.q_buf[qb] == self.seg_of(g) and self.q_rot[t] == self.seg_of(g), ("S before Q", t, g)
            if g >= 1:
                assert (t, g - 1) in self.s_read, ("S over unread scores", t, g)
            self.issue(th, ("S", t, g))

        yield ("wait", f"q_ready{t}", 0)
        yield ("wait", "k_full0", 0)
        issue_s(0, 0)
        self.commit(th, f"s_full{t}")
        if self.segs[0][1] - self.segs[0][0] == 1:
            self.commit(th, "q_empty0")
        g = 0
        for sg, (lo, hi) in enumerate(self.segs):
            n_here = hi - lo
            final = sg == len(self.segs) - 1
            n_next = 0 if final else self.segs[sg + 1][1] - self.segs[sg + 1][0]
            for i in range(n_here):
                st, st1 = g % ST64, (g + 1) % ST64
                boundary = i + 1 == n_here
                more = not (boundary and final)
                next_last = n_next == 1 if boundary else i + 2 == n_here

                def next_s():
                    qb1 = (sg + 1) % QB64 if boundary else sg % QB64
                    yield ("wait", f"k_full{st1}", (g + 1) // ST64)
                    yield ("wait", f"s_free{t}", g)
                    if boundary:
                        yield ("wait", f"q_ready{2 * qb1 + t}", (sg + 1) // QB64)
                    issue_s(g + 1, qb1)
                    self.commit(th, f"s_full{t}")
                    if next_last:
                        self.commit(th, f"q_empty{qb1}")

                if more and not boundary:
                    yield from next_s()
                yield ("wait", f"v_full{st}", g // ST64)
                yield ("wait", f"p_full{t}", g)
                assert (t, g) in self.p_written and g in self.loaded_v, ("PV early", t, g)
                if i == 0:
                    assert self.epilogue_done[t] == sg - 1, ("O overwritten", t, sg)
                self.issue(th, ("PV", t, g))
                self.commit(th, f"o_done{t}")
                self.commit(th, f"k_empty{st}")
                if more and boundary:
                    yield from next_s()
                g += 1

    def softmax(self, t):
        g = 0
        for sg, (lo, hi) in enumerate(self.segs):
            qb = sg % QB64
            yield ("wait", f"q_full{qb}", sg // QB64)
            assert sg in self.q_landed and self.q_buf[qb] == sg
            self.q_rot[t] = sg
            self.B[f"q_ready{2 * qb + t}"].arrive()
            for i in range(hi - lo):
                yield ("wait", f"s_full{t}", g)
                assert ("S", t, g) in self.done_ops, ("scores read early", t, g)
                self.s_read.add((t, g))
                self.B[f"s_free{t}"].arrive()
                if g >= 1:  # P_t(g) goes over P_t(g - 1)
                    yield ("wait", f"o_done{t}", g - 1)
                    assert ("PV", t, g - 1) in self.done_ops, ("P over unread P", t, g)
                self.p_written.add((t, g))
                if i > 0 and self.rng.random() < self.p_redo:
                    # the overflow case: this tile's scores again, from the
                    # queries and keys in shared memory
                    assert self.q_buf[qb] == sg, ("recomputation read overwritten queries", t, g)
                    assert self.stage_k.get(g % ST64) == g and g in self.loaded_k, ("recomputation K", t, g)
                self.tile_done.add((t, g))
                self.B[f"p_full{t}"].arrive()
                g += 1
            if self.softmax_frees_q:
                self.B[f"q_empty{qb}"].arrive()
            yield ("wait", f"o_done{t}", g - 1)
            assert all(("PV", t, g2) in self.done_ops for g2 in range(g)), ("O read early", t, sg)
            self.epilogue_done[t] = sg

    def run(self, max_steps=200000):
        agents = [self.producer(), self.issuer(0), self.issuer(1), self.softmax(0), self.softmax(1)]
        pending = {}

        def advance(i):
            try:
                pending[i] = next(agents[i])
            except StopIteration:
                pending[i] = "done"

        for i in range(len(agents)):
            advance(i)
        for _ in range(max_steps):
            choices = [("agent", i) for i, w in pending.items() if w != "done" and self.wait_ok(w[1], w[2])]
            choices += [("thread", th) for th, q in self.queues.items() if q]
            if self.tma:
                choices.append(("tma", None))
            if not choices:
                break
            kind, x = self.rng.choice(choices)
            if kind == "agent":
                advance(x)
            elif kind == "thread":
                what, item = self.queues[x].pop(0)
                if what == "op":
                    self.done_ops.add(item)
                else:
                    self.B[item].arrive()
            else:
                kind2, a, b = self.tma.pop(self.rng.randrange(len(self.tma)))
                if kind2 == "k":
                    self.loaded_k[a] = b
                    self.B[f"k_full{b}"].arrive()
                elif kind2 == "v":
                    self.loaded_v[a] = b
                    self.B[f"v_full{b}"].arrive()
                else:
                    self.q_landed.add(a)
                    self.B[f"q_full{b}"].arrive()
        stuck = {i: w for i, w in pending.items() if w != "done"}
        assert not stuck, f"deadlock: {stuck}"
        assert not any(self.queues.values()) and not self.tma


@pytest.mark.parametrize("seed", range(120))
def test_d64_protocol_random_schedules(seed):
    rng = random.Random(2000 + seed)
    nkt = rng.choice([1, 2, 3, 5, 8])
    u_lo = rng.randrange(0, 3 * nkt)
    u_hi = u_lo + rng.randint(1, 16)
    Sim64(seed, u_lo, u_hi, nkt, p_redo=rng.choice([0.0, 0.3, 1.0])).run()


def test_d64_model_catches_q_refilled_under_a_recomputation():
    """Without the softmax's own arrival on q_empty, the producer may refill
    a Q buffer once the S products of the segment two back have completed,
    while that segment's softmax can still recompute a tile's scores from
    those queries. This is possible only when segments are shorter than
    the K/V ring (items of at most three key tiles). The model finds the
    hazard, so for such items the kernel's softmax arrives on q_empty at
    the end of each segment; for longer items the copies in between already
    wait for the softmax, and the model finds no hazard without that
    arrival."""
    hits = 0
    for seed in range(200):
        rng = random.Random(5000 + seed)
        nkt = rng.choice([1, 2, 3])
        u_lo = rng.randrange(0, 3 * nkt)
        try:
            Sim64(seed, u_lo, u_lo + rng.randint(4, 12), nkt, p_redo=1.0, softmax_frees_q=False).run()
        except AssertionError as e:
            assert "Q reused" in str(e) or "overwritten queries" in str(e), e
            hits += 1
    assert hits > 0


@pytest.mark.parametrize("nkt", [3, 4, 5, 8])
def test_d64_longer_items_need_no_softmax_arrival(nkt):
    for seed in range(80):
        rng = random.Random(7000 + seed)
        u_lo = rng.randrange(0, 3 * nkt)
        Sim64(seed, u_lo, u_lo + rng.randint(1, 4 * nkt + 4), nkt, p_redo=1.0,
              softmax_frees_q=False).run()


# --------------------------------------------------------------------------
# Split items: the contributors of one query row merge through an arrival
# counter, with no waiting.  Each contributor at the end of its key range
# (one thread per row):
# - loads the counter with acquire; if every other contributor has counted
#   in, it is the last and merges its own O from tensor memory, publishing
#   nothing;
# - otherwise it publishes (O, m, l), then adds 1 with acquire-release; if
#   the old value shows every other contributor counted in, it is the last
#   and merges.
# The merger resets the counter for the next launch.


def merge_round(rng, n):
    """One row with n contributors under a random interleaving; returns
    (mergers, partials the merger could read, counter after the launch)."""
    cnt = [0]
    published = set()
    mergers = []
    # each contributor's steps as a generator; a step is one atomic action
    def contributor(c):
        if cnt[0] == n - 1:  # acquire load: the others have counted in
            mergers.append((c, set(published), "direct"))
            cnt[0] = 0
            return
        yield
        published.add(c)      # the partial, then the count (release)
        yield
        old = cnt[0]
        cnt[0] += 1
        if old == n - 1:
            yield
            mergers.append((c, set(published) - {c}, "counted"))
            cnt[0] = 0

    gens = [contributor(c) for c in range(n)]
    live = list(range(n))
    while live:
        i = rng.choice(live)
        try:
            next(gens[i])
        except StopIteration:
            live.remove(i)
    return mergers, cnt[0]


@pytest.mark.parametrize("n", [2, 3, 4, 7])
def test_split_item_merge_has_one_merger_that_sees_every_partial(n):
    rng = random.Random(n)
    direct = 0
    for _ in range(400):
        mergers, cnt = merge_round(rng, n)
        assert len(mergers) == 1, mergers
        who, seen, path = mergers[0]
        assert seen >= set(range(n)) - {who}, (who, seen)
        assert cnt == 0
        direct += path == "direct"
    assert 0 < direct < 400  # both ways of being last occur
