"""Executable models of the barrier protocols of the persistent backward kernels.

attn_bwd_dkdv_kernel and attn_bwd_dq_kernel run one CTA per SM.  Each CTA takes work items
(key-block pairs, query blocks) from a counter.  Every warp role waits on mbarriers whose
phases count sub-tiles and items over the CTA's whole run.  These models restate each role's
sequence of waits, arrivals, copies and MMA commits as a Python generator.  A randomised
scheduler then interleaves the roles with the asynchronous engines:
- the TMA, whose copies complete in any order;
- the tensor pipe, with one in-order queue per issuing warp, whose commits arrive when that
  warp's earlier MMAs are done.

A run checks three things:
- it ends (no deadlock);
- every parity wait passes exactly at its intended phase, never two phases late (a parity wait
  cannot tell phase k from phase k + 2);
- no copy or MMA overwrites a shared-memory stage, the K/V or Q/dO buffer, or a TMEM region
  (S, dP, P, dS, accumulators) before all its readers are done, and no reader sees the wrong
  contents.

`drop` names waits to leave out, so a test can check that the model catches each missing one.

Abort runs (`expire=True`) model the failure path.  A wait that makes progress may expire at
any moment: the CTA's abort flag goes up and the wait returns False.  Once the flag is up,
every such wait that has not completed returns False, and each role leaves its loops the way
the kernel does.  Drain waits ignore the flag and only pass when their phase completes.  When
the last role of a CTA finishes, which is where the kernel frees tensor memory and exits, no
copy and no MMA of that CTA may still be in flight, and no drain may wait for something never
issued (a deadlock).
"""
import random


class ProtocolError(Exception):
    pass


class Aborted(Exception):
    """A wait returned False: the role leaves its loops (the kernel's `ok = false; break`)."""


def check(cond, msg):
    if not cond:
        raise ProtocolError(msg)


class Bar:
    """An mbarrier: `count` arrivals plus the expected transaction bytes complete a phase."""

    def __init__(self, name, count):
        self.name, self.count, self.pend, self.tx, self.comp = name, count, count, 0, 0

    def arrive(self):
        self.pend -= 1
        check(self.pend >= 0, f"{self.name}: more arrivals than its count")
        self._complete()

    def expect_tx(self, nbytes):
        self.tx += nbytes
        self.arrive()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._complete()

    def _complete(self):
        if self.pend == 0 and self.tx == 0:
            self.comp += 1
            self.pend = self.count


class Model:
    """Shared scheduler: actors are (name, cta, generator) yielding ("wait", bar, phase) or
    ("step",); subclasses define the CTA state, the engines' completions and the roles."""

    SKIPS_EMPTY = True  # items with an empty list produce no epilogue

    def __init__(self, seed, ncta, items, drop=(), expire=False):
        self.rng = random.Random(seed)
        self.items, self.ncta, self.drop = items, ncta, set(drop)
        self.expire = expire
        self.counter = 0
        self.tma = []
        self.processed = []
        self.ctas = [self.make_cta(c) for c in range(ncta)]
        self.actors = []
        for c in self.ctas:
            self.actors += self.roles(c)

    def fetch_next(self):
        x = self.ncta + self.counter
        self.counter += 1
        return x

    @staticmethod
    def wait(bar, phase):
        """A wait that makes progress; raises Aborted when it returns False."""
        ok = yield ("wait", bar, phase)
        if not ok:
            raise Aborted()

    @staticmethod
    def drain(bar, phase):
        """A drain: passes only once the phase has completed, abort flag or not."""
        yield ("drain", bar, phase)

    def take(self, c, n):
        slot = n & 1
        yield from self.wait(c.item_full[slot], n >> 1)
        x = c.slot[slot]
        c.item_free[slot].arrive()
        return x

    def publish(self, c, n):
        """The producer's side of the two-slot item ring: waits until slot n % 2 is free and
        returns it."""
        slot = n & 1
        if n >= 2:
            yield from self.wait(c.item_free[slot], (n >> 1) - 1)
        return slot

    def mma_drain(self, c, bar):
        """An issuing warp waits for its own MMAs before tensor memory may be freed: a drain,
        or -- with "abort_mma_drain" dropped -- a wait that gives up once the flag is up."""
        if "abort_mma_drain" in self.drop:
            yield ("wait", bar, 0)
        else:
            yield from self.drain(bar, 0)

    def check_exit(self, c):
        """The last role of CTA c finished: tensor memory is freed and the CTA exits."""
        check(not any(j[0] is c for j in self.tma), f"cta{c.cid} exits with copies in flight")
        check(not c.mmaq[1] and not c.mmaq[2], f"cta{c.cid} frees tensor memory with MMAs in flight")

    def run(self):
        for c in self.ctas:
            c.abort = False
        pending = {id(a): self._advance(a, None) for a in self.actors}
        live = {c.cid: sum(1 for a in self.actors if a[1] is c and pending[id(a)] is not None) for c in self.ctas}
        for c in self.ctas:
            if live[c.cid] == 0:
                self.check_exit(c)
        while True:
            choices = []
            for a in self.actors:
                p = pending[id(a)]
                if p is None:
                    continue
                if p[0] == "step" or p[1].comp >= p[2] + 1:
                    choices.append(("actor", a, True))
                elif p[0] == "wait" and a[1].abort:
                    choices.append(("actor", a, False))  # the flag is up: the wait gives up
                elif p[0] == "wait" and self.expire and self.rng.random() < 0.02:
                    choices.append(("expire", a, False))  # the wait's time limit runs out
            choices += [("tma", i, None) for i in range(len(self.tma))]
            choices += [("mma", (c, w), None) for c in self.ctas for w in (1, 2) if c.mmaq[w]]
            if not choices:
                stuck = [(a[0], a[1].cid, p[1].name, p[2], p[1].comp) for a in self.actors
                         for p in [pending[id(a)]] if p is not None]
                check(not stuck, f"deadlock: {stuck[:6]}")
                return
            kind, v, ok = self.rng.choice(choices)
            if kind in ("actor", "expire"):
                p = pending[id(v)]
                if kind == "expire":
                    v[1].abort = True
                if p[0] != "step" and ok:
                    check(p[1].comp == p[2] + 1,
                          f"{v[0]} cta{v[1].cid}: {p[1].name} wait for phase {p[2]} passes at {p[1].comp}")
                pending[id(v)] = self._advance(v, ok)
                if pending[id(v)] is None:
                    live[v[1].cid] -= 1
                    if live[v[1].cid] == 0:
                        self.check_exit(v[1])
            elif kind == "tma":
                self.complete_tma(self.tma.pop(v))
            else:
                c, w = v
                self.complete_mma(c, c.mmaq[w].pop(0))
            for a in self.actors:
                p = pending[id(a)]
                if p is not None and p[0] != "step":
                    check(p[1].comp <= p[2] + 1,
                          f"{a[0]} cta{a[1].cid}: {p[1].name} two phases past phase {p[2]}")

    @staticmethod
    def _advance(actor, value):
        try:
            return actor[2].send(value) if value is not None else next(actor[2])
        except StopIteration:
            return None


NE = 8  # element-wise (dK/dV) or row (dQ) warps
ALL = frozenset(range(NE))


class DkdvModel(Model):
    """attn_bwd_dkdv_kernel: items are key-block pairs of `items[x]` 64-row query sub-tiles.
    SBUF is the number of S^T / dP^T buffers in TMEM (1 at d = 128, 2 at d = 64)."""

    STAGES = 4
    SBUF = 1

    def make_cta(self, cid):
        c = type("CTA", (), {})()
        c.cid = cid
        c.kv = Bar("kv", 1)
        c.sfull = [Bar(f"sfull{i}", 1) for i in range(self.SBUF)]
        c.sfree = [Bar(f"sfree{i}", NE) for i in range(self.SBUF)]
        c.full = [Bar(f"full{i}", 1) for i in range(self.STAGES)]
        c.empty = [Bar(f"empty{i}", 1) for i in range(self.STAGES)]
        c.pready = [Bar(f"pready{i}", NE) for i in range(2)]
        c.pfree = [Bar(f"pfree{i}", 1) for i in range(2)]
        c.drain, c.sdrain, c.kvfree, c.gdrain = Bar("drain", 1), Bar("sdrain", 1), Bar("kvfree", 1), Bar("gdrain", 1)
        c.item_full = [Bar(f"item_full{i}", 1) for i in range(2)]
        c.item_free = [Bar(f"item_free{i}", 2 + NE) for i in range(2)]
        c.slot = [None, None]
        c.stage = [None] * self.STAGES
        c.stage_readers = [set() for _ in range(self.STAGES)]
        c.kv_tag, c.kv_readers = None, 0
        c.S, c.S_read, c.DP = [None] * self.SBUF, [set() for _ in range(self.SBUF)], [None] * self.SBUF
        c.P, c.P_readers = [dict(), dict()], [0, 0]
        c.acc, c.acc_read, c.acc_inflight = None, set(ALL), 0
        c.mmaq = {1: [], 2: []}
        return c

    def roles(self, c):
        return ([("producer", c, self.producer(c)), ("s_issuer", c, self.s_issuer(c)),
                 ("g_issuer", c, self.g_issuer(c))] + [(f"ew{g}", c, self.elementwise(c, g)) for g in range(NE)])

    def complete_tma(self, job):
        c, kind, arg = job
        if kind == "stage":
            st, U = arg
            check(not c.stage_readers[st], f"stage {st} overwritten while read by {c.stage_readers[st]}")
            c.stage[st] = U
            c.stage_readers[st] = {"S", "DP", "DV", "DK"} | {f"ew{g}" for g in range(NE)}
            c.full[st].complete_tx(1)
        else:
            check(c.kv_readers == 0, "K/V overwritten while S/dP MMAs read them")
            c.kv_tag = arg
            c.kv.complete_tx(1)

    def complete_mma(self, c, op):
        kind = op[0]
        if kind == "commit":
            op[1].arrive()
        elif kind in ("S", "DP"):
            _, U, st, kvk = op
            sb = U % self.SBUF
            check(c.stage[st] == U and c.kv_tag == kvk, f"{kind}({U}): operands changed before completion")
            c.stage_readers[st].discard(kind)
            c.kv_readers -= 1
            if kind == "S":
                check(c.S[sb] is None or c.S_read[sb] >= ALL, f"S({U}) overwrote S({c.S[sb]}) before it was read")
                c.S[sb], c.S_read[sb] = U, set()
            else:
                c.DP[sb] = U
        else:
            _, W, st, bb, item, w = op
            check(c.stage[st] == W and all(c.P[bb].get(g) == W for g in range(NE)),
                  f"{kind}({W}): operands changed before completion")
            c.stage_readers[st].discard(kind)
            c.P_readers[bb] -= 1
            if kind == "DV":
                if w == 0:
                    check(c.acc_read >= ALL, f"item {item}: accumulators overwritten before the epilogue read them")
                else:
                    check(c.acc == (item, w - 1), f"item {item}: accumulation chain broken at {w}")
                c.acc, c.acc_read = (item, w), set()
            c.acc_inflight -= 1

    def producer(self, c):
        U = kvn = n = 0
        x = c.cid
        try:
            while True:
                slot = yield from self.publish(c, n)
                done = x >= len(self.items)
                c.slot[slot] = -1 if done else x
                c.item_full[slot].arrive()
                if done:
                    break
                xn = self.fetch_next()
                yield ("step",)
                nsub = self.items[x]
                if nsub > 0:
                    if kvn >= 1 and "kvfree" not in self.drop:
                        yield from self.wait(c.kvfree, kvn - 1)
                    check(c.kv_readers == 0, "K/V load issued while S/dP MMAs read them")
                    c.kv.expect_tx(1)
                    self.tma.append((c, "kv", (x, kvn)))
                    kvn += 1
                    for _ in range(nsub):
                        st = U % self.STAGES
                        if U >= self.STAGES and "empty" not in self.drop:
                            yield from self.wait(c.empty[st], U // self.STAGES - 1)
                        check(not c.stage_readers[st], f"stage {st} load issued while read by {c.stage_readers[st]}")
                        c.full[st].expect_tx(1)
                        self.tma.append((c, "stage", (st, U)))
                        U += 1
                        yield ("step",)
                x = xn
                n += 1
        except Aborted:
            if "abort_drain" in self.drop:
                return  # drains skipped on the abort path
        # U and kvn count the loads issued: drain the last one of each stage and the K / V load
        for v in range(max(0, U - self.STAGES), U):
            yield from self.drain(c.full[v % self.STAGES], v // self.STAGES)
        if kvn > 0:
            yield from self.drain(c.kv, kvn - 1)
    def s_issuer(self, c):
        U = kvn = n = 0
        try:
            while True:
                x = yield from self.take(c, n)
                n += 1
                if x < 0:
                    break
                nsub = self.items[x]
                if nsub == 0:
                    continue
                yield from self.wait(c.kv, kvn)
                kvk = (x, kvn)
                kvn += 1
                for _ in range(nsub):
                    st, sb = U % self.STAGES, U % self.SBUF
                    yield from self.wait(c.full[st], U // self.STAGES)
                    if U >= self.SBUF and "sfree" not in self.drop:
                        yield from self.wait(c.sfree[sb], U // self.SBUF - 1)
                    check(c.stage[st] == U and c.kv_tag == kvk, f"S({U}) issued on the wrong operands")
                    c.mmaq[1] += [("S", U, st, kvk), ("DP", U, st, kvk), ("commit", c.sfull[sb])]
                    c.kv_readers += 2
                    U += 1
                    yield ("step",)
                c.mmaq[1].append(("commit", c.kvfree))
        except Aborted:
            pass
        c.mmaq[1].append(("commit", c.sdrain))
        yield from self.mma_drain(c, c.sdrain)
    def g_issuer(self, c):
        W = n = 0
        try:
            while True:
                x = yield from self.take(c, n)
                n += 1
                if x < 0:
                    break
                nsub = self.items[x]
                for w in range(nsub):
                    st, bb = W % self.STAGES, W & 1
                    yield from self.wait(c.pready[bb], W >> 1)
                    yield from self.wait(c.full[st], W // self.STAGES)
                    check(all(c.P[bb].get(g) == W for g in range(NE)), f"dV/dK({W}) issued before P/dS were written")
                    c.mmaq[2] += [("DV", W, st, bb, x, w), ("DK", W, st, bb, x, w), ("commit", c.empty[st]),
                                  ("commit", c.pfree[bb])]
                    c.P_readers[bb] += 2
                    c.acc_inflight += 2
                    W += 1
                    yield ("step",)
                if nsub > 0:
                    c.mmaq[2].append(("commit", c.drain))
        except Aborted:
            pass
        c.mmaq[2].append(("commit", c.gdrain))
        yield from self.mma_drain(c, c.gdrain)
    def elementwise(self, c, g):
        U = an = n = 0
        try:
            while True:
                x = yield from self.take(c, n)
                n += 1
                if x < 0:
                    break
                nsub = self.items[x]
                for _ in range(nsub):
                    st, bb, sb = U % self.STAGES, U & 1, U % self.SBUF
                    yield from self.wait(c.sfull[sb], U // self.SBUF)
                    yield from self.wait(c.full[st], U // self.STAGES)
                    check(c.S[sb] == U and c.DP[sb] == U, f"ew{g}: reads S({U}) while TMEM holds S({c.S[sb]})")
                    check(c.stage[st] == U, f"ew{g}: statistics of sub-tile {U} replaced")
                    c.S_read[sb].add(g)
                    c.stage_readers[st].discard(f"ew{g}")
                    c.sfree[sb].arrive()
                    yield ("step",)
                    if U >= 2 and "pfree" not in self.drop:
                        yield from self.wait(c.pfree[bb], (U >> 1) - 1)
                    check(c.P_readers[bb] == 0, f"ew{g}: P/dS buffer {bb} written while MMAs read it")
                    c.P[bb][g] = U
                    c.pready[bb].arrive()
                    U += 1
                    yield ("step",)
                if nsub == 0:
                    continue
                if "drain" not in self.drop:
                    yield from self.wait(c.drain, an)
                an += 1
                check(c.acc == (x, nsub - 1) and c.acc_inflight == 0, f"ew{g}: epilogue of item {x} sees {c.acc}")
                c.acc_read.add(g)
                if g == 0:
                    self.processed.append(x)
                yield ("step",)
        except Aborted:
            pass

class DkdvModel64(DkdvModel):
    """attn_bwd_dkdv_kernel at d = 64: S^T / dP^T double-buffered in TMEM."""

    SBUF = 2


class DqModel(Model):
    """attn_bwd_dq_kernel: items are query blocks with `items[x]` kept key blocks.  Q and dO
    load into a two-slot ring; the row warps copy each block's Q into TMEM (each warp its
    part) for the S MMAs, the next block's right after the current block's last S was read."""

    KST, VST, QBUF = 4, 2, 2

    def make_cta(self, cid):
        c = type("CTA", (), {})()
        c.cid = cid
        c.q = [Bar(f"q{i}", 1) for i in range(self.QBUF)]
        c.qfree = [Bar(f"qfree{i}", 1) for i in range(self.QBUF)]
        c.qt = Bar("qt", NE)
        c.kfull = [Bar(f"kfull{i}", 1) for i in range(self.KST)]
        c.kempty = [Bar(f"kempty{i}", 1) for i in range(self.KST)]
        c.vfull = [Bar(f"vfull{i}", 1) for i in range(self.VST)]
        c.vempty = [Bar(f"vempty{i}", 1) for i in range(self.VST)]
        c.sfull = [Bar(f"sfull{i}", 1) for i in range(2)]
        c.sfree = [Bar(f"sfree{i}", NE) for i in range(2)]
        c.pready = [Bar(f"pready{i}", NE) for i in range(2)]
        c.pfree = [Bar(f"pfree{i}", 1) for i in range(2)]
        c.dq, c.gdrain, c.sdrain = Bar("dq", 1), Bar("gdrain", 1), Bar("sdrain", 1)
        c.item_full = [Bar(f"item_full{i}", 1) for i in range(2)]
        c.item_free = [Bar(f"item_free{i}", 2 + NE) for i in range(2)]
        c.slot = [None, None]
        # Q / dO slots: contents, S/dP MMAs reading them, row warps that copied its Q out
        c.qtag, c.q_readers = [None] * self.QBUF, [0] * self.QBUF
        c.q_copied = [set(ALL) for _ in range(self.QBUF)]
        # Q in TMEM: the block each row warp's part holds, S MMAs reading it
        c.tq, c.tq_readers = {}, 0
        c.ktag, c.k_readers = [None] * self.KST, [0] * self.KST
        c.vtag, c.v_readers = [None] * self.VST, [0] * self.VST
        c.S, c.S_read = [None, None], [set(ALL), set(ALL)]
        c.DS, c.DS_readers = [dict(), dict()], [0, 0]
        c.acc, c.acc_read, c.acc_inflight = None, set(ALL), 0
        c.mmaq = {1: [], 2: []}
        return c

    def roles(self, c):
        return ([("producer", c, self.producer(c)), ("s_issuer", c, self.s_issuer(c)),
                 ("dq_issuer", c, self.dq_issuer(c))] + [(f"row{g}", c, self.rows(c, g)) for g in range(NE)])

    def complete_tma(self, job):
        c, kind, idx, tag = job
        if kind == "q":
            check(c.q_readers[idx] == 0, f"Q/dO slot {idx} overwritten while S/dP MMAs read it")
            check(c.q_copied[idx] >= ALL, f"Q/dO slot {idx} overwritten before every row warp copied its Q")
            c.qtag[idx], c.q_copied[idx] = tag, set()
            c.q[idx].complete_tx(1)
        elif kind == "k":
            check(c.k_readers[idx] == 0, f"K stage {idx} overwritten while read")
            c.ktag[idx] = tag
            c.kfull[idx].complete_tx(1)
        else:
            check(c.v_readers[idx] == 0, f"V stage {idx} overwritten while read")
            c.vtag[idx] = tag
            c.vfull[idx].complete_tx(1)

    def complete_mma(self, c, op):
        if op[0] == "commit":
            op[1].arrive()
        elif op[0] == "S":
            _, J, ks, vs, bb, qk, qs = op
            check(c.qtag[qs] == qk and c.ktag[ks] == J and c.vtag[vs] == J, f"S/dP({J}): operands changed")
            check(all(c.tq.get(g) == qk for g in range(NE)), f"S({J}) read a Q in TMEM that is not block {qk}'s")
            check(c.S_read[bb] >= ALL, f"S({J}) overwrote buffer {bb} before it was read")
            c.S[bb], c.S_read[bb] = J, set()
            c.q_readers[qs] -= 1
            c.tq_readers -= 1
            c.k_readers[ks] -= 1
            c.v_readers[vs] -= 1
        else:
            _, J, ks, bb, item, j = op
            check(c.ktag[ks] == J and all(c.DS[bb].get(g) == J for g in range(NE)), f"dQ({J}): operands changed")
            if j == 0:
                check(c.acc_read >= ALL, f"item {item}: dQ overwritten before the epilogue read it")
            else:
                check(c.acc == (item, j - 1), f"item {item}: accumulation chain broken at {j}")
            c.acc, c.acc_read = (item, j), set()
            c.k_readers[ks] -= 1
            c.DS_readers[bb] -= 1
            c.acc_inflight -= 1

    def producer(self, c):
        J = qn = n = 0
        nk = nv = 0  # K and V loads issued (J lags one of them when a V wait gives up)
        x = c.cid
        try:
            while True:
                slot = yield from self.publish(c, n)
                done = x >= len(self.items)
                c.slot[slot] = -1 if done else x
                c.item_full[slot].arrive()
                if done:
                    break
                xn = self.fetch_next()
                nkv = self.items[x]
                if nkv > 0:
                    qs = qn % self.QBUF
                    if qn >= self.QBUF and "qfree" not in self.drop:
                        yield from self.wait(c.qfree[qs], qn // self.QBUF - 1)
                    check(c.q_readers[qs] == 0, f"Q/dO load into slot {qs} issued while S/dP MMAs read it")
                    c.q[qs].expect_tx(1)
                    self.tma.append((c, "q", qs, qn))
                    qn += 1
                    for _ in range(nkv):
                        ks, vs = J % self.KST, J % self.VST
                        if J >= self.KST and "kempty" not in self.drop:
                            yield from self.wait(c.kempty[ks], J // self.KST - 1)
                        c.kfull[ks].expect_tx(1)
                        self.tma.append((c, "k", ks, J))
                        nk += 1
                        if J >= self.VST and "vempty" not in self.drop:
                            yield from self.wait(c.vempty[vs], J // self.VST - 1)
                        c.vfull[vs].expect_tx(1)
                        self.tma.append((c, "v", vs, J))
                        nv += 1
                        J += 1
                        yield ("step",)
                x = xn
                n += 1
        except Aborted:
            if "abort_drain" in self.drop:
                return
        for v in range(max(0, nk - self.KST), nk):
            yield from self.drain(c.kfull[v % self.KST], v // self.KST)
        for v in range(max(0, nv - self.VST), nv):
            yield from self.drain(c.vfull[v % self.VST], v // self.VST)
        for v in range(max(0, qn - self.QBUF), qn):
            yield from self.drain(c.q[v % self.QBUF], v // self.QBUF)

    def s_issuer(self, c):
        J = qn = n = 0
        try:
            while True:
                x = yield from self.take(c, n)
                n += 1
                if x < 0:
                    break
                nkv = self.items[x]
                if nkv == 0:
                    continue
                qs, qk = qn % self.QBUF, qn
                yield from self.wait(c.q[qs], qn // self.QBUF)
                if "qt" not in self.drop:
                    yield from self.wait(c.qt, qn)
                qn += 1
                for _ in range(nkv):
                    ks, vs, bb = J % self.KST, J % self.VST, J & 1
                    yield from self.wait(c.kfull[ks], J // self.KST)
                    if J >= 2 and "sfree" not in self.drop:
                        yield from self.wait(c.sfree[bb], (J >> 1) - 1)
                    yield from self.wait(c.vfull[vs], J // self.VST)
                    check(c.qtag[qs] == qk and c.ktag[ks] == J and c.vtag[vs] == J,
                          f"S({J}) issued on the wrong operands")
                    c.mmaq[1] += [("S", J, ks, vs, bb, qk, qs), ("commit", c.sfull[bb]), ("commit", c.vempty[vs])]
                    c.q_readers[qs] += 1
                    c.tq_readers += 1
                    c.k_readers[ks] += 1
                    c.v_readers[vs] += 1
                    J += 1
                    yield ("step",)
                c.mmaq[1].append(("commit", c.qfree[qs]))
        except Aborted:
            pass
        c.mmaq[1].append(("commit", c.sdrain))
        yield from self.mma_drain(c, c.sdrain)

    def dq_issuer(self, c):
        J = n = 0
        try:
            while True:
                x = yield from self.take(c, n)
                n += 1
                if x < 0:
                    break
                nkv = self.items[x]
                for j in range(nkv):
                    ks, bb = J % self.KST, J & 1
                    yield from self.wait(c.pready[bb], J >> 1)
                    yield from self.wait(c.kfull[ks], J // self.KST)
                    check(all(c.DS[bb].get(g) == J for g in range(NE)), f"dQ({J}) issued before dS was written")
                    c.mmaq[2] += [("DQ", J, ks, bb, x, j), ("commit", c.kempty[ks]), ("commit", c.pfree[bb])]
                    c.k_readers[ks] += 1
                    c.DS_readers[bb] += 1
                    c.acc_inflight += 1
                    J += 1
                    yield ("step",)
                if nkv > 0:
                    c.mmaq[2].append(("commit", c.dq))
        except Aborted:
            pass
        c.mmaq[2].append(("commit", c.gdrain))
        yield from self.mma_drain(c, c.gdrain)

    def rows(self, c, g):
        J = an = qc = 0

        def copy_q():
            nonlocal qc
            qs = qc % self.QBUF
            yield from self.wait(c.q[qs], qc // self.QBUF)
            check(c.qtag[qs] == qc, f"row{g}: copies the Q of block {c.qtag[qs]} for block {qc}")
            check(c.tq_readers == 0, f"row{g}: Q in TMEM overwritten while S MMAs read it")
            c.tq[g] = qc
            c.q_copied[qs].add(g)
            c.qt.arrive()
            qc += 1
            yield ("step",)

        try:
            x = yield from self.take(c, 0)
            if x >= 0 and self.items[x] > 0:
                yield from copy_q()
            n = 0
            while x >= 0:
                nkv = self.items[x]
                for _ in range(nkv):
                    bb, jn = J & 1, J >> 1
                    yield from self.wait(c.sfull[bb], jn)
                    check(c.S[bb] == J, f"row{g}: reads S({J}) while buffer {bb} holds S({c.S[bb]})")
                    c.S_read[bb].add(g)
                    c.sfree[bb].arrive()
                    yield ("step",)
                    if jn >= 1 and "pfree" not in self.drop:
                        yield from self.wait(c.pfree[bb], jn - 1)
                    check(c.DS_readers[bb] == 0, f"row{g}: dS buffer {bb} written while the dQ MMA reads it")
                    c.DS[bb][g] = J
                    c.pready[bb].arrive()
                    J += 1
                    yield ("step",)
                n += 1
                xn = yield from self.take(c, n)
                if xn >= 0 and self.items[xn] > 0:
                    yield from copy_q()
                if nkv > 0:
                    if "dq" not in self.drop:
                        yield from self.wait(c.dq, an)
                    an += 1
                    check(c.acc == (x, nkv - 1) and c.acc_inflight == 0,
                          f"row{g}: epilogue of item {x} sees {c.acc}")
                    c.acc_read.add(g)
                    if g == 0:
                        self.processed.append(x)
                    yield ("step",)
                x = xn
        except Aborted:
            pass

class FwdModel(Model):
    """attn_fwd_kernel (one query block per CTA, not persistent): `items` holds one entry, the
    length of the block's list.  K and V stream through 2-deep rings; S_j lands in TMEM buffer
    j % 2 and the softmax warps write P_j over it in place; O accumulates in TMEM and is
    rescaled by the softmax warps when a row maximum grows (a random choice per warp here)."""

    STAGES = 2
    NW = 4  # softmax warps

    def make_cta(self, cid):
        c = type("CTA", (), {})()
        c.cid = cid
        c.q = Bar("q", 1)
        c.kfull = [Bar(f"kfull{i}", 1) for i in range(self.STAGES)]
        c.vfull = [Bar(f"vfull{i}", 1) for i in range(self.STAGES)]
        c.kempty = [Bar(f"kempty{i}", 1) for i in range(self.STAGES)]
        c.vempty = [Bar(f"vempty{i}", 1) for i in range(self.STAGES)]
        c.sfull = [Bar(f"sfull{i}", 1) for i in range(2)]
        c.pfull = [Bar(f"pfull{i}", self.NW) for i in range(2)]
        c.odone, c.drain, c.sdrain = Bar("odone", 1), Bar("drain", 1), Bar("sdrain", 1)
        c.ktag, c.k_readers = [None] * self.STAGES, [0] * self.STAGES
        c.vtag, c.v_readers = [None] * self.STAGES, [0] * self.STAGES
        c.qtag = None
        # TMEM buffer b: ("S", j) after the S MMA, ("P", j, warps written) after the softmax
        c.buf, c.buf_readers = [None, None], [0, 0]
        c.S_read = [set(range(self.NW)), set(range(self.NW))]
        c.o_count, c.o_inflight = 0, 0  # P V products accumulated into O; P V MMAs in flight
        c.mmaq = {1: [], 2: []}
        return c

    def roles(self, c):
        return ([("producer", c, self.producer(c)), ("s_issuer", c, self.s_issuer(c)),
                 ("pv_issuer", c, self.pv_issuer(c))] + [(f"sm{w}", c, self.softmax(c, w)) for w in range(self.NW)])

    def complete_tma(self, job):
        c, kind, idx, tag = job
        if kind == "q":
            c.qtag = tag
            c.q.complete_tx(1)
        elif kind == "k":
            check(c.k_readers[idx] == 0, f"K stage {idx} overwritten while read")
            c.ktag[idx] = tag
            c.kfull[idx].complete_tx(1)
        else:
            check(c.v_readers[idx] == 0, f"V stage {idx} overwritten while read")
            c.vtag[idx] = tag
            c.vfull[idx].complete_tx(1)

    def complete_mma(self, c, op):
        if op[0] == "commit":
            op[1].arrive()
        elif op[0] == "S":
            _, j, st, b = op
            check(c.qtag == 0 and c.ktag[st] == j, f"S({j}): operands changed")
            check(c.buf_readers[b] == 0, f"S({j}) overwrote buffer {b} while P V read it")
            check(c.buf[b] is None or c.S_read[b] >= set(range(self.NW)) and c.buf[b][0] == "P",
                  f"S({j}) overwrote buffer {b} before its P was formed and used")
            c.buf[b], c.S_read[b] = ("S", j), set()
            c.k_readers[st] -= 1
        else:
            _, j, st, b = op
            check(c.vtag[st] == j and c.buf[b] == ("P", j, frozenset(range(self.NW))),
                  f"PV({j}): operands changed before completion")
            check(c.o_count == j, f"PV({j}) accumulated out of order")
            c.o_count += 1
            c.v_readers[st] -= 1
            c.buf_readers[b] -= 1
            c.o_inflight -= 1

    def producer(self, c):
        nkv = self.items[0]
        if nkv == 0:
            return
        c.q.expect_tx(1)
        self.tma.append((c, "q", 0, 0))
        nk = nv = 0  # K and V loads issued
        try:
            for j in range(nkv):
                st = j % self.STAGES
                if j >= self.STAGES and "kempty" not in self.drop:
                    yield from self.wait(c.kempty[st], j // self.STAGES - 1)
                check(c.k_readers[st] == 0, "K load issued while read")
                c.kfull[st].expect_tx(1)
                self.tma.append((c, "k", st, j))
                nk += 1
                if j >= self.STAGES and "vempty" not in self.drop:
                    yield from self.wait(c.vempty[st], j // self.STAGES - 1)
                check(c.v_readers[st] == 0, "V load issued while read")
                c.vfull[st].expect_tx(1)
                self.tma.append((c, "v", st, j))
                nv += 1
                yield ("step",)
        except Aborted:
            if "abort_drain" in self.drop:
                return
        yield from self.drain(c.q, 0)
        for j in range(max(0, nk - self.STAGES), nk):
            yield from self.drain(c.kfull[j % self.STAGES], j // self.STAGES)
        for j in range(max(0, nv - self.STAGES), nv):
            yield from self.drain(c.vfull[j % self.STAGES], j // self.STAGES)
    def s_issuer(self, c):
        nkv = self.items[0]
        if nkv == 0:
            return
        try:
            yield from self.wait(c.q, 0)
            for j in range(nkv):
                st, b = j % self.STAGES, j & 1
                yield from self.wait(c.kfull[st], j // self.STAGES)
                # P_{j-2} V_{j-2} read buffer b: it must have completed (same index as the V stage)
                if j >= 2 and "s_over_p" not in self.drop:
                    yield from self.wait(c.vempty[st], (j - 2) // self.STAGES)
                c.mmaq[1] += [("S", j, st, b), ("commit", c.sfull[b]), ("commit", c.kempty[st])]
                c.k_readers[st] += 1
                yield ("step",)
        except Aborted:
            pass
        c.mmaq[1].append(("commit", c.sdrain))
        yield from self.mma_drain(c, c.sdrain)
    def pv_issuer(self, c):
        nkv = self.items[0]
        if nkv == 0:
            return
        try:
            for j in range(nkv):
                st, b = j % self.STAGES, j & 1
                yield from self.wait(c.pfull[b], j >> 1)
                yield from self.wait(c.vfull[st], j // self.STAGES)
                check(c.buf[b] == ("P", j, frozenset(range(self.NW))), f"PV({j}) issued before P_{j} was written")
                c.mmaq[2] += [("PV", j, st, b), ("commit", c.vempty[st]), ("commit", c.odone)]
                c.v_readers[st] += 1
                c.buf_readers[b] += 1
                c.o_inflight += 1
                yield ("step",)
        except Aborted:
            pass
        c.mmaq[2].append(("commit", c.drain))
        yield from self.mma_drain(c, c.drain)
    def softmax(self, c, w):
        nkv = self.items[0]
        try:
            for j in range(nkv):
                b = j & 1
                yield from self.wait(c.sfull[b], j >> 1)
                check(c.buf[b] is not None and c.buf[b][:2] in (("S", j), ("P", j)),
                      f"sm{w}: reads S({j}) from {c.buf[b]}")
                c.S_read[b].add(w)
                if j > 0 and self.rng.random() < 0.3:
                    # rescale O: every earlier P V product must be in it and none in flight
                    if "odone" not in self.drop:
                        yield from self.wait(c.odone, j - 1)
                    check(c.o_count == j and c.o_inflight == 0, f"sm{w}: rescales O with {c.o_count} of {j} products")
                yield ("step",)
                check(c.buf_readers[b] == 0, f"sm{w}: writes P({j}) while P V reads buffer {b}")
                prev = c.buf[b][2] if c.buf[b][0] == "P" else frozenset()
                c.buf[b] = ("P", j, prev | {w})
                c.pfull[b].arrive()
                yield ("step",)
            if nkv > 0:
                yield from self.wait(c.drain, 0)
                if c.abort:  # the P V issuer gave up and completed `drain` early: no epilogue
                    raise Aborted()
                check(c.o_count == nkv and c.o_inflight == 0, f"sm{w}: epilogue sees {c.o_count} of {nkv} products")
                if w == 0:
                    self.processed.append(0)
        except Aborted:
            pass

def run_forward_trials(trials, drop=(), seed0=0, expire=False):
    """Random list lengths (including 0) on one CTA; returns the first error, or None.  With
    `expire`, waits expire at random (the abort path) and the epilogue is not required."""
    for t in range(seed0, seed0 + trials):
        rng = random.Random(t)
        nkv = rng.choice([0, 1, 2, 3, 4, 5, 7, 10])
        model = FwdModel(t, 1, [nkv], drop, expire)
        try:
            model.run()
            if not expire:
                check(model.processed == ([0] if nkv > 0 else []), "epilogue not reached")
        except ProtocolError as e:
            return f"trial {t}, list length {nkv}: {e}"
    return None


class PoolModel(Model):
    """pool_tc_kernel (mask builder): items are 128-token chunks taken by every CTA's producer
    from one counter (`items[x]` is unused: every chunk is one load and one MMA).  The chunks
    stream through a 2-deep stage ring; each chunk's index goes to a ring of 8 item slots read
    by the MMA warp and the four epilogue warps; the MMA of chunk n writes accumulator n % 2,
    which the epilogue warps read out before the MMA of chunk n + 2 may overwrite it."""

    STAGES, SLOTS, NW = 2, 8, 4
    SKIPS_EMPTY = False  # every chunk is pooled

    def make_cta(self, cid):
        c = type("CTA", (), {})()
        c.cid = cid
        c.full = [Bar(f"full{i}", 1) for i in range(self.STAGES)]
        c.empty = [Bar(f"empty{i}", 1) for i in range(self.STAGES)]
        c.acc = [Bar(f"acc{i}", 1) for i in range(2)]
        c.accfree = [Bar(f"accfree{i}", self.NW) for i in range(2)]
        c.drain = Bar("drain", 1)
        c.item_full = [Bar(f"item_full{i}", 1) for i in range(self.SLOTS)]
        c.item_free = [Bar(f"item_free{i}", 1 + self.NW) for i in range(self.SLOTS)]
        c.slot, c.slot_reads = [None] * self.SLOTS, [1 + self.NW] * self.SLOTS
        c.stage, c.stage_readers = [None] * self.STAGES, [0] * self.STAGES
        c.accv, c.acc_read = [None, None], [set(range(self.NW)), set(range(self.NW))]
        c.mmaq = {1: [], 2: []}
        return c

    def roles(self, c):
        return ([("producer", c, self.producer(c)), ("mma", c, self.mma(c))] +
                [(f"epi{w}", c, self.epilogue(c, w)) for w in range(self.NW)])

    def take(self, c, n):
        slot = n % self.SLOTS
        yield from self.wait(c.item_full[slot], n // self.SLOTS)
        x = c.slot[slot]
        c.slot_reads[slot] += 1
        c.item_free[slot].arrive()
        return x

    def complete_tma(self, job):
        c, kind, st, x = job
        check(c.stage_readers[st] == 0, f"stage {st} overwritten while the MMA reads it")
        c.stage[st] = x
        c.full[st].complete_tx(1)

    def complete_mma(self, c, op):
        if op[0] == "commit":
            op[1].arrive()
            return
        _, n, st, ab, x = op
        check(c.stage[st] == x, f"MMA of chunk {x}: stage {st} holds {c.stage[st]}")
        check(c.acc_read[ab] >= set(range(self.NW)), f"accumulator {ab} overwritten before it was read out")
        c.accv[ab], c.acc_read[ab] = x, set()
        c.stage_readers[st] -= 1

    def producer(self, c):
        n = loads = 0
        try:
            while True:
                slot = n % self.SLOTS
                if n >= self.SLOTS and "item_free" not in self.drop:
                    yield from self.wait(c.item_free[slot], n // self.SLOTS - 1)
                x = self.counter
                self.counter += 1
                done = x >= len(self.items)
                check(c.slot_reads[slot] == 1 + self.NW, f"item slot {slot} overwritten before every role read it")
                c.slot[slot], c.slot_reads[slot] = (-1 if done else x), 0
                c.item_full[slot].arrive()
                if done:
                    break
                st = n % self.STAGES
                if n >= self.STAGES and "empty" not in self.drop:
                    yield from self.wait(c.empty[st], n // self.STAGES - 1)
                c.full[st].expect_tx(1)
                self.tma.append((c, "x", st, x))
                loads += 1
                n += 1
                yield ("step",)
        except Aborted:
            if "abort_drain" in self.drop:
                return
        for v in range(max(0, loads - self.STAGES), loads):
            yield from self.drain(c.full[v % self.STAGES], v // self.STAGES)

    def mma(self, c):
        n = 0
        try:
            while True:
                x = yield from self.take(c, n)
                if x < 0:
                    break
                st, ab = n % self.STAGES, n & 1
                yield from self.wait(c.full[st], n // self.STAGES)
                if n >= 2 and "accfree" not in self.drop:
                    yield from self.wait(c.accfree[ab], (n >> 1) - 1)
                check(c.stage[st] == x, f"MMA of chunk {x} issued on stage {st} holding {c.stage[st]}")
                c.mmaq[1] += [("MMA", n, st, ab, x), ("commit", c.empty[st]), ("commit", c.acc[ab])]
                c.stage_readers[st] += 1
                n += 1
                yield ("step",)
        except Aborted:
            pass
        c.mmaq[1].append(("commit", c.drain))
        yield from self.mma_drain(c, c.drain)

    def epilogue(self, c, w):
        n = 0
        try:
            while True:
                x = yield from self.take(c, n)
                if x < 0:
                    break
                ab = n & 1
                yield from self.wait(c.acc[ab], n >> 1)
                check(c.accv[ab] == x, f"epi{w}: accumulator {ab} holds chunk {c.accv[ab]}, not {x}")
                c.acc_read[ab].add(w)
                c.accfree[ab].arrive()
                if w == 0:
                    self.processed.append(x)
                n += 1
                yield ("step",)
        except Aborted:
            pass


def run_trials(model_cls, trials, drop=(), seed0=0, expire=False):
    """Random item lists (with empty items) on 1-3 CTAs; returns the first error, or None.
    With `expire`, waits expire at random (the abort path) and items may stay unfinished."""
    for t in range(seed0, seed0 + trials):
        rng = random.Random(t)
        nitems = rng.randint(1, 12)
        items = [rng.choice([0, 0, 1, 2, 3, 4, 5, 8]) for _ in range(nitems)]
        model = model_cls(t, rng.randint(1, min(3, nitems)), items, drop, expire)
        try:
            model.run()
            if not expire:
                want = sorted(x for x in range(nitems) if items[x] > 0 or not model_cls.SKIPS_EMPTY)
                check(sorted(model.processed) == want, f"items processed {sorted(model.processed)}, want {want}")
        except ProtocolError as e:
            return f"trial {t}, items {items}: {e}"
    return None
