"""A model of the tensor-core backward kernel's per-CTA barrier protocol, run under random schedules.

The main kernel (csrc/bwd_sm103.cu) is a set of warp roles that hand TMEM buffers and shared-memory
tiles to one another through mbarriers waited on by phase parity.  A parity wait is only correct
while its barrier is at most one phase from the awaited one: behind by one, it passes at once;
ahead by two, it waits for a phase that may never come.  Two earlier bugs of these kernels were
exactly that (the forward epilogue, and a staged-dQ barrier shared by two dS tiles).

This model restates the protocol as the kernel runs it (the same roles, waits, arrivals, commits
and parity formulas) with the data movements reduced to labels ("this buffer holds S(3)"), and
runs it under many random interleavings, with every MMA queue, TMA load and bulk reduce completing
at a random later time.  It checks that
  * every wait sees its barrier either at the awaited phase (blocks) or one past it (passes),
  * no schedule deadlocks,
  * every read of a TMEM buffer or shared tile finds the data the reader expects.
It covers the configurations the backward has: two TMEM buffers, one MMA issuer and separate Q and
dO rings (d = 128), three buffers, two dS tiles, two issuers and one ring for both tiles (d = 64),
each with the drain's first thread or (the deterministic instance) a reduce warp issuing the dQ
reduce-adds; and the forward kernel (csrc/fwd_sm103.cu) with three S buffers (d <= 128) or two
(d = 256), one item per CTA or (the persistent kernel) a sequence of items.

The model is not generated from the kernel: a change to the kernel's protocol needs the same change
here, and this test then says whether the new protocol is sound.
"""
import random

import pytest


class ProtocolError(AssertionError):
    pass


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.completed = name, count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.completed += 1
            self.pending = self.count


class Model:
    """One CTA of the backward kernel with n_it iterations."""

    def __init__(self, n_it, d, det, rng):
        self.n, self.rng, self.det = n_it, rng, det
        self.NBUF = 3 if d == 64 else 2
        self.NDS = 2 if d == 64 else 1
        self.STAGES = 3 if d == 64 else 2
        self.d = d
        self.split = self.NBUF == 3          # two MMA issuers
        self.use_red = det                    # reduce warp (deterministic instance)
        # d = 128: separate Q and dO rings (the drain stages half of dQ in the dO tile, whose
        # "empty" then takes the MMA commit and the drain's / reduce warp's arrival); d = 64: one
        # pair of barriers per stage for both tiles
        self.split_ring = d == 128
        self.bars = {}

        def bar(name, count=1):
            self.bars[name] = Bar(name, count)

        for name in ("KV", "DP_FULL", "DS_READY", "DQ_FULL", "DQ_EMPTY", "G3", "G4", "ACC", "FINAL",
                     "FINAL_A"):
            bar(name)
        for k in range(3):
            bar(f"S_FULL{k}")
            bar(f"P_READY{k}")
            bar(f"YFREE{k}")
        for t in range(2):
            bar(f"DS_EMPTY{t}")
            bar(f"DQ_STAGED{t}")
        for s in range(self.STAGES):
            bar(f"FULLQ{s}")
            bar(f"EMPTYQ{s}")
            if self.split_ring:
                bar(f"FULLDO{s}")
                bar(f"EMPTYDO{s}", 2)
            else:  # the same barriers serve both tiles
                self.bars[f"FULLDO{s}"] = self.bars[f"FULLQ{s}"]
                self.bars[f"EMPTYDO{s}"] = self.bars[f"EMPTYQ{s}"]
        self.res = {}            # resource -> label of its content
        self.mma_q = {}          # issuer -> list of queued ops (executed in order)
        self.async_ops = []      # TMA loads and bulk reads in flight
        self.async_done = set()  # handles of completed bulk reads
        self.handle = 0

    # ---- the kernel's index helpers
    def xb(self, i):
        return (2 * i) % 3 if self.NBUF == 3 else (i & 1)

    def yb(self, i):
        return (2 * i + 1) % 3 if self.NBUF == 3 else ((i & 1) ^ 1)

    def sp_slot(self, i):
        return (2 * i) % 3 if self.NBUF == 3 else 0

    def sp_phase(self, i):  # the phase index whose parity the kernel waits for
        return i // 3 if self.NBUF == 3 else i

    def dt(self, i):
        return (i & 1) if self.NDS == 2 else 0

    # ---- primitives used by the roles (generators yield these requests)
    @staticmethod
    def wait(bar, phase):
        return ("wait", bar, phase)

    @staticmethod
    def arrive(bar):
        return ("arrive", bar)

    # time passes inside a role (a TMEM load, the arithmetic, shared-memory stores): other roles,
    # MMAs and copies may run meanwhile
    STEP = ("step",)

    def expect(self, resource, label):
        got = self.res.get(resource)
        if got != label:
            raise ProtocolError(f"{resource} holds {got}, expected {label}")

    def put(self, resource, label):
        self.res[resource] = label

    # ---- roles
    def producer(self):
        """K, V, then the Q tiles with the lse2 / D rows (and, one shared ring, the dO tiles)."""
        self.async_ops.append(("tma", [("K", "K"), ("V", "V")], "KV"))
        for it in range(self.n):
            s = it % self.STAGES
            if it >= self.STAGES:
                yield self.wait(f"EMPTYQ{s}", it // self.STAGES - 1)
            writes = [(f"Q{s}", ("Q", it)), (f"row{s}", ("row", it))]
            if not self.split_ring:
                writes.append((f"dO{s}", ("dO", it)))
            self.async_ops.append(("tma", writes, f"FULLQ{s}"))
        # the producer then waits for its loads to land (drain_wait): modelled by the loads
        # completing before the CTA ends, which the scheduler guarantees

    def producer_do(self):
        """The dO ring of the split case: the kernel's one producer thread polls both "empty"
        barriers without blocking on either, which is two independent streams."""
        for it in range(self.n):
            s = it % self.STAGES
            if it >= self.STAGES:
                yield self.wait(f"EMPTYDO{s}", it // self.STAGES - 1)
            self.async_ops.append(("tma", [(f"dO{s}", ("dO", it))], f"FULLDO{s}"))

    def mma_op(self, issuer, reads, writes):
        return ("mma", issuer, reads, writes)

    def commit(self, issuer, bar):
        return ("commit", issuer, bar)

    def gemm_s(self, issuer, i, buf):      # S^T(i) = K Q(i)^T into buf
        return self.mma_op(issuer, [("K", "K"), (f"Q{i % self.STAGES}", ("Q", i))], [(f"buf{buf}", ("S", i))])

    def gemm_dp(self, issuer, i, buf):     # dP^T(i) = V dO(i)^T into buf
        return self.mma_op(issuer, [("V", "V"), (f"dO{i % self.STAGES}", ("dO", i))], [(f"buf{buf}", ("dP", i))])

    def issuer_sd(self, who):
        """S and dP products: the single issuer's first part or warp 13 of the pair."""
        yield self.wait("KV", 0)
        yield self.wait("FULLQ0", 0)
        yield self.gemm_s(who, 0, self.xb(0))
        yield self.commit(who, f"S_FULL{self.sp_slot(0)}")
        yield self.wait("FULLDO0", 0)
        yield self.gemm_dp(who, 0, self.yb(0))
        yield self.commit(who, "DP_FULL")

    def issuer_single(self):
        yield from self.issuer_sd("A")
        yield from self.issuer_g("A", single=True)

    def issuer_a(self):
        yield from self.issuer_sd("A")
        for it in range(self.n):
            if it + 1 < self.n:
                s1 = (it + 1) % self.STAGES
                yield self.wait(f"FULLQ{s1}", (it + 1) // self.STAGES)
                if it > 0:
                    yield self.wait(f"YFREE{self.yb(it - 1)}", (it - 1) // 3)
                yield self.gemm_s("A", it + 1, self.xb(it + 1))
                yield self.commit("A", f"S_FULL{self.sp_slot(it + 1)}")
                yield self.wait("DQ_EMPTY", it)
                yield self.wait(f"FULLDO{s1}", (it + 1) // self.STAGES)
                yield self.gemm_dp("A", it + 1, self.xb(it))
                yield self.commit("A", "DP_FULL")
        yield self.commit("A", "FINAL_A")
        yield self.wait("FINAL_A", 0)

    def issuer_g(self, who, single=False):
        """dV, dQ, dK products (and, single issuer, the next S and dP)."""
        for it in range(self.n):
            s = it % self.STAGES
            X, Y = f"buf{self.xb(it)}", f"buf{self.yb(it)}"
            yield self.wait(f"P_READY{self.sp_slot(it)}", self.sp_phase(it))
            yield self.mma_op(who, [(X, ("P", it)), (f"dO{s}", ("dO", it))], [])          # dV
            yield self.commit(who, "G3")
            yield self.wait("DS_READY", it)
            yield self.wait("G3", it)
            yield self.mma_op(who, [(f"dstile{self.dt(it)}", ("dS", it)), ("K", "K")], [(X, ("dQ", it))])  # dQ
            yield self.commit(who, "DQ_FULL")
            yield self.mma_op(who, [(Y, ("dS", it)), (f"Q{s}", ("Q", it))], [])            # dK
            yield self.commit(who, f"YFREE{self.yb(it)}" if self.NBUF == 3 else "G4")
            yield self.commit(who, f"EMPTYQ{s}")
            if self.split_ring:
                yield self.commit(who, f"EMPTYDO{s}")
            if single and it + 1 < self.n:
                s1 = (it + 1) % self.STAGES
                yield self.wait(f"FULLQ{s1}", (it + 1) // self.STAGES)
                yield self.wait("G4", it)
                yield self.gemm_s(who, it + 1, self.yb(it))
                yield self.commit(who, f"S_FULL{self.sp_slot(it + 1)}")
                yield self.wait("DQ_EMPTY", it)
                yield self.wait(f"FULLDO{s1}", (it + 1) // self.STAGES)
                yield self.gemm_dp(who, it + 1, self.xb(it))
                yield self.commit(who, "DP_FULL")
        yield self.commit(who, "ACC")
        yield self.commit(who, "FINAL")
        yield self.wait("FINAL", 0)

    def softmax(self):
        for it in range(self.n):
            s = it % self.STAGES
            X, Y = f"buf{self.xb(it)}", f"buf{self.yb(it)}"
            yield self.wait(f"FULLQ{s}", it // self.STAGES)  # Q with the lse2 / D rows
            yield self.wait(f"S_FULL{self.sp_slot(it)}", self.sp_phase(it))
            self.expect(f"row{s}", ("row", it))        # LSE row
            self.expect(X, ("S", it))
            yield self.STEP
            self.put(X, ("P", it))
            yield self.STEP
            yield self.arrive(f"P_READY{self.sp_slot(it)}")
            yield self.wait("DP_FULL", it)
            if it >= self.NDS:
                yield self.wait(f"DS_EMPTY{self.dt(it)}", (it - self.NDS) // self.NDS)
            self.expect(f"row{s}", ("row", it))        # D row
            self.expect(Y, ("dP", it))
            yield self.STEP
            self.put(Y, ("dS", it))
            tile = f"dstile{self.dt(it)}"
            self.put(tile, ("dS", it))
            yield self.STEP
            yield self.arrive("DS_READY")
        if self.n > 0:
            yield self.wait("ACC", 0)

    def reduce_staged(self, it):
        """The bulk reduce-adds of iteration it and the releases after TMA read them (one thread)."""
        s = it % self.STAGES
        tile = f"dstile{self.dt(it)}"
        h1 = self.bulk([(tile, ("dQ", it))])
        if self.d == 128:
            h2 = self.bulk([(f"dO{s}", ("dQhi", it))])
            yield ("wait_async", h1)
            yield self.arrive(f"DS_EMPTY{self.dt(it)}")
            yield ("wait_async", h2)
            yield self.arrive(f"EMPTYDO{s}")
        else:
            yield ("wait_async", h1)
            yield self.arrive(f"DS_EMPTY{self.dt(it)}")

    def bulk(self, reads):
        self.handle += 1
        self.async_ops.append(("bulk", reads, self.handle))
        return self.handle

    def drain(self):
        for it in range(self.n):
            s = it % self.STAGES
            X = f"buf{self.xb(it)}"
            yield self.wait("DQ_FULL", it)
            self.expect(X, ("dQ", it))
            yield self.arrive("DQ_EMPTY")
            yield self.STEP
            tile = f"dstile{self.dt(it)}"
            # staging overwrites dS(it), which the dQ product has read (B_DQ_FULL), and at
            # d = 128 the dO tile, which the dV product has read
            self.expect(tile, ("dS", it))
            self.put(tile, ("dQ", it))
            if self.d == 128:
                self.expect(f"dO{s}", ("dO", it))
                self.put(f"dO{s}", ("dQhi", it))
            yield self.STEP
            if self.use_red:
                yield self.arrive(f"DQ_STAGED{self.dt(it)}")
            else:
                yield from self.reduce_staged(it)

    def reducer(self):
        for it in range(self.n):
            yield self.wait(f"DQ_STAGED{self.dt(it)}", it // self.NDS)
            yield from self.reduce_staged(it)

    def make_roles(self):
        roles = {"producer": self.producer(), "softmax": self.softmax(), "drain": self.drain()}
        if self.split_ring:
            roles["producer_do"] = self.producer_do()
        if self.n > 0:
            if self.split:
                roles["mma_a"] = self.issuer_a()
                roles["mma_b"] = self.issuer_g("B")
            else:
                roles["mma"] = self.issuer_single()
        if self.use_red:
            roles["reducer"] = self.reducer()
        return roles

    # ---- scheduler
    def run(self):
        roles = self.make_roles()
        blocked = {name: None for name in roles}  # pending request of each role
        for name in list(roles):
            self.advance(roles, blocked, name, None)
        steps = 0
        while roles or any(self.mma_q.values()) or self.async_ops:
            steps += 1
            if steps > 100000:
                raise ProtocolError("no progress")
            choices = []
            for name, req in blocked.items():
                if name in roles and self.ready(req):
                    choices.append(("role", name))
            for who, q in self.mma_q.items():
                if q:
                    choices.append(("mma", who))
            for k in range(len(self.async_ops)):
                choices.append(("async", k))
            if not choices:
                raise ProtocolError("deadlock: " + ", ".join(f"{n} at {blocked[n]}" for n in roles))
            kind, key = self.rng.choice(choices)
            if kind == "role":
                self.advance(roles, blocked, key, blocked[key])
            elif kind == "mma":
                self.exec_mma(key)
            else:
                self.exec_async(self.async_ops.pop(key))
        return True

    def ready(self, req):
        if req[0] == "wait":
            b = self.bars[req[1]]
            if b.completed == req[2] + 1:
                return True
            if b.completed == req[2]:
                return False
            raise ProtocolError(f"wait on {req[1]} for phase {req[2]} while {b.completed} phases completed")
        if req[0] == "wait_async":
            return req[1] in self.async_done
        if req[0] == "step":
            return True
        raise AssertionError(req)

    def advance(self, roles, blocked, name, _req):
        gen = roles[name]
        while True:
            try:
                req = next(gen)
            except StopIteration:
                del roles[name]
                return
            if req[0] == "step":
                blocked[name] = req
                return
            if req[0] in ("wait", "wait_async"):
                if req[0] == "wait":
                    self.ready(req)  # raises on a wrong phase even if it would block
                blocked[name] = req
                if self.ready(req):
                    continue
                return
            if req[0] == "arrive":
                self.bars[req[1]].arrive()
            elif req[0] in ("mma", "mma_pv", "commit"):
                self.mma_q.setdefault(req[1], []).append(req)
            else:
                raise AssertionError(req)

    def exec_mma(self, who):
        op = self.mma_q[who].pop(0)
        if op[0] == "commit":
            self.bars[op[2]].arrive()
            return
        _, _, reads, writes = op
        for r, label in reads:
            self.expect(r, label)
        for r, label in writes:
            self.put(r, label)

    def exec_async(self, op):
        if op[0] == "tma":
            for r, label in op[1]:
                self.put(r, label)
            self.bars[op[2]].arrive()
        else:
            for r, label in op[1]:
                self.expect(r, label)
            self.async_done.add(op[2])


CONFIGS = [(128, False), (128, True), (64, False), (64, True)]


@pytest.mark.parametrize("d,det", CONFIGS, ids=[f"d{d}-{'det' if det else 'default'}" for d, det in CONFIGS])
def test_protocol_sound_under_random_schedules(d, det):
    rng = random.Random(1000 + d + det)
    for trial in range(400):
        n_it = rng.choice([1, 2, 3, 4, 5, 6, 7, 9])
        Model(n_it, d, det, random.Random(rng.random())).run()


def test_model_catches_a_shared_staged_barrier_with_two_tiles():
    # the incident: one staged-dQ barrier for both dS tiles lets the drain run two phases ahead
    # of the reduce warp; the model must find schedules where that happens
    class Shared(Model):
        def drain(self):
            for req in super().drain():
                if req == ("arrive", "DQ_STAGED1"):
                    req = ("arrive", "DQ_STAGED0")
                yield req

        def reducer(self):
            for it in range(self.n):
                yield self.wait("DQ_STAGED0", it)
                yield from self.reduce_staged(it)

    rng = random.Random(7)
    failures = 0
    for _ in range(400):
        try:
            Shared(7, 64, True, random.Random(rng.random())).run()
        except ProtocolError:
            failures += 1
    assert failures > 0


def test_model_catches_a_missing_wait():
    # S(i+1) issued without waiting for the dK product that still reads that buffer
    class NoYfree(Model):
        def issuer_a(self):
            for req in super().issuer_a():
                if req[0] == "wait" and req[1].startswith("YFREE"):
                    continue
                yield req

    rng = random.Random(11)
    failures = 0
    for _ in range(400):
        try:
            NoYfree(7, 64, False, random.Random(rng.random())).run()
        except ProtocolError:
            failures += 1
    assert failures > 0


def _fails(model_cls, d, det, n_it=7, trials=400, seed=13):
    rng = random.Random(seed)
    for _ in range(trials):
        try:
            model_cls(n_it, d, det, random.Random(rng.random())).run()
        except ProtocolError:
            return True
    return False


def test_model_catches_a_skipped_ds_tile_wait():
    # dS(i) written into a tile whose previous dQ staging the bulk reduce has not read yet
    class NoDsEmpty(Model):
        def softmax(self):
            for req in super().softmax():
                if req[0] == "wait" and req[1].startswith("DS_EMPTY"):
                    continue
                yield req

    # at d = 64 in the default mode the drain's own order implies the wait (it frees dQ(i+1)'s
    # buffer only after the reduce of iteration i read its tile); with the reduce warp it does not
    assert _fails(NoDsEmpty, 64, True) and _fails(NoDsEmpty, 128, False)
    assert not _fails(NoDsEmpty, 64, False, trials=100)


def test_model_catches_one_s_and_p_barrier_with_three_buffers():
    # with two issuers the softmax can finish P(i+1) before the dV issuer waited for P(i)
    class SharedSP(Model):
        def sp_slot(self, i):
            return 0

        def sp_phase(self, i):
            return i

    assert _fails(SharedSP, 64, False)


def test_model_catches_dp_issued_before_the_drain_read_dq():
    # dP(i+1) overwrites the buffer that still holds dQ(i) for the drain
    class NoDqEmpty(Model):
        def issuer_g(self, who, single=False):
            for req in super().issuer_g(who, single):
                if req[0] == "wait" and req[1] == "DQ_EMPTY":
                    continue
                yield req

        def issuer_a(self):
            for req in super().issuer_a():
                if req[0] == "wait" and req[1] == "DQ_EMPTY":
                    continue
                yield req

    assert _fails(NoDqEmpty, 128, False) and _fails(NoDqEmpty, 64, False)


def test_model_reads_one_threads_mmas_in_order():
    # with one issuing thread its MMAs run in issue order, so S(i+1) cannot overtake the dK
    # product of iteration i even without the wait the kernel keeps for it (the model agrees:
    # dropping that wait is not a protocol error for the single issuer)
    class NoG4(Model):
        def issuer_g(self, who, single=False):
            for req in super().issuer_g(who, single):
                if req[0] == "wait" and req[1] == "G4":
                    continue
                yield req

    assert not _fails(NoG4, 128, False, trials=100)


class FwdModel(Model):
    """One CTA of the tensor-core forward (csrc/fwd_sm103.cu) over n key tiles: a TMA warp
    (Q once, K / V through a ring), a warp issuing S(j) = Q K(j)^T into TMEM buffer j % NB, a warp
    issuing O += P(j) V(j) from that buffer, and the softmax warps (one actor here), which turn
    S(j) into P(j) in place, sometimes rescale the O rows in TMEM (after P V(j-1) completed) and
    finally read O.  NB = 3 S buffers for d <= 128, 2 for d = 256."""

    def __init__(self, n_tiles, d, rng):
        self.n, self.rng, self.d = n_tiles, rng, d
        self.NB = 3 if d <= 128 else 2
        self.STAGES = {64: 4, 128: 3, 256: 2}[d]
        self.bars = {}
        for name in ("Q", "FINAL"):
            self.bars[name] = Bar(name, 1)
        for k in range(3):
            for kind in ("S", "P", "PV"):
                self.bars[f"{kind}{k}"] = Bar(f"{kind}{k}", 1)
        for st in range(self.STAGES):
            self.bars[f"FULL{st}"] = Bar(f"FULL{st}", 1)
            self.bars[f"EMPTY{st}"] = Bar(f"EMPTY{st}", 1)
        self.res = {"O": 0}      # O: number of P V products accumulated
        self.mma_q, self.async_ops, self.async_done, self.handle = {}, [], set(), 0

    def make_roles(self):
        roles = {"tma": self.f_tma(), "softmax": self.f_softmax()}
        if self.n > 0:
            roles["s_issuer"] = self.f_s_issuer()
            roles["pv_issuer"] = self.f_pv_issuer()
        return roles

    def f_tma(self):
        self.async_ops.append(("tma", [("Qt", "Q")], "Q"))
        for j in range(self.n):
            st = j % self.STAGES
            if j >= self.STAGES:
                yield self.wait(f"EMPTY{st}", j // self.STAGES - 1)
            self.async_ops.append(("tma", [(f"K{st}", ("K", j)), (f"V{st}", ("V", j))], f"FULL{st}"))

    def f_s_issuer(self):
        yield self.wait("Q", 0)
        for j in range(self.n):
            st, b = j % self.STAGES, j % self.NB
            yield self.wait(f"FULL{st}", j // self.STAGES)
            if j >= self.NB:  # P V(j - NB) has read P out of buffer b
                yield self.wait(f"PV{b}", j // self.NB - 1)
            yield ("mma", "S", [("Qt", "Q"), (f"K{st}", ("K", j))], [(f"sbuf{b}", ("S", j))])
            yield ("commit", "S", f"S{b}")

    def f_pv_issuer(self):
        for j in range(self.n):
            st, b = j % self.STAGES, j % self.NB
            yield self.wait(f"P{b}", j // self.NB)
            yield ("mma_pv", "PV", j, b, st)
            yield ("commit", "PV", f"PV{b}")
            yield ("commit", "PV", f"EMPTY{st}")  # S(j) completed before P(j)
        yield ("commit", "PV", "FINAL")
        yield self.wait("FINAL", 0)

    def f_softmax(self):
        for j in range(self.n):
            b = j % self.NB
            yield self.wait(f"S{b}", j // self.NB)
            self.expect(f"sbuf{b}", ("S", j))
            yield self.STEP
            self.put(f"sbuf{b}", ("P", j))
            if j > 0 and self.rng.random() < 0.5:  # the running max moved: rescale O
                yield self.wait(f"PV{(j - 1) % self.NB}", (j - 1) // self.NB)
                self.expect("O", j)
                yield self.STEP
                self.expect("O", j)
            yield self.arrive(f"P{b}")
        if self.n > 0:
            yield from self.f_epilogue()
        self.expect("O", self.n)

    def f_epilogue(self):
        yield self.wait("FINAL", 0)

    def exec_mma(self, who):
        op = self.mma_q[who][0]
        if op[0] == "mma_pv":
            self.mma_q[who].pop(0)
            _, _, j, b, st = op
            self.expect(f"sbuf{b}", ("P", j))
            self.expect(f"V{st}", ("V", j))
            self.expect("O", j)
            self.put("O", j + 1)
            return
        super().exec_mma(who)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_forward_protocol_sound_under_random_schedules(d):
    rng = random.Random(2000 + d)
    for _ in range(400):
        FwdModel(rng.choice([1, 2, 3, 4, 5, 7, 9]), d, random.Random(rng.random())).run()


def test_forward_model_catches_one_shared_pv_barrier():
    # one P V barrier for all S buffers (the design before the per-buffer ones): a parity wait
    # for P V(j) can see the barrier a phase behind (P V(j-1) pending: the old epilogue read O
    # early) or ahead
    class SharedPV(FwdModel):
        def f_s_issuer(self):
            for req in super().f_s_issuer():
                if req[0] == "wait" and req[1].startswith("PV"):
                    req = self.wait("PV0", req[2] * self.NB + int(req[1][2:]))
                yield req

        def f_pv_issuer(self):
            for req in super().f_pv_issuer():
                if req[0] == "commit" and req[2].startswith("PV"):
                    req = ("commit", req[1], "PV0")
                yield req

        def f_softmax(self):
            for req in super().f_softmax():
                if req[0] == "wait" and req[1].startswith("PV"):
                    req = self.wait("PV0", req[2] * self.NB + int(req[1][2:]))
                yield req

        def f_epilogue(self):
            yield self.wait("PV0", self.n - 1)

    rng = random.Random(5)
    caught = 0
    for _ in range(400):
        try:
            SharedPV(rng.choice([4, 5, 7]), 128, random.Random(rng.random())).run()
        except ProtocolError:
            caught += 1
    assert caught > 0


class PersistentFwdModel(FwdModel):
    """One CTA of the persistent forward (csrc/fwd_sm103.cu, fwd_sm103_persistent_kernel) over a
    list of items, each with its number of key tiles (0 for an item whose rows see no key, which
    every role skips).  The producer thread's two polled streams (Q tiles, gated on the S issuer's
    commit after an item's last S product; K / V tiles through the ring, running on into the next
    item) are two actors here.  The P V issuer commits "O full" after an item's last product and
    waits for "O free" (the softmax warps have read O) before the next item's first product, which
    overwrites O.  Per-item barriers count the items with work, per-tile ones all key tiles."""

    def __init__(self, items, d, rng):
        super().__init__(sum(items), d, rng)
        self.items = items
        for name in ("QE", "OFULL", "OFREE"):
            self.bars[name] = Bar(name, 1)
        self.res = {"O": None}

    def active(self):
        return [(k, c) for k, c in enumerate(self.items) if c > 0]

    def make_roles(self):
        roles = {"tma_q": self.p_q(), "tma_kv": self.p_kv(), "softmax": self.p_softmax()}
        if self.n > 0:
            roles["s_issuer"] = self.p_s()
            roles["pv_issuer"] = self.p_pv()
        return roles

    def p_q(self):
        for a, (k, _) in enumerate(self.active()):
            if a > 0:
                yield self.wait("QE", a - 1)
            self.async_ops.append(("tma", [("Qt", ("Q", k))], "Q"))

    def p_kv(self):
        jg = 0
        for _, c in self.active():
            for _ in range(c):
                st = jg % self.STAGES
                if jg >= self.STAGES:
                    yield self.wait(f"EMPTY{st}", jg // self.STAGES - 1)
                self.async_ops.append(("tma", [(f"K{st}", ("K", jg)), (f"V{st}", ("V", jg))], f"FULL{st}"))
                jg += 1

    def p_s(self):
        jg = 0
        for a, (k, c) in enumerate(self.active()):
            yield self.wait("Q", a)
            for _ in range(c):
                st, b = jg % self.STAGES, jg % self.NB
                yield self.wait(f"FULL{st}", jg // self.STAGES)
                if jg >= self.NB:
                    yield self.wait(f"PV{b}", jg // self.NB - 1)
                yield ("mma", "S", [("Qt", ("Q", k)), (f"K{st}", ("K", jg))], [(f"sbuf{b}", ("S", jg))])
                yield ("commit", "S", f"S{b}")
                jg += 1
            yield ("commit", "S", "QE")

    def p_pv(self):
        jg = 0
        for a, (k, c) in enumerate(self.active()):
            for j in range(c):
                st, b = jg % self.STAGES, jg % self.NB
                yield self.wait(f"P{b}", jg // self.NB)
                if j == 0 and a > 0:
                    yield self.wait("OFREE", a - 1)
                yield ("mma_pv", "PV", jg, b, st, k, j)
                yield ("commit", "PV", f"PV{b}")
                yield ("commit", "PV", f"EMPTY{st}")
                jg += 1
            yield ("commit", "PV", "OFULL")
        yield ("commit", "PV", "FINAL")
        yield self.wait("FINAL", 0)

    def p_softmax(self):
        jg, a = 0, 0
        for k, c in enumerate(self.items):
            for j in range(c):
                b = jg % self.NB
                yield self.wait(f"S{b}", jg // self.NB)
                self.expect(f"sbuf{b}", ("S", jg))
                yield self.STEP
                self.put(f"sbuf{b}", ("P", jg))
                if j > 0 and self.rng.random() < 0.5:  # the running max moved: rescale O
                    yield self.wait(f"PV{(jg - 1) % self.NB}", (jg - 1) // self.NB)
                    self.expect("O", (k, j))
                    yield self.STEP
                    self.expect("O", (k, j))
                yield self.arrive(f"P{b}")
                jg += 1
            if c > 0:  # epilogue: read O, then let the next item's first P V product in
                yield self.wait("OFULL", a)
                self.expect("O", (k, c))
                yield self.STEP
                self.expect("O", (k, c))
                yield self.arrive("OFREE")
                a += 1

    def exec_mma(self, who):
        op = self.mma_q[who][0]
        if op[0] == "mma_pv":
            self.mma_q[who].pop(0)
            _, _, jg, b, st, k, j = op
            self.expect(f"sbuf{b}", ("P", jg))
            self.expect(f"V{st}", ("V", jg))
            if j > 0:
                self.expect("O", (k, j))
            self.put("O", (k, j + 1))
            return
        Model.exec_mma(self, who)


def _random_items(rng):
    return [rng.choice([0, 1, 1, 2, 3, 4, 6]) for _ in range(rng.choice([1, 2, 3, 4, 6]))]


@pytest.mark.parametrize("d", [64, 128])
def test_persistent_forward_protocol_sound_under_random_schedules(d):
    rng = random.Random(3000 + d)
    for _ in range(400):
        PersistentFwdModel(_random_items(rng), d, random.Random(rng.random())).run()


def _persistent_fails(model_cls, d=128, trials=400, seed=17):
    rng = random.Random(seed)
    for _ in range(trials):
        try:
            model_cls([3, 0, 2, 4, 1], d, random.Random(rng.random())).run()
        except ProtocolError:
            return True
    return False


def test_persistent_forward_o_free_is_implied_by_the_next_p():
    # the next item's first P V product also waits for that item's first P, which the softmax
    # warps produce only after their epilogue has read O: the "O free" wait the kernel keeps (it
    # names the dependency) is implied, and the model agrees that dropping it is no error
    class NoOFree(PersistentFwdModel):
        def p_pv(self):
            for req in super().p_pv():
                if req[0] == "wait" and req[1] == "OFREE":
                    continue
                yield req

    assert not _persistent_fails(NoOFree, trials=100)


def test_persistent_forward_model_catches_an_o_read_after_the_next_p():
    # an epilogue that read O only after producing the next item's first P (a reordering the
    # kernel must not make) lets the next item's first P V product overwrite O: with the "O free"
    # wait dropped too, the model finds it
    class LateRead(PersistentFwdModel):
        def p_pv(self):
            for req in super().p_pv():
                if req[0] == "wait" and req[1] == "OFREE":
                    continue
                yield req

        def p_softmax(self):
            jg, a, pending = 0, 0, None
            for k, c in enumerate(self.items):
                for j in range(c):
                    b = jg % self.NB
                    yield self.wait(f"S{b}", jg // self.NB)
                    self.expect(f"sbuf{b}", ("S", jg))
                    yield self.STEP
                    self.put(f"sbuf{b}", ("P", jg))
                    yield self.arrive(f"P{b}")
                    jg += 1
                    if pending is not None:  # the previous item's O read, too late
                        yield self.STEP
                        self.expect("O", pending)
                        pending = None
                if c > 0:
                    yield self.wait("OFULL", a)
                    pending = (k, c)
                    a += 1

    assert _persistent_fails(LateRead)


def test_persistent_forward_model_catches_an_early_q_load():
    # the next item's Q tile loaded before the S products of this item have read Q
    class NoQe(PersistentFwdModel):
        def p_q(self):
            for req in super().p_q():
                if req[0] == "wait" and req[1] == "QE":
                    continue
                yield req

    assert _persistent_fails(NoQe)
