"""The barrier protocols of the attention kernels, on the host (no GPU).

Each role of a CTA -- the TMA producer, the MMA-issuing thread and each of the
eight elementwise warps -- is restated as the sequence of mbarrier waits and
arrivals, tcgen05 commits, TMA loads, MMAs and tensor-memory accesses it makes,
in the order of the kernels in fa_backward_sm103.cu.  A scheduler then runs the
roles under many random interleavings, with the tensor core executing the MMAs
in issue order (each one reads its operands and writes its result when it
runs) and TMA loads completing in any order.  Every run must finish (no
deadlock), every parity wait must see the phase it waits for before the
barrier can complete the next one (no skipped phase), and every read of tensor
or shared memory must find the item it expects there (no overwrite too early,
no read too late).  The forward kernel's roles are restated the same way, for
both head sizes.  Planted mistakes, one or two per kernel, check that the model
catches them.
"""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.done = count, 0, 0


class ProtocolError(AssertionError):
    pass


class Sim:
    def __init__(self, seed):
        self.rng = random.Random(seed)
        self.bars = {}
        self.mem = {}
        self.mma_q = []
        self.tma = []
        self.roles = []

    def bar(self, name, count=1):
        self.bars[name] = Bar(count)

    def arrive(self, name):
        b = self.bars[name]
        b.pending += 1
        if b.pending == b.count:
            b.pending, b.done = 0, b.done + 1

    def check_read(self, region, expect, who):
        got = self.mem.get(region)
        if got != expect:
            raise ProtocolError(f"{who} read {region}: found {got}, expected {expect}")

    def role(self, name, gen):
        self.roles.append([name, gen, None, False])  # name, generator, pending action, finished

    def _advance(self, r, send=None):
        # the role's next action (send delivers the result of a non-blocking test)
        try:
            r[2] = r[1].send(send)
        except StopIteration:
            r[3] = True

    def _ready(self, r):
        act = r[2]
        if act[0] == "wait":
            return self.bars[act[1]].done >= act[2] + 1
        return True

    def _step(self, r):
        act, name = r[2], r[0]
        kind = act[0]
        result = None
        if kind == "wait":
            b = self.bars[act[1]]
            if b.done >= act[2] + 2:
                raise ProtocolError(f"{name}: {act[1]} completed phase {act[2] + 1} before the wait "
                                    f"for phase {act[2]} was seen")
        elif kind == "test":
            b = self.bars[act[1]]
            if b.done >= act[2] + 2:
                raise ProtocolError(f"{name}: {act[1]} skipped a phase under a test")
            result = b.done >= act[2] + 1
        elif kind == "arrive":
            self.arrive(act[1])
        elif kind == "read":
            self.check_read(act[1], act[2], name)
        elif kind == "write":
            self.mem[act[1]] = act[2]
        elif kind == "mma":
            self.mma_q.append(("mma", act[1], act[2], name))
        elif kind == "commit":
            self.mma_q.append(("commit", act[1]))
        elif kind == "load":
            self.tma.append((act[1], act[2]))
        else:
            raise ValueError(kind)
        self._advance(r, result)

    def run(self, max_steps=200000):
        for r in self.roles:
            self._advance(r)  # to the first action
        for _ in range(max_steps):
            choices = [("role", r) for r in self.roles if not r[3] and self._ready(r)]
            if self.mma_q:
                choices.append(("mma", None))
            if self.tma:
                choices.append(("tma", None))
            if not choices:
                stuck = [(r[0], r[2]) for r in self.roles if not r[3]]
                if stuck:
                    raise ProtocolError(f"deadlock: {stuck[:4]}")
                return
            kind, r = self.rng.choice(choices)
            if kind == "role":
                self._step(r)
            elif kind == "mma":
                op = self.mma_q.pop(0)
                if op[0] == "commit":
                    self.arrive(op[1])
                else:
                    for region, expect in op[1]:
                        self.check_read(region, expect, f"MMA issued by {op[3]}")
                    for region, value in op[2]:
                        self.mem[region] = value
            else:
                writes, bar = self.tma.pop(self.rng.randrange(len(self.tma)))
                for region, value in writes:
                    self.mem[region] = value
                self.arrive(bar)
        raise ProtocolError("no end within the step limit")


WARPS = [(wq, hf) for hf in range(2) for wq in range(4)]  # warp w: quadrant w % 4, half w // 4


def cols(prefix, n_sub=8):
    # every 16-column piece of a 128-column TMEM area in every lane quadrant
    return [f"{prefix}{wq}.{sb}" for wq in range(4) for sb in range(n_sub)]


def dq_kernel(sim, units, plant=None):
    """bwd_dq_kernel: one persistent CTA runs its query tiles (units) in turn, each
    with n_iter key tiles.  S and dP of key tile j+1 are issued once every warp
    holds tile j's (across a unit boundary too), dS has columns of its own, K and
    V stream through rings of their own (3 and 2 stages) that run on across
    units, and Q, dO of the next unit are loaded once the last score products of
    the unit before have read them.  The accumulator is read by the epilogue
    before the next unit's first product overwrites it."""
    if isinstance(units, int):
        units = [units]
    KS, VS = 3, 2
    for name, count in [("s_full", 1), ("s_loaded", 8), ("p_ready", 8), ("dq_done", 1), ("acc_done", 1),
                        ("fix_full", 1), ("fix_empty", 1)]:
        sim.bar(name, count)
    for s in range(KS):
        sim.bar(f"k_full{s}"), sim.bar(f"k_empty{s}")
    for s in range(VS):
        sim.bar(f"v_full{s}"), sim.bar(f"v_empty{s}")

    def producer():
        g = 0
        for k, n_iter in enumerate(units):
            if k > 0 and plant != "no_fix_empty":
                yield ("wait", "fix_empty", k - 1)
            yield ("load", [("QDO", ("Q", k))], "fix_full")
            for n in range(n_iter):
                ks, vs = g % KS, g % VS
                if g >= KS:
                    yield ("wait", f"k_empty{ks}", g // KS - 1)
                yield ("load", [(f"K{ks}", ("K", g))], f"k_full{ks}")
                if g >= VS:
                    yield ("wait", f"v_empty{vs}", g // VS - 1)
                yield ("load", [(f"V{vs}", ("V", g))], f"v_full{vs}")
                g += 1

    def mma():
        def scores(j, k):
            ks, vs = j % KS, j % VS
            yield ("wait", f"k_full{ks}", j // KS)
            yield ("wait", f"v_full{vs}", j // VS)
            yield ("mma", [(f"K{ks}", ("K", j)), ("QDO", ("Q", k))], [(x, ("S", j)) for x in cols("X")])
            yield ("mma", [(f"V{vs}", ("V", j)), ("QDO", ("Q", k))], [(y, ("dP", j)) for y in cols("Y")])
            yield ("commit", "s_full")
            yield ("commit", f"v_empty{vs}")
        g = 0
        for k, n_iter in enumerate(units):
            yield ("wait", "fix_full", k)
            if g > 0:  # implied by p_ready of the unit before, waited for all the same
                yield ("wait", "s_loaded", g - 1)
            yield from scores(g, k)
            if n_iter == 1:
                yield ("commit", "fix_empty")
            for n in range(n_iter):
                gi = g + n
                if n + 1 < n_iter:
                    if plant != "scores_before_loaded":
                        yield ("wait", "s_loaded", gi)
                    yield from scores(gi + 1, k)
                    if n + 2 == n_iter:
                        yield ("commit", "fix_empty")  # the unit's last reads of Q and dO
                yield ("wait", "p_ready", gi)
                ks = gi % KS
                reads = [(f"DS{wq}.{q}", ("dS", gi)) for wq in range(4) for q in range(4)] + [(f"K{ks}", ("K", gi))]
                if n > 0:
                    reads.append(("ACC", ("dQ", k, n - 1)))
                yield ("mma", reads, [("ACC", ("dQ", k, n))])
                yield ("commit", f"k_empty{ks}")
                yield ("commit", "dq_done")
            yield ("commit", "acc_done")
            g += n_iter

    def elementwise(wq, hf):
        mine = [4 * hf + i for i in range(4)]
        g = 0
        late = None  # planted: an epilogue left until after the next unit's first item
        for k, n_iter in enumerate(units):
            for n in range(n_iter):
                gi = g + n
                yield ("wait", "s_full", gi)
                for sb in mine:
                    yield ("read", f"X{wq}.{sb}", ("S", gi))
                    yield ("read", f"Y{wq}.{sb}", ("dP", gi))
                yield ("arrive", "s_loaded")
                if gi > 0 and plant != "no_dq_done":
                    yield ("wait", "dq_done", gi - 1)
                for h in range(2):
                    yield ("write", f"DS{wq}.{2 * hf + h}", ("dS", gi))
                yield ("arrive", "p_ready")
                if late is not None:
                    yield ("read", "ACC", late)
                    late = None
            yield ("wait", "acc_done", k)
            if plant == "late_epilogue" and k + 1 < len(units):
                late = ("dQ", k, n_iter - 1)
            else:
                yield ("read", "ACC", ("dQ", k, n_iter - 1))
            g += n_iter

    sim.role("tma", producer())
    sim.role("mma", mma())
    for wq, hf in WARPS:
        sim.role(f"warp{wq + 4 * hf}", elementwise(wq, hf))


def dkdv_kernel_128(sim, units, plant=None):
    """bwd_dkdv_kernel at d = 128: one persistent CTA runs its key tiles (units) in
    turn, each with n_iter (query head, query tile) items.  P^T then dS^T are
    written over S^T and dP^T in two steps, the next item's S^T is issued right
    after dV when its stage has landed (within a unit), K and V of the next unit
    are loaded once the last score products of the unit before have read them,
    and the ring and the per-item barriers run on across units."""
    if isinstance(units, int):
        units = [units]
    S = 2
    for name, count in [("s_full", 1), ("s_loaded", 8), ("p_ready", 8), ("dp_full", 1), ("dp_loaded", 8),
                        ("ds_ready", 8), ("acc_done", 1), ("fix_full", 1), ("fix_empty", 1)]:
        sim.bar(name, count)
    for s in range(S):
        sim.bar(f"ring_full{s}"), sim.bar(f"ring_empty{s}")

    def producer():
        g = 0
        for k, n_iter in enumerate(units):
            if k > 0 and plant != "no_fix_empty":
                yield ("wait", "fix_empty", k - 1)
            yield ("load", [("KV", ("KV", k))], "fix_full")
            for n in range(n_iter):
                slot = g % S
                if g >= S:
                    yield ("wait", f"ring_empty{slot}", g // S - 1)
                yield ("load", [(f"Q{slot}", ("Q", g)), (f"dO{slot}", ("dO", g)), (f"vec{slot}", ("vec", g))],
                       f"ring_full{slot}")
                g += 1

    def mma():
        def issue_s(j, k):
            slot = j % S
            yield ("mma", [(f"Q{slot}", ("Q", j)), ("KV", ("KV", k))], [(x, ("S", j)) for x in cols("X")])
            yield ("commit", "s_full")

        def issue_dp(j, k):
            slot = j % S
            yield ("mma", [(f"dO{slot}", ("dO", j)), ("KV", ("KV", k))], [(y, ("dP", j)) for y in cols("Y")])
            yield ("commit", "dp_full")
        g = 0
        for k, n_iter in enumerate(units):
            yield ("wait", "fix_full", k)
            yield ("wait", f"ring_full{g % S}", g // S)
            yield from issue_s(g, k)
            yield from issue_dp(g, k)
            if n_iter == 1:
                yield ("commit", "fix_empty")
            for n in range(n_iter):
                gi = g + n
                slot = gi % S
                nx, s_issued = n + 1, False
                yield ("wait", "p_ready", gi)
                if nx < n_iter and plant == "s_before_dv":
                    # the mistake: the next S^T goes ahead of the dV product that reads P^T
                    yield ("wait", f"ring_full{(gi + 1) % S}", (gi + 1) // S)
                    yield from issue_s(gi + 1, k)
                    s_issued = True
                reads = [(f"X{wq}.{sb}", ("P", gi)) for wq in range(4) for sb in range(4)] + \
                        [(f"dO{slot}", ("dO", gi))]
                if n > 0:
                    reads.append(("dV", ("dV", k, n - 1)))
                yield ("mma", reads, [("dV", ("dV", k, n))])
                if nx < n_iter and not s_issued:
                    landed = yield ("test", f"ring_full{(gi + 1) % S}", (gi + 1) // S)
                    if landed:
                        yield from issue_s(gi + 1, k)
                        s_issued = True
                yield ("wait", "ds_ready", gi)
                reads = [(f"Y{wq}.{sb}", ("dS", gi)) for wq in range(4) for sb in range(4)] + \
                        [(f"Q{slot}", ("Q", gi))]
                if n > 0:
                    reads.append(("dK", ("dK", k, n - 1)))
                yield ("mma", reads, [("dK", ("dK", k, n))])
                yield ("commit", f"ring_empty{slot}")
                if nx < n_iter:
                    if not s_issued:
                        yield ("wait", f"ring_full{(gi + 1) % S}", (gi + 1) // S)
                        yield from issue_s(gi + 1, k)
                    yield from issue_dp(gi + 1, k)
                    if nx + 1 == n_iter:
                        yield ("commit", "fix_empty")  # the unit's last reads of K and V
            yield ("commit", "acc_done")
            g += n_iter

    def elementwise(wq, hf):
        mine = [4 * hf + i for i in range(4)]
        g = 0
        for k, n_iter in enumerate(units):
            for n in range(n_iter):
                gi = g + n
                slot = gi % S
                yield ("wait", f"ring_full{slot}", gi // S)
                yield ("wait", "s_full", gi)
                for sb in mine:
                    yield ("read", f"X{wq}.{sb}", ("S", gi))
                yield ("arrive", "s_loaded")
                if plant != "no_intra_sync":
                    yield ("wait", "s_loaded", gi)
                yield ("read", f"vec{slot}", ("vec", gi))
                for h in range(2):
                    yield ("write", f"X{wq}.{2 * hf + h}", ("P", gi))
                yield ("arrive", "p_ready")
                yield ("wait", "dp_full", gi)
                for sb in mine:
                    yield ("read", f"Y{wq}.{sb}", ("dP", gi))
                yield ("arrive", "dp_loaded")
                yield ("wait", "dp_loaded", gi)
                yield ("read", f"vec{slot}", ("vec", gi))
                for h in range(2):
                    yield ("write", f"Y{wq}.{2 * hf + h}", ("dS", gi))
                yield ("arrive", "ds_ready")
            yield ("wait", "acc_done", k)
            yield ("read", "dV", ("dV", k, n_iter - 1))
            yield ("read", "dK", ("dK", k, n_iter - 1))
            g += n_iter

    sim.role("tma", producer())
    sim.role("mma", mma())
    for wq, hf in WARPS:
        sim.role(f"warp{wq + 4 * hf}", elementwise(wq, hf))


def dkdv_kernel_64(sim, units, plant=None):
    """bwd_dkdv_kernel at d = 64: P^T and dS^T in columns of their own, the next
    item's S^T and dP^T issued once every warp holds the current ones (across a
    unit boundary once K and V of the next unit have landed)."""
    if isinstance(units, int):
        units = [units]
    S = 3
    for name, count in [("s_full", 1), ("s_loaded", 8), ("p_ready", 8), ("pd_done", 1), ("acc_done", 1),
                        ("fix_full", 1), ("fix_empty", 1)]:
        sim.bar(name, count)
    for s in range(S):
        sim.bar(f"ring_full{s}"), sim.bar(f"ring_empty{s}")

    def producer():
        g = 0
        for k, n_iter in enumerate(units):
            if k > 0 and plant != "no_fix_empty":
                yield ("wait", "fix_empty", k - 1)
            yield ("load", [("KV", ("KV", k))], "fix_full")
            for n in range(n_iter):
                slot = g % S
                if g >= S:
                    yield ("wait", f"ring_empty{slot}", g // S - 1)
                yield ("load", [(f"Q{slot}", ("Q", g)), (f"dO{slot}", ("dO", g)), (f"vec{slot}", ("vec", g))],
                       f"ring_full{slot}")
                g += 1

    def mma():
        def scores(j, k):
            slot = j % S
            yield ("wait", f"ring_full{slot}", j // S)
            yield ("mma", [(f"Q{slot}", ("Q", j)), ("KV", ("KV", k))], [(x, ("S", j)) for x in cols("X")])
            yield ("mma", [(f"dO{slot}", ("dO", j)), ("KV", ("KV", k))], [(y, ("dP", j)) for y in cols("Y")])
            yield ("commit", "s_full")
        g = 0
        for k, n_iter in enumerate(units):
            yield ("wait", "fix_full", k)
            if g > 0:  # implied by p_ready of the unit before, waited for all the same
                yield ("wait", "s_loaded", g - 1)
            yield from scores(g, k)
            if n_iter == 1:
                yield ("commit", "fix_empty")
            for n in range(n_iter):
                gi = g + n
                slot = gi % S
                if n + 1 < n_iter:
                    yield ("wait", "s_loaded", gi)
                    yield from scores(gi + 1, k)
                    if n + 2 == n_iter:
                        yield ("commit", "fix_empty")
                yield ("wait", "p_ready", gi)
                pr = [(f"PP{wq}.{q}", ("P", gi)) for wq in range(4) for q in range(4)]
                dr = [(f"DD{wq}.{q}", ("dS", gi)) for wq in range(4) for q in range(4)]
                yield ("mma", pr + [(f"dO{slot}", ("dO", gi))] + ([("dV", ("dV", k, n - 1))] if n else []),
                       [("dV", ("dV", k, n))])
                yield ("mma", dr + [(f"Q{slot}", ("Q", gi))] + ([("dK", ("dK", k, n - 1))] if n else []),
                       [("dK", ("dK", k, n))])
                yield ("commit", f"ring_empty{slot}")
                yield ("commit", "pd_done")
            yield ("commit", "acc_done")
            g += n_iter

    def elementwise(wq, hf):
        mine = [4 * hf + i for i in range(4)]
        g = 0
        late = None  # planted: an epilogue left until after the next unit's first item
        for k, n_iter in enumerate(units):
            for n in range(n_iter):
                gi = g + n
                slot = gi % S
                yield ("wait", f"ring_full{slot}", gi // S)
                yield ("wait", "s_full", gi)
                for sb in mine:
                    yield ("read", f"X{wq}.{sb}", ("S", gi))
                    yield ("read", f"Y{wq}.{sb}", ("dP", gi))
                yield ("arrive", "s_loaded")
                yield ("read", f"vec{slot}", ("vec", gi))
                if gi > 0 and plant != "no_pd_done":
                    yield ("wait", "pd_done", gi - 1)
                for h in range(2):
                    yield ("write", f"PP{wq}.{2 * hf + h}", ("P", gi))
                    yield ("write", f"DD{wq}.{2 * hf + h}", ("dS", gi))
                yield ("arrive", "p_ready")
                if late is not None:
                    yield ("read", "dV", late)
                    late = None
            yield ("wait", "acc_done", k)
            if plant == "late_epilogue" and k + 1 < len(units):
                late = ("dV", k, n_iter - 1)
            else:
                yield ("read", "dV", ("dV", k, n_iter - 1))
            yield ("read", "dK", ("dK", k, n_iter - 1))
            g += n_iter

    sim.role("tma", producer())
    sim.role("mma", mma())
    for wq, hf in WARPS:
        sim.role(f"warp{wq + 4 * hf}", elementwise(wq, hf))


def dq_gemm_kernel(sim, units, plant=None):
    """bwd_dq_gemm_kernel: dQ of one query tile (a unit) is the sum over its n_iter
    key tiles of dS K.  One ring of 3 stages carries the dS block and K tile of
    each product and runs on across units; the units alternate between two TMEM
    accumulators, so the epilogue (4 warps) reads one while the next unit's
    products fill the other.  The MMA thread takes an accumulator back only once
    the epilogue of the unit two before has read it."""
    if isinstance(units, int):
        units = [units]
    S = 3
    for s in range(S):
        sim.bar(f"full{s}"), sim.bar(f"empty{s}")
    for b in range(2):
        sim.bar(f"acc_full{b}"), sim.bar(f"acc_free{b}", 4)

    def producer():
        g = 0
        for k, n_iter in enumerate(units):
            for n in range(n_iter):
                st = g % S
                if g >= S and plant != "no_empty_wait":
                    yield ("wait", f"empty{st}", g // S - 1)
                yield ("load", [(f"DS{st}", ("dS", k, n)), (f"K{st}", ("K", k, n))], f"full{st}")
                g += 1

    def acc(k):
        return 0 if plant == "one_accumulator" else k & 1

    def mma():
        g = 0
        for k, n_iter in enumerate(units):
            b = acc(k)
            if k >= 2 and plant != "no_acc_free":
                yield ("wait", f"acc_free{b}", (k - 2) >> 1)
            for n in range(n_iter):
                st = g % S
                yield ("wait", f"full{st}", g // S)
                reads = [(f"DS{st}", ("dS", k, n)), (f"K{st}", ("K", k, n))]
                if n > 0:
                    reads.append((f"ACC{b}", ("dQ", k, n - 1)))
                yield ("mma", reads, [(f"ACC{b}", ("dQ", k, n))])
                yield ("commit", f"empty{st}")
                g += 1
            yield ("commit", f"acc_full{b}")

    def epilogue(w):
        for k, n_iter in enumerate(units):
            b = k & 1
            yield ("wait", f"acc_full{b}", k >> 1)
            yield ("read", f"ACC{acc(k)}", ("dQ", k, n_iter - 1))
            yield ("arrive", f"acc_free{b}")

    sim.role("tma", producer())
    sim.role("mma", mma())
    for w in range(4):
        sim.role(f"warp{w}", epilogue(w))


KERNELS = {"dq": dq_kernel, "dkdv128": dkdv_kernel_128, "dkdv64": dkdv_kernel_64, "dq_gemm": dq_gemm_kernel}


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("n_iter", [1, 2, 3, 7])
def test_protocol_holds_under_random_interleavings(kernel, n_iter):
    for seed in range(150):
        sim = Sim(1000 * n_iter + seed)
        KERNELS[kernel](sim, n_iter)
        sim.run()


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("units", [[1, 1], [2, 3], [3, 1, 2], [7, 2]])
def test_persistent_protocol_holds_under_random_interleavings(kernel, units):
    # one CTA running several units (query tiles for dQ, key tiles for dK/dV) in turn
    for seed in range(150):
        sim = Sim(7000 + seed)
        KERNELS[kernel](sim, units)
        sim.run()


@pytest.mark.parametrize("kernel,plant", [("dq", "no_fix_empty"), ("dq", "late_epilogue"),
                                          ("dkdv128", "no_fix_empty"), ("dkdv64", "no_fix_empty"),
                                          ("dkdv64", "late_epilogue"), ("dq_gemm", "no_acc_free"),
                                          ("dq_gemm", "one_accumulator")])
def test_the_model_catches_a_planted_unit_boundary_mistake(kernel, plant):
    caught = 0
    for seed in range(150):
        sim = Sim(seed)
        KERNELS[kernel](sim, [2, 1, 3], plant)
        try:
            sim.run()
        except ProtocolError:
            caught += 1
    assert caught > 0, f"{kernel} with {plant} passed every interleaving"


@pytest.mark.parametrize("kernel,plant", [("dq", "no_dq_done"), ("dq", "scores_before_loaded"),
                                          ("dkdv128", "no_intra_sync"), ("dkdv128", "s_before_dv"),
                                          ("dkdv64", "no_pd_done"), ("dq_gemm", "no_empty_wait")])
def test_the_model_catches_a_planted_mistake(kernel, plant):
    caught = 0
    for seed in range(150):
        sim = Sim(seed)
        KERNELS[kernel](sim, 5, plant)
        try:
            sim.run()
        except ProtocolError:
            caught += 1
    assert caught > 0, f"{kernel} with {plant} passed every interleaving"


def prefill_kernel(sim, units, sep_p, plant=None):
    """prefill_kernel, one CTA running `units` = [(j0, n0, n1), ...] back to back:
    whole units (j0 = 0) or stream-K pieces (j0 > 0), query tile t taking key
    tiles [j0, n_t) of the piece's [j0, max(n0, n1)) (none when n_t <= j0).
    d = 128 (sep_p False): P over S, o_done after a tile's last PV.  d = 64
    (sep_p True): P in columns of its own, s_free / pv_done, both Q K^T products
    of a step before both PV products.  Each softmax warp may rescale O at any
    step after a piece's first."""
    for name in ["q_full", "q_empty", "kv_full0", "kv_full1", "kv_empty0", "kv_empty1"]:
        sim.bar(name)
    for t in range(2):
        sim.bar(f"s_full{t}"), sim.bar(f"o_done{t}"), sim.bar(f"pv_done{t}")
        sim.bar(f"p_full{t}", 4), sim.bar(f"s_free{t}", 4)

    def producer():
        gc = 0

        def group(writes):
            nonlocal gc
            st = gc % 2
            if gc >= 2:
                yield ("wait", f"kv_empty{st}", gc // 2 - 1)
            yield ("load", [(f"ring{2 * st + half}", v) for half, v in writes], f"kv_full{st}")
            gc += 1
        for u, (j0, n0, n1) in enumerate(units):
            if u > 0:
                yield ("wait", "q_empty", u - 1)
            yield ("load", [(f"Q{t}", ("Q", u, t)) for t in range(2) if (n0, n1)[t] > j0], "q_full")
            j1 = max(n0, n1)
            yield from group([(0, ("K", u, j0))])
            for j in range(j0, j1):
                writes = [(0, ("V", u, j))] + ([(1, ("K", u, j + 1))] if j + 1 < j1 else [])
                yield from group(writes)

    def mma():
        gc, pc, qk = 0, [0, 0], [0, 0]

        def take_group():
            nonlocal gc
            st = gc % 2
            yield ("wait", f"kv_full{st}", gc // 2)
            return st

        def qk_mma(u, t, j, kslot):
            reads = [(f"Q{t}", ("Q", u, t)), (f"ring{kslot}", ("K", u, j))]
            return ("mma", reads, [(f"S{t}.{w}", ("S", u, t, j)) for w in range(4)])

        def pv_mma(u, t, j, j0, vslot):
            reads = [(f"P{t}.{w}", ("P", u, t, j)) for w in range(4)]
            reads += [(f"ring{vslot}", ("V", u, j))]
            if j > j0:
                reads += [(f"O{t}.{w}", ("O", u, t, j - 1)) for w in range(4)]
            return ("mma", reads, [(f"O{t}.{w}", ("O", u, t, j)) for w in range(4)])
        for u, (j0, *n) in enumerate(units):
            j1 = max(n)
            yield ("wait", "q_full", u)
            st = yield from take_group()
            for t in range(2):
                if n[t] > j0:
                    if sep_p and qk[t] > 0:
                        yield ("wait", f"s_free{t}", qk[t] - 1)
                    yield qk_mma(u, t, j0, 2 * st)
                    yield ("commit", f"s_full{t}")
                    qk[t] += 1
            yield ("commit", f"kv_empty{st}")
            gc += 1
            if j1 - j0 == 1:
                yield ("commit", "q_empty")
            for j in range(j0, j1):
                st = yield from take_group()
                if not sep_p:
                    for t in range(2):
                        if j >= n[t]:
                            continue
                        yield ("wait", f"p_full{t}", pc[t])
                        pc[t] += 1
                        if plant == "qk_before_pv" and j + 1 < n[t]:
                            yield qk_mma(u, t, j + 1, 2 * st + 1)
                        yield pv_mma(u, t, j, j0, 2 * st)
                        if j == n[t] - 1:
                            yield ("commit", f"o_done{t}")
                        if j + 1 < n[t]:
                            if plant != "qk_before_pv":
                                yield qk_mma(u, t, j + 1, 2 * st + 1)
                            yield ("commit", f"s_full{t}")
                else:
                    for t in range(2):
                        if j + 1 < n[t]:
                            if plant != "qk_without_s_free":
                                yield ("wait", f"s_free{t}", qk[t] - 1)
                            yield qk_mma(u, t, j + 1, 2 * st + 1)
                            yield ("commit", f"s_full{t}")
                            qk[t] += 1
                    for t in range(2):
                        if j >= n[t]:
                            continue
                        yield ("wait", f"p_full{t}", pc[t])
                        pc[t] += 1
                        yield pv_mma(u, t, j, j0, 2 * st)
                        yield ("commit", f"pv_done{t}")
                yield ("commit", f"kv_empty{st}")
                gc += 1
                if j + 1 == j1 - 1:
                    yield ("commit", "q_empty")

    def softmax(t, w):
        sc = oc = pvc = 0
        for u, (j0, *n) in enumerate(units):
            for j in range(j0, n[t]):
                yield ("wait", f"s_full{t}", sc)
                sc += 1
                yield ("read", f"S{t}.{w}", ("S", u, t, j))
                if sep_p:
                    yield ("arrive", f"s_free{t}")
                    if j > j0:
                        yield ("wait", f"pv_done{t}", pvc)
                        pvc += 1
                yield ("write", f"P{t}.{w}", ("P", u, t, j))
                if j > j0 and sim.rng.random() < 0.3:  # the lazy rescale of O
                    yield ("read", f"O{t}.{w}", ("O", u, t, j - 1))
                    yield ("write", f"O{t}.{w}", ("O", u, t, j - 1))
                yield ("arrive", f"p_full{t}")
                if plant == "double_arrive":  # two lanes of a warp arriving, not one
                    yield ("arrive", f"p_full{t}")
            if n[t] > j0:
                if sep_p:
                    yield ("wait", f"pv_done{t}", pvc)
                    pvc += 1
                else:
                    yield ("wait", f"o_done{t}", oc)
                    oc += 1
                yield ("read", f"O{t}.{w}", ("O", u, t, n[t] - 1))

    if not sep_p:
        # P is written over S: the same tensor-memory area under two names
        class Alias(dict):
            def _k(self, k):
                return k.replace("P", "S", 1) if k.startswith("P") else k

            def get(self, k, d=None):
                return dict.get(self, self._k(k), d)

            def __setitem__(self, k, v):
                dict.__setitem__(self, self._k(k), v)
        sim.mem = Alias()
    sim.role("tma", producer())
    sim.role("mma", mma())
    for t in range(2):
        for w in range(4):
            sim.role(f"softmax{t}.{w}", softmax(t, w))


# whole units, causal units whose tiles end apart, and stream-K pieces: a cut
# piece first, whole units after, tiles without keys in a piece
PREFILL_UNITS = [[(0, 3, 3)], [(0, 1, 1), (0, 2, 2)], [(0, 2, 3), (0, 3, 2), (0, 1, 1)],
                 [(0, 4, 4), (0, 1, 2), (0, 2, 1)], [(2, 5, 5), (0, 3, 3), (0, 2, 2)],
                 [(1, 2, 4), (0, 3, 1), (3, 4, 4)], [(3, 2, 5), (0, 1, 3), (2, 4, 2)]]


@pytest.mark.parametrize("sep_p", [False, True], ids=["d128", "d64"])
@pytest.mark.parametrize("units", PREFILL_UNITS, ids=lambda u: "-".join(f"{a}{b}{c}" for a, b, c in u))
def test_prefill_protocol_holds_under_random_interleavings(sep_p, units):
    for seed in range(150):
        sim = Sim(seed)
        prefill_kernel(sim, units, sep_p)
        sim.run()


@pytest.mark.parametrize("sep_p,plant", [(False, "qk_before_pv"), (True, "qk_without_s_free"),
                                         (False, "double_arrive"), (True, "double_arrive")])
def test_the_prefill_model_catches_a_planted_mistake(sep_p, plant):
    caught = 0
    for seed in range(150):
        sim = Sim(seed)
        prefill_kernel(sim, [(0, 3, 3), (1, 2, 3)], sep_p, plant)
        try:
            sim.run()
        except ProtocolError:
            caught += 1
    assert caught > 0, f"prefill sep_p={sep_p} with {plant} passed every interleaving"
