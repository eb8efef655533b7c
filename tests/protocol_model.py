"""Models of the tensor-core forward kernels' synchronisation, run under random
interleavings on the CPU (Kernel: attn_tc_kernel, d = 64 / 128; Kernel256:
attn_tc256_kernel, described in its own docstring).

The kernel (attn_tc_kernel for 16-bit inputs and for e4m3 with V widened once
per call; with `conv`, e4m3 with V widened on chip) has these roles, and the
model gives each its own agent:

* the producer warp, filling a ring of K/V slots by TMA (item 2j = K_j,
  item 2j + 1 = V_j) after waiting for the slot's release (kv_empty);
* one MMA issuer per query tile t in {A, B}: S = Q_t K_j^T into the one score
  buffer the two tiles share, in the order A_0, B_0, A_1, B_1, ... (each score
  MMA waits until the softmax of the one before it has loaded its scores,
  s_free), then O_t += P_t V_j once P_t is in (p_full); each MMA is followed by
  commits (s_full, pv_done, and the slot's kv_empty);
* four softmax warps per tile: wait for the scores (s_full), load them, signal
  s_free, wait until the previous P_t V has completed (pv_done) before
  overwriting P_t, then signal p_full; at the end wait for the last P_t V;
* on-chip widening (`conv`): each e4m3 V tile is widened into fp16 buffer
  j mod 2 in four shares, by a converter warp, the producer (its share of V_c
  once V_{c+3} has been loaded) and each issuer (right after its P V of the
  step before); a share waits for the V tile (kv_full) and for the buffer
  (v16_empty: both tiles' P V of V_{j-2} done), then arrives on v16_full and
  on the V slot's release (kv_empty, four releases per V slot); P V reads the
  fp16 buffer once v16_full is complete and releases it with its commit.

The asynchronous parts are modelled as events the scheduler may take at any
time: a TMA load lands (completing the slot's kv_full phase); the tensor core
executes the oldest pending operation of either issuer (one issuer's MMAs and
commits complete in issue order, the two issuers' interleave freely).

An mbarrier completes a phase once its arrival count and its expected
transactions are both used up.  A wait for phase n (parity n & 1) passes when
the barrier's completed-phase count differs in parity from n; that is only the
right answer when exactly n + 1 phases have completed, so the model raises on
any pass at another count (a waiter two phases off would be fooled).  It also
checks every buffer at the moment an operation touches it: the score buffer is
overwritten only after all four warps of the tile that owns it loaded it, an
MMA reads the K or V tile it expects, P_t is overwritten only after the
P_t V that reads it has executed, O_t is rescaled only between two P_t V, and
a slot is refilled only after every MMA reading it has executed.  A run that
stops with agents still waiting is a deadlock.  With `timeout_p` the forward
model also takes the abort path: one blocked wait runs out at a random moment,
and the CTA must not exit with a TMA load or an MMA in flight.
"""

from __future__ import annotations

import random


class ProtocolError(AssertionError):
    pass


class Bar:
    """An mbarrier: arrival count, expected transactions, completed phases."""

    def __init__(self, name: str, count: int):
        self.name, self.count, self.pending, self.tx, self.k = name, count, count, 0, 0

    def arrive(self):
        if self.pending <= 0:
            raise ProtocolError(f"{self.name}: arrival beyond the count")
        self.pending -= 1
        self._complete()

    def expect_tx(self, n: int = 1):
        self.tx += n

    def land(self):
        self.tx -= 1
        if self.tx < 0:
            raise ProtocolError(f"{self.name}: more bytes landed than expected")
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.k += 1
            self.pending = self.count

    def passes(self, n: int) -> bool:
        """The parity rule of a wait (or test) for phase n."""
        ok = (self.k & 1) != (n & 1)
        if ok and self.k != n + 1:
            raise ProtocolError(f"{self.name}: a wait for phase {n} passed with {self.k} "
                                f"phases completed")
        return ok


class Wait:
    """A bounded wait an agent yields: resumed with True once the phase passes,
    or with False when the CTA's abort flag is set (or this wait runs out)."""

    def __init__(self, pred):
        self.pred = pred


class Drain:
    """A drain-only wait of the abort path: ignores the abort flag."""

    def __init__(self, pred):
        self.pred = pred


class Model:
    """Random scheduler shared by the kernel models: at each step it takes one
    of the runnable agents (a generator whose last yielded wait now passes, or
    that yielded None), a TMA load in flight, or the oldest pending operation of
    one MMA issuer, uniformly at random.  Agents may yield a bare predicate (a
    wait that only ever passes), a Wait, a Drain or None.  With `timeout_p` > 0
    a blocked Wait may run out at any step (once per run): it raises the abort
    flag, and from then on every blocked Wait returns False."""

    abort = False
    timeout_p = 0.0

    def agents(self):
        raise NotImplementedError

    def barriers(self):
        raise NotImplementedError

    def _ready(self, w):
        if w is None:
            return True
        if isinstance(w, Wait):
            return self.abort or w.pred()
        if isinstance(w, Drain):
            return w.pred()
        return w()

    def run(self, max_events=200000):
        agents = self.agents()
        waits = [None] * len(agents)
        alive = [True] * len(agents)
        started = [False] * len(agents)
        for _ in range(max_events):
            if self.timeout_p and not self.abort and self.rnd.random() < self.timeout_p:
                blocked = [i for i in range(len(agents)) if alive[i] and isinstance(waits[i], Wait)
                           and not waits[i].pred()]
                if blocked:
                    self.abort = True                    # this wait ran out
            choices = [("agent", i) for i, a in enumerate(agents)
                       if alive[i] and self._ready(waits[i])]
            choices += [("land", k) for k in range(len(self.landings))]
            choices += [("mma", t) for t in range(len(self.fifo)) if self.fifo[t]]
            if not choices:
                if any(alive):
                    raise ProtocolError("deadlock: agents " + ", ".join(
                        str(i) for i in range(len(agents)) if alive[i]) + " wait forever")
                break
            kind, i = self.rnd.choice(choices)
            if kind == "land":
                self.land(self.landings.pop(i))
            elif kind == "mma":
                self.execute(i)
            else:
                w = waits[i]
                value = (w.pred() if isinstance(w, Wait) else True) if w is not None else None
                try:
                    waits[i] = agents[i].send(value) if started[i] else next(agents[i])
                    started[i] = True
                except StopIteration:
                    alive[i] = False
                if not any(alive) and (self.landings or any(
                        op[0] != "commit" for f in self.fifo for op in f)):
                    raise ProtocolError("the CTA exits with a TMA load or an MMA in flight")
        else:
            raise ProtocolError("no end within the event budget")
        if self.abort:
            return
        for b in self.barriers():
            if b.pending != b.count or b.tx:
                raise ProtocolError(f"{b.name} left with a partial phase")
        self.finish()


class Kernel(Model):
    """attn_tc_kernel, one CTA: two query tiles with n_kv = (nt_A, nt_B) key
    tiles each, a ring of `slots` K/V slots.  `mutant` plants one protocol
    mistake (for the tests that show the model catches it)."""

    LAG = 3   # the producer widens its share of V_c after loading V_{c+LAG}

    def __init__(self, n_kv, slots, seed, mutant=None, conv=False, timeout_p=0.0,
                 drain_always=False):
        self.n_kv, self.S, self.mutant, self.conv = tuple(n_kv), slots, mutant, conv
        self.timeout_p, self.drain_always = timeout_p, drain_always
        if mutant == "lag_half_ring":
            self.LAG = slots // 2
        elif conv and (slots % 2 or self.LAG >= slots // 2):
            raise ValueError("on-chip widening needs an even ring deeper than 2 * LAG")
        self.n_max = max(n_kv)
        self.rnd = random.Random(seed)
        self.q_full = Bar("q_full", 1)
        self.s_full = [Bar(f"s_full{t}", 1) for t in range(2)]
        self.p_full = [Bar(f"p_full{t}", 4) for t in range(2)]
        self.pv_done = [Bar(f"pv_done{t}", 1) for t in range(2)]
        self.s_free = [Bar(f"s_free{t}", 4) for t in range(2)]
        release = 1 if mutant == "one_release_per_slot" else 2
        self.kv_full = [Bar(f"kv_full{s}", 1) for s in range(slots)]
        # with on-chip widening V items (odd slots) are released by the four warps that widen them
        self.kv_empty = [Bar(f"kv_empty{s}", 4 if conv and s % 2 else release) for s in range(slots)]
        self.v16_full = [Bar(f"v16_full{b}", 4) for b in range(2)]
        self.v16_empty = [Bar(f"v16_empty{b}", 2) for b in range(2)]
        self.drain = [Bar(f"drain{t}", 1) for t in range(2)]
        self.v16_item = [None, None]         # V tile whose shares the fp16 buffer holds
        self.v16_shares = [set(), set()]
        self.pv_of_v = {}                    # V index -> P V executed that read it
        # buffer state
        self.slot_item = [None] * slots      # item whose bytes are in the slot (None: in flight)
        self.slot_readers = [0] * slots      # issued MMAs that still have to read the slot
        self.q_landed = [False, False]
        self.S_owner = None                  # (t, j) of the scores in the shared buffer
        self.S_loaded = set()                # softmax warps that loaded them
        self.P = [[-1] * 4 for _ in range(2)]    # step whose P each warp's rows hold
        self.pv_done_n = [0, 0]              # P_t V executed
        self.qk_done_n = [0, 0]              # Q_t K^T executed
        self.fifo = [[], []]                 # issued, not yet executed tensor-core operations
        self.landings = []                   # TMA loads in flight: ("q", t) or ("kv", slot, item)

    # ------------------------------------------------------------ roles
    # Each role follows the kernel's own code, abort path included: a Wait
    # that returns False makes the role leave its loop; the producer then
    # drains the loads it issued (Q and the last `slots` ring items), an issuer
    # commits its drain barrier and waits for it, the other roles just stop.
    def producer(self):
        if self.n_max == 0:
            return
        S = self.S
        nq = sum(1 for t in range(2) if self.n_kv[t] > 0)
        self.q_full.expect_tx(nq)
        self.q_full.arrive()
        for t in range(2):
            if self.n_kv[t] > 0:
                self.landings.append(("q", t))
        it, next_share, ok = 0, 0, True
        while ok and it < 2 * self.n_max:
            slot = it % S
            ok = yield Wait(lambda s=slot, n=it // S - 1: self.kv_empty[s].passes(n))
            if not ok:
                break
            if self.slot_readers[slot]:
                raise ProtocolError(f"slot {slot} refilled with item {it} while an MMA still "
                                    f"has to read item {self.slot_item[slot]}")
            self.slot_item[slot] = None
            self.kv_full[slot].expect_tx()
            self.kv_full[slot].arrive()
            self.landings.append(("kv", slot, it))
            cur, it = it, it + 1
            if self.conv and cur % 2 and cur // 2 >= self.LAG:
                ok = yield from self.widen_share(next_share, "producer")
                next_share += 1
        while self.conv and ok and next_share < self.n_max:
            ok = yield from self.widen_share(next_share, "producer")
            next_share += 1
        if not ok or self.drain_always:
            yield Drain(lambda: self.q_full.passes(0))
            for k in range(max(0, it - S), it):
                yield Drain(lambda k=k: self.kv_full[k % S].passes(k // S))

    def widen_share(self, j, who):
        """One warp's share of V_j: e4m3 ring slot -> fp16 buffer j mod 2."""
        it, b = 2 * j + 1, j % 2
        slot = it % self.S
        ok = yield Wait(lambda: self.kv_full[slot].passes(it // self.S))
        if ok and self.mutant != "no_v16_empty_wait":
            ok = yield Wait(lambda: self.v16_empty[b].passes(j // 2 - 1))
        if not ok:
            return False
        if self.slot_item[slot] != it:
            raise ProtocolError(f"{who} widened slot {slot} holding {self.slot_item[slot]} as V_{j}")
        if j >= 2 and self.pv_of_v.get(j - 2, 0) != sum(n > j - 2 for n in self.n_kv):
            raise ProtocolError(f"{who} overwrote fp16 V_{j - 2} before both P V read it")
        if self.v16_item[b] != j:
            self.v16_item[b], self.v16_shares[b] = j, set()
        self.slot_readers[slot] += 1
        yield None                                       # loads, conversion, stores
        self.slot_readers[slot] -= 1
        self.v16_shares[b].add(who)
        self.v16_full[b].arrive()
        self.kv_empty[slot].arrive()
        return True

    def converter(self):
        for j in range(self.n_max if self.conv else 0):
            if not (yield from self.widen_share(j, "converter")):
                break

    def issuer(self, t):
        nt, nt_o = self.n_kv[t], self.n_kv[1 - t]
        if self.n_max == 0:
            return
        S = self.S

        def wait_full(it):
            return Wait(lambda: self.kv_full[it % S].passes(it // S))

        def s_ready(j):
            # the score MMA before tile t's j-th in the order A_0 B_0 A_1 B_1 ...
            if t == 0:
                prev = ((1 if j - 1 < nt_o else 0), j - 1) if j >= 1 else None
            elif j < nt_o:
                prev = (0, j)
            else:
                prev = (1, j - 1) if j >= 1 else None
            if prev is None or self.mutant == "no_s_free_wait":
                return None
            pt, pj = prev
            return Wait(lambda: self.s_free[pt].passes(pj))

        def issue(op, slot):
            self.slot_readers[slot] += 1
            self.fifo[t].append(op)

        def qk(j, itK):
            issue(("qk", t, j, itK % S), itK % S)
            self.fifo[t] += [("commit", self.s_full[t]), ("commit", self.kv_empty[itK % S])]

        ok = yield Wait(lambda: self.q_full.passes(0))
        if ok and nt > 0:
            ok = yield wait_full(0)
            w = s_ready(0)
            if ok and w:
                ok = yield w
            if ok:
                qk(0, 0)
        if ok and self.conv:
            ok = yield from self.widen_share(0, f"issuer{t}")
        j = 0
        while ok and j < nt:
            itK, itV = 2 * j + 2, 2 * j + 1
            if j + 1 < nt:
                ok = yield wait_full(itK)
                w = s_ready(j + 1)
                if ok and w:
                    ok = yield w
                if not ok:
                    break
                qk(j + 1, itK)
            if self.conv:
                ok = yield Wait(lambda j=j: self.v16_full[j % 2].passes(j // 2))
            else:
                ok = yield wait_full(itV)
            if ok:
                ok = yield Wait(lambda j=j: self.p_full[t].passes(j))
            if not ok:
                break
            if self.conv:
                self.fifo[t] += [("pv16", t, j, j % 2), ("commit", self.pv_done[t]),
                                 ("commit", self.v16_empty[j % 2])]
                if j + 1 < self.n_max:
                    ok = yield from self.widen_share(j + 1, f"issuer{t}")
            else:
                issue(("pv", t, j, itV % S), itV % S)
                self.fifo[t] += [("commit", self.pv_done[t]), ("commit", self.kv_empty[itV % S])]
            j += 1
        j = nt
        while ok and j < self.n_max:
            # key tiles this tile never reads: release them once filled
            ok = yield wait_full(2 * j)
            if ok:
                self.kv_empty[(2 * j) % S].arrive()
            if self.conv:
                if ok:
                    ok = yield Wait(lambda j=j: self.v16_full[j % 2].passes(j // 2))
                if ok:
                    self.v16_empty[j % 2].arrive()
                if ok and j + 1 < self.n_max:
                    ok = yield from self.widen_share(j + 1, f"issuer{t}")
            else:
                if ok:
                    ok = yield wait_full(2 * j + 1)
                if ok:
                    self.kv_empty[(2 * j + 1) % S].arrive()
            j += 1
        if not ok or self.drain_always:
            # none of this issuer's MMAs may still run when TMEM is freed
            self.fifo[t].append(("commit", self.drain[t]))
            yield Drain(lambda: self.drain[t].passes(0))

    def softmax(self, t, w):
        nt = self.n_kv[t]
        s_pre, ok = False, True
        for j in range(nt):
            if not s_pre:
                ok = yield Wait(lambda j=j: self.s_full[t].passes(j))
                if not ok:
                    break
            if self.S_owner != (t, j):
                raise ProtocolError(f"softmax {t}.{w} step {j} found the scores of {self.S_owner}")
            self.S_loaded.add(w)
            self.s_free[t].arrive()
            pv_pre = j > 0 and self.pv_done[t].passes(j - 1)
            yield None                                   # exponentials
            if j > 0 and not pv_pre and self.mutant != "no_pv_wait":
                ok = yield Wait(lambda j=j: self.pv_done[t].passes(j - 1))
                if not ok:
                    break
            if self.pv_done_n[t] < j:
                raise ProtocolError(f"softmax {t}.{w} overwrote P of step {j - 1} before its P V ran")
            self.P[t][w] = j
            s_pre = j + 1 < nt and self.s_full[t].passes(j + 1)
            if self.pv_done_n[t] != j:                   # the O rescale of this step
                raise ProtocolError(f"softmax {t}.{w} rescaled O while P V {self.pv_done_n[t]} ran")
            yield None
            self.p_full[t].arrive()
        if ok and nt > 0:
            ok = yield Wait(lambda: self.pv_done[t].passes(nt - 1))
            if ok and (self.pv_done_n[t] != nt or self.qk_done_n[t] != nt):
                raise ProtocolError(f"epilogue of tile {t} ran before its MMAs completed")

    # ------------------------------------------------------- async events
    def land(self, ev):
        if ev[0] == "q":
            self.q_landed[ev[1]] = True
            self.q_full.land()
        else:
            _, slot, it = ev
            self.slot_item[slot] = it
            self.kv_full[slot].land()

    def execute(self, t):
        op = self.fifo[t].pop(0)
        if op[0] == "commit":
            op[1].arrive()
            return
        kind, tt, j, slot = op
        if kind == "pv16":
            b = slot
            if self.v16_item[b] != j or len(self.v16_shares[b]) != 4:
                raise ProtocolError(f"P V ({tt}, {j}) read fp16 buffer {b} holding V_{self.v16_item[b]} "
                                    f"({len(self.v16_shares[b])} of 4 shares)")
            if any(p != j for p in self.P[tt]) or self.pv_done_n[tt] != j:
                raise ProtocolError(f"P V ({tt}, {j}) out of step")
            self.pv_done_n[tt] += 1
            self.pv_of_v[j] = self.pv_of_v.get(j, 0) + 1
            return
        if kind == "qk":
            if self.slot_item[slot] != 2 * j or not self.q_landed[tt]:
                raise ProtocolError(f"Q K^T ({tt}, {j}) read slot {slot} holding {self.slot_item[slot]}")
            if self.S_owner is not None and len(self.S_loaded) < 4:
                raise ProtocolError(f"Q K^T ({tt}, {j}) overwrote the unloaded scores of {self.S_owner}")
            if self.qk_done_n[tt] != j:
                raise ProtocolError("score MMAs of one tile out of order")
            self.S_owner, self.S_loaded = (tt, j), set()
            self.qk_done_n[tt] += 1
        else:
            if self.slot_item[slot] != 2 * j + 1:
                raise ProtocolError(f"P V ({tt}, {j}) read slot {slot} holding {self.slot_item[slot]}")
            if any(p != j for p in self.P[tt]):
                raise ProtocolError(f"P V ({tt}, {j}) read P of steps {self.P[tt]}")
            if self.pv_done_n[tt] != j:
                raise ProtocolError("P V of one tile out of order")
            self.pv_done_n[tt] += 1
        self.slot_readers[slot] -= 1

    # ---------------------------------------------------------- scheduler
    def agents(self):
        return ([self.producer(), self.issuer(0), self.issuer(1), self.converter()]
                + [self.softmax(t, w) for t in range(2) for w in range(4)])

    def barriers(self):
        return ([self.q_full] + self.s_full + self.p_full + self.pv_done + self.s_free
                + self.kv_full + self.kv_empty + self.v16_full + self.v16_empty)

    def finish(self):
        if self.pv_done_n != [n for n in self.n_kv]:
            raise ProtocolError("not every P V ran")


class Kernel256(Model):
    """attn_tc256_kernel, one CTA: one 128-row query tile, n key tiles.

    Two score buffers: the scores of key tile j go to buffer j mod 2 and the
    softmax writes P_j over them; the one MMA issuer sends P_j V_j and then the
    scores of key tile j + 2 into the same buffer (its MMAs run in issue order).
    The softmax can therefore run two key tiles ahead of the issuer's wait for
    P, so P has one barrier per buffer (p_full), and the epilogue waits on
    o_done, committed once after the last P V.  An occasional O rescale waits
    for the previous P V (pv_done).  The ring moves half tiles: 16-bit inputs
    load K_0, K_1, then V_j, K_{j+2}, ... (one release per item, by the issuer's
    commit); e4m3 (`e4m3`) loads K_0, V_0, K_1, V_1, ... into 4 slots, so slots
    0-1 only ever hold K and 2-3 only V, and two converter warps widen V_j's
    halves into fp16 buffer j mod 2 (each frees its slot once its half is in
    registers, then waits for the buffer: v16_empty, the P V of V_{j-2})."""

    def __init__(self, n, seed, e4m3=False, mutant=None):
        self.n, self.e4, self.mutant = n, e4m3, mutant
        self.S = 4 if e4m3 else 5
        self.rnd = random.Random(seed)
        self.q_full = Bar("q_full", 1)
        self.s_full = [Bar(f"s_full{b}", 1) for b in range(2)]
        p0 = Bar("p_full0", 4)
        self.p_full = [p0, p0] if mutant == "one_p_barrier" else [p0, Bar("p_full1", 4)]
        self.pv_done = Bar("pv_done", 1)
        self.o_done = Bar("o_done", 1)
        self.v16_full = [Bar(f"v16_full{b}", 2) for b in range(2)]
        self.v16_empty = [Bar(f"v16_empty{b}", 1) for b in range(2)]
        self.kv_full = [Bar(f"kv_full{s}", 1) for s in range(self.S)]
        self.kv_empty = [Bar(f"kv_empty{s}", 1) for s in range(self.S)]
        self.slot_item = [None] * self.S
        self.slot_readers = [0] * self.S
        self.q_landed = False
        self.buf = [[None] * 4 for _ in range(2)]   # per softmax warp: ("S", j) or ("P", j)
        self.v16 = [[None, None], [None, None]]     # V index in each half of each fp16 buffer
        self.pv_n = self.qk_n = 0
        self.fifo = [[]]
        self.landings = []

    def groups(self):
        n = self.n
        if self.e4:
            return [(g % 2 == 1, g // 2) for g in range(2 * n)]
        order = [(False, t) for t in range(min(2, n))]
        for j in range(n):
            order.append((True, j))
            if j + 2 < n:
                order.append((False, j + 2))
        return order

    def producer(self):
        if self.n == 0:
            return
        self.q_full.expect_tx()
        self.q_full.arrive()
        self.landings.append(("q",))
        it = 0
        for is_v, t in self.groups():
            for half in range(2):
                slot = it % self.S
                yield lambda s=slot, n=it // self.S - 1: self.kv_empty[s].passes(n)
                if self.slot_readers[slot]:
                    raise ProtocolError(f"slot {slot} refilled while {self.slot_item[slot]} is read")
                self.slot_item[slot] = None
                self.kv_full[slot].expect_tx()
                self.kv_full[slot].arrive()
                self.landings.append(("kv", slot, (is_v, t, half)))
                it += 1

    def issuer(self):
        n, S = self.n, self.S
        if n == 0:
            return
        yield lambda: self.q_full.passes(0)

        def wait_items(pos):
            for q in (pos, pos + 1):
                yield lambda q=q: self.kv_full[q % S].passes(q // S)

        def qk(j, b, pos):
            for q in (pos, pos + 1):
                self.slot_readers[q % S] += 1
            self.fifo[0] += [("qk", j, b, pos), ("commit", self.s_full[b]),
                             ("commit", self.kv_empty[pos % S]), ("commit", self.kv_empty[(pos + 1) % S])]

        it = 0
        for t in range(min(2, n)):
            pos = 4 * t if self.e4 else it
            yield from wait_items(pos)
            qk(t, t, pos)
            it += 2
        for j in range(n):
            b = j & 1
            if self.e4:
                yield lambda j=j: self.v16_full[j & 1].passes(j >> 1)
            else:
                yield from wait_items(it)
            yield lambda j=j, b=b: self.p_full[b].passes(j if self.mutant == "one_p_barrier" else j >> 1)
            ops = [("pv", j, b, None if self.e4 else it), ("commit", self.pv_done)]
            if j + 1 == n:
                ops.append(("commit", self.o_done))
            if self.e4:
                ops.append(("commit", self.v16_empty[b]))
            else:
                for q in (it, it + 1):
                    self.slot_readers[q % S] += 1
                ops += [("commit", self.kv_empty[it % S]), ("commit", self.kv_empty[(it + 1) % S])]
            self.fifo[0] += ops
            it += 2
            if j + 2 < n:
                pos = 4 * (j + 2) if self.e4 else it
                yield from wait_items(pos)
                qk(j + 2, b, pos)
                it += 2

    def converter(self, hh):
        for jv in range(self.n if self.e4 else 0):
            it = 4 * jv + 2 + hh
            slot = it % self.S
            yield lambda: self.kv_full[slot].passes(it // self.S)
            if self.slot_item[slot] != (True, jv, hh):
                raise ProtocolError(f"converter {hh} found {self.slot_item[slot]} for V_{jv}")
            self.slot_readers[slot] += 1
            yield None                                   # the half tile into registers
            self.slot_readers[slot] -= 1
            self.kv_empty[slot].arrive()
            yield lambda: self.v16_empty[jv & 1].passes((jv >> 1) - 1)
            if jv >= 2 and self.pv_n < jv - 1:
                raise ProtocolError(f"converter {hh} overwrote fp16 V_{jv - 2} before its P V")
            self.v16[jv & 1][hh] = None
            yield None                                   # conversion and stores
            self.v16[jv & 1][hh] = jv
            self.v16_full[jv & 1].arrive()

    def softmax(self, w):
        for j in range(self.n):
            b = j & 1
            yield lambda j=j, b=b: self.s_full[b].passes(j >> 1)
            if self.buf[b][w] != ("S", j):
                raise ProtocolError(f"softmax {w} step {j} found {self.buf[b][w]} in buffer {b}")
            yield None                                   # exponentials
            self.buf[b][w] = ("P", j)
            if j > 0 and self.rnd.random() < 0.3:        # this warp rescales O
                yield lambda j=j: self.pv_done.passes(j - 1)
                if self.pv_n != j:
                    raise ProtocolError(f"softmax {w} rescaled O at step {j} with {self.pv_n} P V done")
            yield None
            self.p_full[b].arrive()
        if self.n > 0:
            if self.mutant == "epilogue_on_pv_done":
                yield lambda: self.pv_done.passes(self.n - 1)
            else:
                yield lambda: self.o_done.passes(0)
            if self.pv_n != self.n:
                raise ProtocolError(f"epilogue read O with {self.pv_n} of {self.n} P V done")

    def land(self, ev):
        if ev[0] == "q":
            self.q_landed = True
            self.q_full.land()
        else:
            _, slot, item = ev
            self.slot_item[slot] = item
            self.kv_full[slot].land()

    def execute(self, _):
        op = self.fifo[0].pop(0)
        if op[0] == "commit":
            op[1].arrive()
            return
        kind, j, b, pos = op
        S = self.S
        if kind == "qk":
            got = [self.slot_item[q % S] for q in (pos, pos + 1)]
            if got != [(False, j, 0), (False, j, 1)] or not self.q_landed:
                raise ProtocolError(f"Q K^T {j} read {got}")
            if j >= 2 and (any(c != ("P", j - 2) for c in self.buf[b]) or self.pv_n < j - 1):
                raise ProtocolError(f"Q K^T {j} overwrote buffer {b} holding {self.buf[b]}")
            if self.qk_n != j:
                raise ProtocolError("score MMAs out of order")
            self.buf[b] = [("S", j)] * 4
            self.qk_n += 1
        else:
            if self.e4:
                if self.v16[b] != [j, j]:
                    raise ProtocolError(f"P V {j} read fp16 buffer {b} holding {self.v16[b]}")
            else:
                got = [self.slot_item[q % S] for q in (pos, pos + 1)]
                if got != [(True, j, 0), (True, j, 1)]:
                    raise ProtocolError(f"P V {j} read {got}")
                for q in (pos, pos + 1):
                    self.slot_readers[q % S] -= 1
            if any(c != ("P", j) for c in self.buf[b]) or self.pv_n != j:
                raise ProtocolError(f"P V {j} read buffer {b} holding {self.buf[b]}")
            self.pv_n += 1
            return
        for q in (pos, pos + 1):
            self.slot_readers[q % S] -= 1

    def agents(self):
        return ([self.producer(), self.issuer(), self.converter(0), self.converter(1)]
                + [self.softmax(w) for w in range(4)])

    def barriers(self):
        return ([self.q_full, self.pv_done, self.o_done] + self.s_full + list({id(b): b for b in self.p_full}.values())
                + self.v16_full + self.v16_empty + self.kv_full + self.kv_empty)

    def finish(self):
        if self.pv_n != self.n or self.qk_n != self.n:
            raise ProtocolError("not every MMA ran")


class KernelBwdDkdv(Model):
    """bwd_dkdv_kernel, one CTA: one 128-key tile of one K/V head, `steps`
    query tiles.  K and V are loaded once (kv_full); each step's item (Q, dO,
    lse and D of 128 queries) comes through a ring of `slots`.  The issuer sends
    S^T = K Q^T and dP^T = V dO^T (commit s_full), then for each half of the
    queries waits for that half's P^T / dS^T (p_half, 4 warps each), sends the
    accumulating dV, dK MMAs, and after both halves releases the item
    (item_empty); acc_done after the last step.  Eight elementwise warps, two
    groups of four (one per query half), read S^T, dP^T and the item's lse / D,
    write P^T / dS^T over their half's columns and arrive on p_half."""

    def __init__(self, steps, slots, seed):
        self.n, self.S = steps, slots
        self.rnd = random.Random(seed)
        self.kv_full = Bar("kv_full", 1)
        self.s_full = Bar("s_full", 1)
        self.p_half = [Bar("p_half0", 4), Bar("p_half1", 4)]
        self.acc_done = Bar("acc_done", 1)
        self.item_full = [Bar(f"item_full{s}", 1) for s in range(slots)]
        self.item_empty = [Bar(f"item_empty{s}", 1) for s in range(slots)]
        self.slot_item = [None] * slots
        self.slot_readers = [0] * slots
        self.kv_landed = False
        self.tm = [[None] * 4 for _ in range(2)]   # per query half, per warp: ("S", s) / ("P", s)
        self.acc_n = [0, 0]                         # accumulating MMAs done per half
        self.s_n = 0
        self.fifo = [[]]
        self.landings = []

    def producer(self):
        if self.n == 0:
            return
        self.kv_full.expect_tx()
        self.kv_full.arrive()
        self.landings.append(("kv",))
        for s in range(self.n):
            slot = s % self.S
            yield lambda sl=slot, k=s // self.S - 1: self.item_empty[sl].passes(k)
            if self.slot_readers[slot]:
                raise ProtocolError(f"item slot {slot} refilled while step {self.slot_item[slot]} is read")
            self.slot_item[slot] = None
            self.item_full[slot].expect_tx()
            self.item_full[slot].arrive()
            self.landings.append(("item", slot, s))

    def issuer(self):
        if self.n == 0:
            return
        yield lambda: self.kv_full.passes(0)
        for s in range(self.n):
            slot = s % self.S
            yield lambda sl=slot, k=s // self.S: self.item_full[sl].passes(k)
            self.slot_readers[slot] += 3             # S^T / dP^T, then dV / dK of each half
            self.fifo[0] += [("s", s, slot), ("commit", self.s_full)]
            for h in range(2):
                yield lambda h=h, s=s: self.p_half[h].passes(s)
                self.fifo[0].append(("acc", s, slot, h))
            self.fifo[0].append(("commit", self.item_empty[slot]))
        self.fifo[0].append(("commit", self.acc_done))

    def elementwise(self, h, w):
        for s in range(self.n):
            yield lambda s=s: self.s_full.passes(s)
            slot = s % self.S
            if self.tm[h][w] != ("S", s) or self.slot_item[slot] != s:
                raise ProtocolError(f"elementwise {h}.{w} step {s} found {self.tm[h][w]}, item "
                                    f"{self.slot_item[slot]}")
            self.slot_readers[slot] += 1             # lse, D of the item
            yield None
            self.slot_readers[slot] -= 1
            self.tm[h][w] = ("P", s)
            self.p_half[h].arrive()
        if self.n:
            yield lambda: self.acc_done.passes(0)
            if self.acc_n != [self.n, self.n]:
                raise ProtocolError("epilogue read dV / dK before the last accumulation")

    def land(self, ev):
        if ev[0] == "kv":
            self.kv_landed = True
            self.kv_full.land()
        else:
            self.slot_item[ev[1]] = ev[2]
            self.item_full[ev[1]].land()

    def execute(self, _):
        op = self.fifo[0].pop(0)
        if op[0] == "commit":
            op[1].arrive()
        elif op[0] == "s":
            _, s, slot = op
            if not self.kv_landed or self.slot_item[slot] != s:
                raise ProtocolError(f"S^T {s} read item {self.slot_item[slot]}")
            if s and (any(c != ("P", s - 1) for half in self.tm for c in half) or self.acc_n != [s, s]):
                raise ProtocolError(f"S^T {s} overwrote {self.tm} before the accumulations read it")
            self.tm = [[("S", s)] * 4 for _ in range(2)]
            self.s_n += 1
            self.slot_readers[slot] -= 1
        else:
            _, s, slot, h = op
            if self.slot_item[slot] != s or any(c != ("P", s) for c in self.tm[h]) or self.acc_n[h] != s:
                raise ProtocolError(f"dV / dK {s} half {h} read {self.tm[h]}, item {self.slot_item[slot]}")
            self.acc_n[h] += 1
            self.slot_readers[slot] -= 1

    def agents(self):
        return [self.producer(), self.issuer()] + [self.elementwise(h, w) for h in range(2)
                                                   for w in range(4)]

    def barriers(self):
        return ([self.kv_full, self.s_full, self.acc_done] + self.p_half + self.item_full
                + self.item_empty)

    def finish(self):
        if self.acc_n != [self.n, self.n]:
            raise ProtocolError("not every accumulation ran")


class KernelBwdDq(Model):
    """bwd_dq_kernel, one CTA: one 128-row query tile, n key tiles.  Q and dO
    are loaded once; K_j and V_j come through rings of their own (`ks`, `vs`
    slots).  S_j = Q K_j^T goes to score buffer j mod 2 and dS_j over it, dP_j
    to one dP buffer.  The issuer sends S_{j+1} at once, dP_{j+1} once dP_j has
    been read (dp_free), commits s_full, then for each half of the keys waits
    for that half of dS_j (p_half) and sends dQ += dS K_j; K_j is released after
    dQ_j, V_j after dP_j.  Four elementwise warps (one query row per thread)
    read S_j and dP_j per half, arrive on dp_free once all of dP_j is read,
    write dS over the S columns they read and arrive on p_half.  `robust`
    models p_half as one barrier per (half, step parity), which keeps every
    wait within one phase whatever the warps' relative speeds."""

    def __init__(self, n, seed, ks=3, vs=2, robust=False):
        self.n, self.KS, self.VS, self.robust = n, ks, vs, robust
        self.rnd = random.Random(seed)
        self.q_full = Bar("q_full", 1)
        self.s_full = Bar("s_full", 1)
        self.dp_free = Bar("dp_free", 4)
        self.acc_done = Bar("acc_done", 1)
        self.p_half = [[Bar(f"p_half{h}_{q}", 4) for q in range(2)] for h in range(2)]
        if not robust:
            self.p_half = [[b[0], b[0]] for b in self.p_half]
        self.k_full = [Bar(f"k_full{s}", 1) for s in range(ks)]
        self.k_empty = [Bar(f"k_empty{s}", 1) for s in range(ks)]
        self.v_full = [Bar(f"v_full{s}", 1) for s in range(vs)]
        self.v_empty = [Bar(f"v_empty{s}", 1) for s in range(vs)]
        self.k_item, self.v_item = [None] * ks, [None] * vs
        self.k_readers, self.v_readers = [0] * ks, [0] * vs
        self.q_landed = False
        self.sbuf = [[None] * 4 for _ in range(2)]  # per buffer, per warp: ("S", j) / ("dS", j)
        self.dp = [None] * 4                         # per warp: ("dP", j) or ("read", j)
        self.dq_n = [0, 0]
        self.fifo = [[]]
        self.landings = []

    def _p_wait(self, h, j):
        if self.robust:
            return lambda: self.p_half[h][j & 1].passes(j >> 1)
        return lambda: self.p_half[h][0].passes(j)

    def producer(self):
        if self.n == 0:
            return
        self.q_full.expect_tx()
        self.q_full.arrive()
        self.landings.append(("q",))
        for j in range(self.n):
            ks, vs = j % self.KS, j % self.VS
            yield lambda ks=ks, k=j // self.KS - 1: self.k_empty[ks].passes(k)
            if self.k_readers[ks]:
                raise ProtocolError(f"K slot {ks} refilled while K_{self.k_item[ks]} is read")
            self.k_item[ks] = None
            self.k_full[ks].expect_tx()
            self.k_full[ks].arrive()
            self.landings.append(("k", ks, j))
            yield lambda vs=vs, k=j // self.VS - 1: self.v_empty[vs].passes(k)
            if self.v_readers[vs]:
                raise ProtocolError(f"V slot {vs} refilled while V_{self.v_item[vs]} is read")
            self.v_item[vs] = None
            self.v_full[vs].expect_tx()
            self.v_full[vs].arrive()
            self.landings.append(("v", vs, j))

    def issuer(self):
        n, KS, VS = self.n, self.KS, self.VS
        if n == 0:
            return
        yield lambda: self.q_full.passes(0)
        yield lambda: self.k_full[0].passes(0)
        yield lambda: self.v_full[0].passes(0)
        self.k_readers[0] += 1
        self.v_readers[0] += 1
        self.fifo[0] += [("s", 0), ("dp", 0), ("commit", self.s_full), ("commit", self.v_empty[0])]
        for j in range(n):
            if j + 1 < n:
                yield lambda j=j: self.k_full[(j + 1) % KS].passes((j + 1) // KS)
                self.k_readers[(j + 1) % KS] += 1
                self.fifo[0].append(("s", j + 1))
                yield lambda j=j: self.v_full[(j + 1) % VS].passes((j + 1) // VS)
                yield lambda j=j: self.dp_free.passes(j)
                self.v_readers[(j + 1) % VS] += 1
                self.fifo[0] += [("dp", j + 1), ("commit", self.s_full),
                                 ("commit", self.v_empty[(j + 1) % VS])]
            self.k_readers[j % KS] += 1
            for h in range(2):
                yield self._p_wait(h, j)
                self.fifo[0].append(("dq", j, h))
            self.fifo[0].append(("commit", self.k_empty[j % KS]))
        self.fifo[0].append(("commit", self.acc_done))

    def elementwise(self, w):
        for j in range(self.n):
            b = j & 1
            yield lambda j=j: self.s_full.passes(j)
            for h in range(2):
                if self.sbuf[b][w] not in (("S", j), ("dS0", j)) or self.dp[w] not in (("dP", j), ("read", j)):
                    raise ProtocolError(f"elementwise {w} step {j} half {h} found {self.sbuf[b][w]}, "
                                        f"{self.dp[w]}")
                if h == 1:
                    self.dp[w] = ("read", j)
                    self.dp_free.arrive()
                yield None
                self.sbuf[b][w] = ("dS0", j) if h == 0 else ("dS", j)
                [self.p_half[h][j & 1] if self.robust else self.p_half[h][0]][0].arrive()
        if self.n:
            yield lambda: self.acc_done.passes(0)
            if self.dq_n != [self.n, self.n]:
                raise ProtocolError("epilogue read dQ before the last accumulation")

    def land(self, ev):
        if ev[0] == "q":
            self.q_landed = True
            self.q_full.land()
        elif ev[0] == "k":
            self.k_item[ev[1]] = ev[2]
            self.k_full[ev[1]].land()
        else:
            self.v_item[ev[1]] = ev[2]
            self.v_full[ev[1]].land()

    def execute(self, _):
        op = self.fifo[0].pop(0)
        if op[0] == "commit":
            op[1].arrive()
            return
        kind, j = op[0], op[1]
        b = j & 1
        if kind == "s":
            if not self.q_landed or self.k_item[j % self.KS] != j:
                raise ProtocolError(f"S_{j} read K_{self.k_item[j % self.KS]}")
            if j >= 2 and (any(c != ("dS", j - 2) for c in self.sbuf[b]) or self.dq_n != [j - 1, j - 1]):
                raise ProtocolError(f"S_{j} overwrote buffer {b} holding {self.sbuf[b]}")
            self.sbuf[b] = [("S", j)] * 4
            self.k_readers[j % self.KS] -= 1
        elif kind == "dp":
            if self.v_item[j % self.VS] != j:
                raise ProtocolError(f"dP_{j} read V_{self.v_item[j % self.VS]}")
            if j and any(c != ("read", j - 1) for c in self.dp):
                raise ProtocolError(f"dP_{j} overwrote dP still unread: {self.dp}")
            self.dp = [("dP", j)] * 4
            self.v_readers[j % self.VS] -= 1
        else:
            h = op[2]
            want = ("dS0", j) if h == 0 else ("dS", j)
            ok = all(c in (("dS0", j), ("dS", j)) for c in self.sbuf[b]) if h == 0 else \
                all(c == ("dS", j) for c in self.sbuf[b])
            if not ok or self.dq_n[h] != j or self.k_item[j % self.KS] != j:
                raise ProtocolError(f"dQ_{j} half {h} read {self.sbuf[b]} (want {want})")
            self.dq_n[h] += 1
            if h == 1:
                self.k_readers[j % self.KS] -= 1

    def agents(self):
        return [self.producer(), self.issuer()] + [self.elementwise(w) for w in range(4)]

    def barriers(self):
        ph = {id(b): b for row in self.p_half for b in row}.values()
        return ([self.q_full, self.s_full, self.dp_free, self.acc_done] + list(ph)
                + self.k_full + self.k_empty + self.v_full + self.v_empty)

    def finish(self):
        if self.dq_n != [self.n, self.n]:
            raise ProtocolError("not every dQ accumulation ran")
