"""Models of the kernel's barrier protocols, run on the CPU over random
interleavings of its roles: `simulate` for the three rotating score buffers
of the FA_SCORE_ROTATION build option (D=64), `simulate_default` for the
default order (one score buffer per slot, P published once per step, the
ring freed by the softmax in two-tile D=64 units, the V converters covering
the next K for bf16 at D=128).

Each role of one CTA (TMA loader, MMA issuer, the 4 warps of each softmax
warpgroup, the 4 epilogue warps, the 2 V converters of bf16 inputs) is a
generator that performs its arrivals and yields its waits in the kernel's
order; an arrival completes a barrier phase once the barrier's count is
reached.  MMAs, commits and copies take effect at issue, the most aggressive
timing for phase run-ahead.  A scheduler with random per-role speeds runs one
ready role at a time.  It reports:
  - deadlock (no role can move);
  - a wait whose parity is not its phase's, or that is evaluated while its
    barrier is not at that phase or the next (parity aliasing);
  - a score buffer read (by a softmax warp or a P*V) that holds another op's
    data, or written by a QK while it still holds live data;
  - a K/V ring entry overwritten before every MMA that reads it was issued;
  - O rescaled while one of the slot's P*Vs is still to be issued.
The `mistake` argument plants one known error so the tests can check that
the model catches it."""
import random


class Bar:
    def __init__(self, count):
        self.count, self.arr, self.C = count, 0, 0   # C: completed phases

    def arrive(self):
        self.arr += 1
        assert self.arr <= self.count, "more arrivals than the barrier's count"
        if self.arr == self.count:
            self.arr = 0
            self.C += 1


class OpMap:
    """A unit's ops: its two slots' key steps in issue order (both slots
    alternate while both have steps, then the longer one runs alone)."""

    def __init__(self, unit):
        j0, n0, n1 = unit
        c0, c1 = max(0, n0 - j0), max(0, n1 - j0)
        self.j0, self.cm, self.tl, self.n = j0, min(c0, c1), 0 if c0 > c1 else 1, c0 + c1

    def slot(self, m):
        return (m & 1) if m < 2 * self.cm else self.tl

    def step(self, m):
        return self.j0 + (m >> 1) if m < 2 * self.cm else self.j0 + m - self.cm

    def op(self, t, j):
        return 2 * (j - self.j0) + t if j - self.j0 < self.cm else j - self.j0 + self.cm

    def first_of_step(self, m):
        return m >= 2 * self.cm or not (m & 1)

    def last_of_step(self, m):
        return m >= 2 * self.cm or bool(m & 1)


class ProtocolError(AssertionError):
    pass


def simulate(units, kp, bf16, rng, mistake=None, full_pairs=None, kslots=None, pv_split=False):
    """units: (j0, nkv0, nkv1) per unit (nkv: end of the slot's steps, 0 =
    absent).  kp: key-parity units (one Q buffer, 4 double ring slots).
    pv_split: P published in two halves, the issuer waiting for each.
    Returns (True, None), or (False, waits) on deadlock; raises ProtocolError."""
    if full_pairs is None:
        full_pairs = not kp
    n_slots = kslots or (4 if kp else 8)
    n_pairs = n_slots // 2
    step_bars = 2 if mistake == "two_step_barriers" else 3
    loader_on_scores, n_sbars = False, 1   # (the loader below is shared in form with simulate_default's)
    look = 4 if mistake == "lookahead_too_deep" else 3
    B = {}
    for t in range(2):
        for name, c in (("QFull", 1), ("QEmpty", 1), ("OFull", 1), ("OEmpty", 4), ("StFull", 4), ("StEmpty", 4)):
            B[(name, t)] = Bar(c)
        for i in range(3):
            B[("SFull", t, i)] = Bar(1)
            B[("PHalf", t, i)] = Bar(4)
            B[("PFull", t, i)] = Bar(4)
        for i in range(2):
            B[("PVDone", t, i)] = Bar(1)
    for s in range(n_slots):
        B[("KVFull", s)] = Bar(2 if full_pairs else 1)
        B[("KVEmpty", s)] = Bar(1)
        B[("VConv", s)] = Bar(2)
    buf = [None] * 3              # (unit, op, state) of each score buffer
    slot_entry = [None] * n_slots
    reads_left = {}               # ring entry -> MMAs still to read it
    pv_issued = {}
    p_arrivals = {}
    e = 0
    for (j0, n0, n1) in units:
        for j in range(j0, max(n0, n1)):
            act = (j < n0) + (j < n1)
            reads_left[e] = reads_left[e + 1] = act
            e += 2

    def W(name, par, n):
        return ("wait", name, par, n)

    def check(cond, msg):
        if not cond:
            raise ProtocolError(msg)

    def loader():
        ph_qe, kvc, nq = 0, 0, [0, 0]
        g, cnt, hist = 0, [0, 0], [None, None]
        for (j0, n0, n1) in units:
            nkv = (n0, n1)
            for t in range(2):
                if nkv[t] == 0 or (kp and t == 1):
                    continue
                yield W(("QEmpty", t), ((ph_qe >> t) & 1) ^ 1, nq[t] - 1)
                ph_qe ^= 1 << t
                nq[t] += 1
                B[("QFull", t)].arrive()
            for j in range(j0, max(n0, n1)):
                last = 1 if j < n1 else 0
                info = (last, cnt[last])
                for kind in range(2):
                    idx, s = kvc, kvc % n_slots
                    if idx >= n_slots:
                        if loader_on_scores:
                            sl, n = hist[(g + kind) & 1]
                            yield W(("SFull", sl, n % n_sbars), (n // n_sbars) & 1, n // n_sbars)
                        else:
                            pr = (idx - n_slots + 1) // 2
                            yield W(("KVEmpty", pr % n_pairs), (pr // n_pairs) & 1, pr // n_pairs)
                        old = slot_entry[s]
                        check(reads_left[old] == 0, f"ring entry {old} overwritten with {reads_left[old]} reads left")
                    if kind == 0:
                        hist[g & 1] = info
                    kvc += 1
                    slot_entry[s] = idx
                    B[("KVFull", (idx // 2) % n_pairs if full_pairs else s)].arrive()
                for t in range(2):
                    cnt[t] += j < nkv[t]
                g += 1

    def converter():
        kvc = 0
        for (j0, n0, n1) in units:
            for _ in range(j0, max(n0, n1)):
                iv = kvc + 1
                kvc += 2
                if full_pairs:
                    q = iv // 2
                    yield W(("KVFull", q % n_pairs), (q // n_pairs) & 1, q // n_pairs)
                else:
                    yield W(("KVFull", iv % n_slots), (iv // n_slots) & 1, iv // n_slots)
                B[("VConv", iv % n_slots)].arrive()

    def issuer():
        ph_q = ph_oe = pph = 0
        kvc = 0
        qb, pb, pvn, nqf, noe = [0, 0], [0, 0], [0, 0], [0, 0], [0, 0]
        npw = {}

        def kv_wait(idx):
            if full_pairs:
                q = idx // 2
                yield W(("KVFull", q % n_pairs), (q // n_pairs) & 1, q // n_pairs)
            else:
                yield W(("KVFull", idx % n_slots), (idx // n_slots) & 1, idx // n_slots)

        def v_wait(idx):
            if bf16:
                yield W(("VConv", idx % n_slots), (idx // n_slots) & 1, idx // n_slots)
            else:
                yield from kv_wait(idx)

        def release(idx):
            B[("KVEmpty", ((idx + 1) // 2) % n_pairs)].arrive()

        def read_entry(idx):
            check(slot_entry[idx % n_slots] == idx, f"ring entry {idx} read while not in its slot")
            reads_left[idx] -= 1

        for ui, unit in enumerate(units):
            j0, n0, n1 = unit
            nkv, nmax, om = (n0, n1), max(n0, n1), OpMap(unit)
            if om.n == 0:
                continue
            kvb, k_in = kvc, [j0 - 1]
            pv_issued[(ui, 0)] = pv_issued[(ui, 1)] = 0

            def qk_op(m):
                nonlocal ph_q
                t, j = om.slot(m), om.step(m)
                if j == j0 and (not kp or t == 0):
                    yield W(("QFull", t), (ph_q >> t) & 1, nqf[t])
                    ph_q ^= 1 << t
                    nqf[t] += 1
                ik = kvb + 2 * (j - j0)
                if j > k_in[0]:
                    yield from kv_wait(ik)
                    k_in[0] = j
                read_entry(ik)
                b = m % 3
                check(buf[b] is None or buf[b][2] == "done", f"QK of op {m} overwrites buffer {b} holding {buf[b]}")
                buf[b] = (ui, m, "S")
                B[("SFull", t, qb[t])].arrive()
                qb[t] = (qb[t] + 1) % step_bars
                if (m == om.n - 1) if kp else (j == nkv[t] - 1):
                    B[("QEmpty", 0 if kp else t)].arrive()

            for m in range(min(om.n, look)):
                yield from qk_op(m)
            release(kvb)
            for m in range(om.n):
                t, j = om.slot(m), om.step(m)
                bi, iv = pb[t], kvb + 2 * (j - j0) + 1
                n_ = npw.get((t, bi), 0)
                yield W(("PHalf" if pv_split else "PFull", t, bi), (pph >> (3 * t + bi)) & 1, n_)
                if j == j0:
                    yield W(("OEmpty", t), ((ph_oe >> t) & 1) ^ 1, noe[t] - 1)
                    ph_oe ^= 1 << t
                    noe[t] += 1
                if not (full_pairs and not bf16) and om.first_of_step(m):
                    yield from v_wait(iv)
                if pv_split:
                    yield W(("PFull", t, bi), (pph >> (3 * t + bi)) & 1, n_)
                npw[(t, bi)] = n_ + 1
                pph ^= 1 << (3 * t + bi)
                pb[t] = (bi + 1) % step_bars
                check(buf[m % 3] == (ui, m, "P"), f"P*V of op {m} reads buffer holding {buf[m % 3]}")
                buf[m % 3] = (ui, m, "done")
                read_entry(iv)
                pv_issued[(ui, t)] += 1
                if j == nkv[t] - 1:
                    B[("OFull", t)].arrive()
                else:
                    B[("PVDone", t, pvn[t])].arrive()
                    pvn[t] ^= 1
                at = om.first_of_step(m) if mistake == "early_release" else om.last_of_step(m)
                if at and j + 1 < nmax:
                    release(iv + 1)
                if m + look < om.n:
                    yield from qk_op(m + look)
            kvc = kvb + 2 * (nmax - j0)

    def softmax(t):
        ph_s = sb = pvd = ph_te = nte = 0
        ns = [0, 0, 0]
        for ui, unit in enumerate(units):
            j0, n0, n1 = unit
            nkv = (n0, n1)[t]
            if nkv == 0:
                continue
            om = OpMap(unit)
            for j in range(j0, nkv):
                m, bs = om.op(t, j), sb
                yield W(("SFull", t, sb), (ph_s >> sb) & 1, ns[sb])
                ns[sb] += 1
                ph_s ^= 1 << sb
                sb = (sb + 1) % step_bars
                check(buf[m % 3] is not None and buf[m % 3][:2] == (ui, m),
                      f"softmax {t} reads op {m}'s scores from a buffer holding {buf[m % 3]}")
                rescale = j > j0 and rng.random() < 0.5
                if rescale:
                    if mistake != "no_pv_done_wait":
                        yield W(("PVDone", t, pvd & 1), (pvd >> 1) & 1, pvd >> 1)
                    pvd += 1
                    check(pv_issued[(ui, t)] == j - j0, "O rescaled while a P*V of the slot is outstanding")
                if pv_split:
                    B[("PHalf", t, bs)].arrive()
                p_arrivals[(ui, m)] = p_arrivals.get((ui, m), 0) + 1
                if p_arrivals[(ui, m)] == 4:
                    buf[m % 3] = (ui, m, "P")
                B[("PFull", t, bs)].arrive()
                if j > j0 and not rescale:
                    yield W(("PVDone", t, pvd & 1), (pvd >> 1) & 1, pvd >> 1)
                    pvd += 1
            yield W(("StEmpty", t), ph_te ^ 1, nte - 1)
            ph_te ^= 1
            nte += 1
            B[("StFull", t)].arrive()

    def epilogue():
        ph_o, no = 0, [0, 0]
        for (j0, n0, n1) in units:
            nkv = (n0, n1)
            if kp:
                if n0 == 0:
                    continue
                has1 = n1 > 0
                yield W(("OFull", 0), ph_o & 1, no[0])
                yield W(("StFull", 0), ph_o & 1, no[0])
                no[0] += 1
                if has1:
                    yield W(("OFull", 1), (ph_o >> 1) & 1, no[1])
                    yield W(("StFull", 1), (ph_o >> 1) & 1, no[1])
                    no[1] += 1
                ph_o ^= 3 if has1 else 1
                for t in range(2 if has1 else 1):
                    B[("StEmpty", t)].arrive()
                    B[("OEmpty", t)].arrive()
                continue
            for t in range(2):
                if nkv[t] == 0:
                    continue
                yield W(("OFull", t), (ph_o >> t) & 1, no[t])
                yield W(("StFull", t), (ph_o >> t) & 1, no[t])
                no[t] += 1
                ph_o ^= 1 << t
                B[("StEmpty", t)].arrive()
                B[("OEmpty", t)].arrive()

    roles = {"load": loader(), "mma": issuer()}
    for t in range(2):
        for w in range(4):
            roles[f"softmax{t}.{w}"] = softmax(t)
    for w in range(4):
        roles[f"epilogue.{w}"] = epilogue()
    if bf16:
        for w in range(2):
            roles[f"convert.{w}"] = converter()
    pending = {k: None for k in roles}
    done = set()
    speed = {k: rng.choice([0.02, 0.2, 1.0, 1.0, 5.0]) for k in roles}

    def advance(k):
        if pending[k] is None:
            try:
                pending[k] = next(roles[k])
            except StopIteration:
                done.add(k)
            return True
        _, name, par, n = pending[k]
        b = B[name]
        check(par == (n & 1), f"{k} waits {name} with parity {par} for phase {n}")
        check(n <= b.C <= n + 1, f"{k}: {name} has completed {b.C} phases while phase {n} is awaited (aliased)")
        if (b.C & 1) != par:
            pending[k] = None
            return True
        return False

    while len(done) < len(roles):
        live = sorted((k for k in roles if k not in done), key=lambda k: -rng.random() * speed[k])
        if not any(advance(k) for k in live):   # the first role (in random order) that can move
            return False, {k: pending[k] for k in roles if k not in done}
    return True, None


def random_units(rng, kp):
    """A CTA's unit list: two-tile units (equal slots, causal slot 1 one step
    longer, slot 1 absent, split-KV chunks starting past key step 0), or
    key-parity units (slot 0 with the even steps, slot 1 one fewer or equal)."""
    units = []
    for _ in range(rng.randint(1, 6)):
        if kp:
            count = rng.randint(1, 9)
            units.append((0, (count + 1) // 2, count // 2))
            continue
        n0, kind = rng.randint(1, 9), rng.random()
        if kind < 0.3:
            units.append((0, n0, n0))
        elif kind < 0.6:
            units.append((0, n0, n0 + 1))
        elif kind < 0.75:
            units.append((0, n0, 0))
        else:
            j0 = rng.randint(1, 6)
            end = j0 + rng.randint(1, 4)
            units.append((j0, end, end if rng.random() < 0.6 else 0))
    return units


def simulate_default(units, kp, bf16, rng, d128=False, softmax_release=False, covers_k=False, loader_on_scores=False,
                     mistake=None):
    """The default order (one score buffer per slot): per key step j, slot
    0's P*V then its QK(j+1), then slot 1's; P is published once per step.
    d128: head dim 128 (K and V on separate full barriers, a 4-entry ring;
    else a step's K and V share one, and two-tile units have 8 entries).
    softmax_release: the ring pair (V_{j-1}, K_j) is freed by warp 0 of the
    softmax warpgroup that sees step j's last scores (slot 1's, or slot 0's
    when slot 1 has no step j), not by an issuer commit.  covers_k (bf16,
    d128): the V converters announce V_j only once K_{j+1} has landed, and the
    issuer's wait for the converted V_j covers the next QKs' K.
    loader_on_scores (d128 two-tile): no ring release at all; before reusing
    the slots of the pair (V_{g-1}, K_g) the loader waits on the score barrier
    of key step g's last QK, each slot's score barriers alternating between
    two.  mistake="converter_skips_k": the issuer relies on covers_k, the
    converters do not wait for K_{j+1}; mistake="one_score_barrier": the
    loader waits on scores with one barrier per slot."""
    n_sbars = 2 if (loader_on_scores and mistake != "one_score_barrier") else 1
    full_pairs = not d128
    n_slots = 4 if (kp or d128) else 8
    n_pairs = n_slots // 2
    B = {}
    for t in range(2):
        for name, c in (("QFull", 1), ("QEmpty", 1), ("OFull", 1), ("OEmpty", 4), ("StFull", 4), ("StEmpty", 4),
                        ("PFull", 4)):
            B[(name, t)] = Bar(c)
        for i in range(2):
            B[("SFull", t, i)] = Bar(1)
    for s in range(n_slots):
        B[("KVFull", s)] = Bar(2 if full_pairs else 1)
        B[("KVEmpty", s)] = Bar(1)
        B[("VConv", s)] = Bar(2)
    S = [None, None]              # (unit, step, state) of each slot's score/P buffer
    slot_entry = [None] * n_slots
    reads_left = {}
    pv_issued = {}
    e = 0
    for (j0, n0, n1) in units:
        for j in range(j0, max(n0, n1)):
            reads_left[e] = reads_left[e + 1] = (j < n0) + (j < n1)
            e += 2

    def W(name, par, n):
        return ("wait", name, par, n)

    def check(cond, msg):
        if not cond:
            raise ProtocolError(msg)

    def release(idx):
        B[("KVEmpty", ((idx + 1) // 2) % n_pairs)].arrive()

    def loader():
        ph_qe, kvc, nq = 0, 0, [0, 0]
        g, cnt, hist = 0, [0, 0], [None, None]
        for (j0, n0, n1) in units:
            nkv = (n0, n1)
            for t in range(2):
                if nkv[t] == 0 or (kp and t == 1):
                    continue
                yield W(("QEmpty", t), ((ph_qe >> t) & 1) ^ 1, nq[t] - 1)
                ph_qe ^= 1 << t
                nq[t] += 1
                B[("QFull", t)].arrive()
            for j in range(j0, max(n0, n1)):
                last = 1 if j < n1 else 0
                info = (last, cnt[last])
                for kind in range(2):
                    idx, s = kvc, kvc % n_slots
                    if idx >= n_slots:
                        if loader_on_scores:
                            sl, n = hist[(g + kind) & 1]
                            yield W(("SFull", sl, n % n_sbars), (n // n_sbars) & 1, n // n_sbars)
                        else:
                            pr = (idx - n_slots + 1) // 2
                            yield W(("KVEmpty", pr % n_pairs), (pr // n_pairs) & 1, pr // n_pairs)
                        old = slot_entry[s]
                        check(reads_left[old] == 0, f"ring entry {old} overwritten with {reads_left[old]} reads left")
                    if kind == 0:
                        hist[g & 1] = info
                    kvc += 1
                    slot_entry[s] = idx
                    B[("KVFull", (idx // 2) % n_pairs if full_pairs else s)].arrive()
                for t in range(2):
                    cnt[t] += j < nkv[t]
                g += 1

    def converter():
        kvc = 0
        for (j0, n0, n1) in units:
            nmax = max(n0, n1)
            for j in range(j0, nmax):
                iv = kvc + 1
                kvc += 2
                if full_pairs:
                    q = iv // 2
                    yield W(("KVFull", q % n_pairs), (q // n_pairs) & 1, q // n_pairs)
                else:
                    yield W(("KVFull", iv % n_slots), (iv // n_slots) & 1, iv // n_slots)
                if covers_k and j + 1 < nmax and mistake != "converter_skips_k":
                    ik = iv + 1
                    yield W(("KVFull", ik % n_slots), (ik // n_slots) & 1, ik // n_slots)
                B[("VConv", iv % n_slots)].arrive()

    def issuer():
        ph_q = ph_p = ph_oe = 0
        kvc = 0
        nqf, noe, npf = [0, 0], [0, 0], [0, 0]

        def kv_wait(idx):
            if full_pairs:
                q = idx // 2
                yield W(("KVFull", q % n_pairs), (q // n_pairs) & 1, q // n_pairs)
            else:
                yield W(("KVFull", idx % n_slots), (idx // n_slots) & 1, idx // n_slots)

        def v_wait(idx):
            if bf16:
                yield W(("VConv", idx % n_slots), (idx // n_slots) & 1, idx // n_slots)
            else:
                yield from kv_wait(idx)

        def read_entry(idx):
            check(slot_entry[idx % n_slots] == idx, f"ring entry {idx} read while not in its slot")
            reads_left[idx] -= 1

        sq = [0, 0]

        def qk(ui, t, j, idx):
            read_entry(idx)
            check(S[t] is None or S[t][2] == "done", f"QK of slot {t} step {j} overwrites {S[t]}")
            S[t] = (ui, j, "S")
            B[("SFull", t, sq[t])].arrive()
            sq[t] = (sq[t] + 1) % n_sbars

        for ui, (j0, n0, n1) in enumerate(units):
            nkv, nmax = (n0, n1), max(n0, n1)
            kvb = kvc
            pv_issued[(ui, 0)] = pv_issued[(ui, 1)] = 0
            k_in = False
            qe_slot = (0 if n0 > n1 else 1) if kp else 0
            for t in range(2):
                if nkv[t] == 0:
                    continue
                if not kp or t == 0:
                    yield W(("QFull", t), (ph_q >> t) & 1, nqf[t])
                    ph_q ^= 1 << t
                    nqf[t] += 1
                if not k_in:
                    yield from kv_wait(kvb)
                    k_in = True
                qk(ui, t, j0, kvb)
                if nkv[t] == j0 + 1 and (not kp or t == qe_slot):
                    B[("QEmpty", 0 if kp else t)].arrive()
            if not softmax_release and not loader_on_scores:
                release(kvb)
            for j in range(j0, nmax):
                iv, ik = kvb + 2 * (j - j0) + 1, kvb + 2 * (j - j0) + 2
                v_ready = full_pairs and not bf16
                k_ready = False
                for t in range(2):
                    if j < nkv[t]:
                        yield W(("PFull", t), (ph_p >> t) & 1, npf[t])
                        ph_p ^= 1 << t
                        npf[t] += 1
                        if j == j0:
                            yield W(("OEmpty", t), ((ph_oe >> t) & 1) ^ 1, noe[t] - 1)
                            ph_oe ^= 1 << t
                            noe[t] += 1
                        if not v_ready:
                            yield from v_wait(iv)
                            v_ready = True
                        check(S[t] == (ui, j, "P"), f"P*V of slot {t} step {j} reads {S[t]}")
                        S[t] = (ui, j, "done")
                        read_entry(iv)
                        pv_issued[(ui, t)] += 1
                        if j == nkv[t] - 1:
                            B[("OFull", t)].arrive()
                    if j + 1 < nkv[t]:
                        if not k_ready:
                            if not covers_k:
                                yield from kv_wait(ik)
                            k_ready = True
                        qk(ui, t, j + 1, ik)
                        if j + 1 == nkv[t] - 1 and (not kp or t == qe_slot):
                            B[("QEmpty", 0 if kp else t)].arrive()
                if not softmax_release and not loader_on_scores and j + 1 < nmax:
                    release(ik)
            kvc = kvb + 2 * (nmax - j0)

    def softmax(t, w):
        ph_te = nte = sb = 0
        ns = [0, 0]
        kv_next = 0
        for ui, (j0, n0, n1) in enumerate(units):
            nkv = (n0, n1)[t]
            kvb = kv_next
            kv_next += 2 * max(0, max(n0, n1) - j0)
            if nkv == 0:
                continue
            for j in range(j0, nkv):
                yield W(("SFull", t, sb), ns[sb] & 1, ns[sb])
                ns[sb] += 1
                sb = (sb + 1) % n_sbars
                check(S[t] is not None and S[t][:2] == (ui, j), f"softmax {t} step {j} reads {S[t]}")
                # O is stable: the commit that announced these scores covers the slot's previous P*V
                check(pv_issued[(ui, t)] == j - j0, "scores announced with a P*V of the slot outstanding")
                if softmax_release and w == 0 and (t == 1 or j >= n1):
                    release(kvb + 2 * (j - j0))
                if w == 3:
                    S[t] = (ui, j, "P")   # the last of the four warps publishes
                B[("PFull", t)].arrive()
            yield W(("StEmpty", t), ph_te ^ 1, nte - 1)
            ph_te ^= 1
            nte += 1
            B[("StFull", t)].arrive()

    def epilogue():
        ph_o, no = 0, [0, 0]
        for (j0, n0, n1) in units:
            nkv = (n0, n1)
            if kp:
                if n0 == 0:
                    continue
                has1 = n1 > 0
                yield W(("OFull", 0), ph_o & 1, no[0])
                yield W(("StFull", 0), ph_o & 1, no[0])
                no[0] += 1
                if has1:
                    yield W(("OFull", 1), (ph_o >> 1) & 1, no[1])
                    yield W(("StFull", 1), (ph_o >> 1) & 1, no[1])
                    no[1] += 1
                ph_o ^= 3 if has1 else 1
                for t in range(2 if has1 else 1):
                    B[("StEmpty", t)].arrive()
                    B[("OEmpty", t)].arrive()
                continue
            for t in range(2):
                if nkv[t] == 0:
                    continue
                yield W(("OFull", t), (ph_o >> t) & 1, no[t])
                yield W(("StFull", t), (ph_o >> t) & 1, no[t])
                no[t] += 1
                ph_o ^= 1 << t
                B[("StEmpty", t)].arrive()
                B[("OEmpty", t)].arrive()

    roles = {"load": loader(), "mma": issuer()}
    for t in range(2):
        for w in range(4):
            roles[f"softmax{t}.{w}"] = softmax(t, w)
    for w in range(4):
        roles[f"epilogue.{w}"] = epilogue()
    if bf16:
        for w in range(2):
            roles[f"convert.{w}"] = converter()
    return _run_roles(roles, B, rng)


def _run_roles(roles, B, rng):
    pending = {k: None for k in roles}
    done = set()
    speed = {k: rng.choice([0.02, 0.2, 1.0, 1.0, 5.0]) for k in roles}

    def advance(k):
        if pending[k] is None:
            try:
                pending[k] = next(roles[k])
            except StopIteration:
                done.add(k)
            return True
        _, name, par, n = pending[k]
        b = B[name]
        if par != (n & 1):
            raise ProtocolError(f"{k} waits {name} with parity {par} for phase {n}")
        if not n <= b.C <= n + 1:
            raise ProtocolError(f"{k}: {name} has completed {b.C} phases while phase {n} is awaited (aliased)")
        if (b.C & 1) != par:
            pending[k] = None
            return True
        return False

    while len(done) < len(roles):
        live = sorted((k for k in roles if k not in done), key=lambda k: -rng.random() * speed[k])
        if not any(advance(k) for k in live):
            return False, {k: pending[k] for k in roles if k not in done}
    return True, None
