"""Host-side model of one CTA of the persistent attention kernel, all roles at once (no GPU needed).

attn_fwd_ws.cuh runs a producer warp (TMA loads), eight prologue warps (QK-norm + RoPE in place),
three MMA-issuing threads (S jobs; P.V jobs of each query tile) and four softmax warps per query
tile, which hand work to each other through mbarriers waited by phase parity. This model restates each role's sequence of waits, arrivals, TMA
loads, MMA issues and commits (the same order and the same phase arithmetic as the kernel) as a
Python generator, and runs them under random interleavings together with
- an in-order tensor pipe shared by the issuing threads: MMAs and commits complete in the order they
  were issued, a commit arriving once everything issued before it is done, at random later times;
- a TMA engine that completes loads in any order, at random times;
- mbarriers with arrival counts, transaction bytes and phases.

Each wait is checked for exactness: a parity wait is only correct while the barrier is at most one
phase ahead of the phase the waiter means (two ahead reads as not yet complete and hangs, one behind
reads as complete too early). Each data access is checked too: S, P and O in the TMEM buffers, Q
tiles and K/V ring stages in shared memory must hold the tile of the job that reads them, and a
buffer or stage may only be overwritten once its last reader is done. Runs cover the D = 64
configuration (two Q slots, 4-stage ring, three S/P buffers) and D = 128 (one Q slot, 2-stage ring,
two buffers), several shapes, windows and random ticket splits, and must finish without deadlock.
"""
import random

import pytest

from test_ring_schedule import KT, shared_steps, ticket_decode, unit_geom


class Deadlock(Exception):
    pass


class Bar:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pending, self.tx, self.completed = count, 0, 0

    def arrive(self, tx=0):
        self.tx += tx
        self.pending -= 1
        assert self.pending >= 0, f"{self.name}: more arrivals than its count in one phase"
        self._maybe_complete()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        assert self.tx >= 0, f"{self.name}: transaction bytes below zero"
        self._maybe_complete()

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.completed += 1
            self.pending = self.count


def units_for(B, H, T, window, causal, tickets, S, n_long=0):
    """The CTA's units in order, with r_in / r_out (the producer's decode and reuse rule)."""
    n_qb = (T + 2 * KT - 1) // (2 * KT)
    out = []
    for c in tickets:
        bh, qb, left = ticket_decode(c, B * H, n_qb, 1 << 20, n_long)
        first, r_prev = True, 0
        while left:
            g = unit_geom(T, window, causal, bh, qb)
            g["r_in"] = 0 if first else r_prev
            first = False
            g["r_out"] = 0
            if left >= 2:
                nb = unit_geom(T, window, causal, bh, qb - 1)
                R = nb["ke_all"] - g["kb_all"] + 1
                g["r_out"] = R if (shared_steps(g, nb) and R <= S) else 0
            r_prev = g["r_out"]
            for t in range(2):
                qs = g["qs0"] + KT * t
                if qs < T:
                    qe = min(T - 1, qs + KT - 1)
                    lo = max(0, qs - window) if window >= 0 else 0
                    hi = qe if causal else (min(T - 1, qe + window) if window >= 0 else T - 1)
                    g[f"kb{t}"], g[f"ke{t}"] = lo // KT, hi // KT
                else:
                    g[f"kb{t}"], g[f"ke{t}"] = 1, 0
            out.append(g)
            left, qb = left - 1, qb - 1
    return out


def has(g, t, j):
    return g[f"kb{t}"] <= j <= g[f"ke{t}"]


def valid(g, t):
    return g[f"kb{t}"] <= g[f"ke{t}"]


class CTA:
    def __init__(self, units, S, NB, QS, rng, rescale_prob=0.3, q_release=True, softmax_release=True):
        self.units, self.S, self.NB, self.QS, self.rng = units, S, NB, QS, rng
        self.rescale_prob = rescale_prob
        b = {}

        def mk(name, count, n=1):
            b[name] = [Bar(f"{name}[{i}]", count) for i in range(n)]

        # a Q slot is freed by the S issuer's commit after the unit's last S job, both P.V issuers and
        # the eight softmax warps (after reading the slot's unit id and geometry)
        mk("QFull", 1, 2); mk("QReady", 8, 2); mk("Unit", 1, 2)
        mk("QEmpty", (1 if q_release else 0) + 2 + (8 if softmax_release else 0), 2)
        self.q_release, self.softmax_release = q_release, softmax_release
        mk("KFull", 1, S); mk("KReady", 8, S); mk("VFull", 1, S); mk("KFree", 1, S); mk("VFree", 2, S)
        mk("SFull", 1, 4); mk("BufFree", 1, NB); mk("PFull", 4, 4); mk("PVDone", 1, 4); mk("Final", 1, 3)
        self.b = b
        # shared state of the CTA
        self.unit_id = [None, None]
        self.unit_geo = [None, None]
        self.qtile = {}      # (slot, t) -> ("raw"|"hat"|"free", unit index)
        self.q_left = {}     # (slot, t) -> S jobs of the slot's unit still to read the Q^ tile
        self.kstage = {}     # stage -> ("raw"|"hat", (bh, j)) ; K
        self.vstage = {}     # stage -> (bh, j) ; V
        self.buf = {}        # (buffer, warp) -> ("S"|"P"|"Pread", global job): the warp's 32 TMEM lanes
        self.o = [None, None]  # O_t: (unit index, job index in tile of the last P.V)
        self.o_read = [{}, {}]  # tile t: softmax warp -> the unit whose O rows it has read
        self.pipe = []       # tensor pipe queue
        self.tma = []        # loads in flight
        self.jobs = {}       # global S job -> dict(t, unit, j, slot, pos, n)

    # ---- helpers used by the roles ----
    def wait(self, bar, k):
        """Parity wait for phase k of `bar` (k = -1: the phase before the first, already done)."""
        return ("wait", bar, k)


def producer(c):
    S, QS = c.S, c.QS
    kcnt = 0
    for ul in range(len(c.units) + 1):
        slot, ph = ul % QS, ul // QS
        yield c.wait(c.b["QEmpty"][slot], ph - 1)
        g = c.units[ul] if ul < len(c.units) else None
        c.unit_id[slot] = ul if g else -1
        c.unit_geo[slot] = g
        c.b["Unit"][slot].arrive()
        if g is None:
            c.b["QFull"][slot].arrive()
            return
        two = valid(g, 1)
        c.b["QFull"][slot].arrive(tx=2 if two else 1)
        for t in range(2 if two else 1):
            assert c.qtile.get((slot, t), ("free",))[0] == "free", "Q slot reloaded while in use"
            c.tma.append(("Q", (slot, t), ul, c.b["QFull"][slot]))
        for i in range(g["r_in"], g["n"]):
            j = g["ke_all"] - i
            st, ph = kcnt % S, kcnt // S
            yield c.wait(c.b["KFree"][st], ph - 1)
            yield c.wait(c.b["VFree"][st], ph - 1)
            c.b["KFull"][st].arrive(tx=1)
            c.tma.append(("K", st, (g["bh"], j), c.b["KFull"][st]))
            c.b["VFull"][st].arrive(tx=1)
            c.tma.append(("V", st, (g["bh"], j), c.b["VFull"][st]))
            kcnt += 1


def prologue(c, w):
    S, QS = c.S, c.QS
    kcnt = 0
    for ul in range(len(c.units) + 1):
        slot, ph = ul % QS, ul // QS
        yield c.wait(c.b["QFull"][slot], ph)
        if c.unit_id[slot] == -1:
            return
        u = c.unit_id[slot]
        g = dict(c.unit_geo[slot])
        assert u == ul
        n_jobs = 2 + g["n"] - g["r_in"]
        for jb in range(n_jobs):
            if jb < 2:
                if not valid(g, jb):
                    if jb == 1:
                        c.b["QReady"][slot].arrive()
                    continue
                cur = c.qtile[(slot, jb)]
                assert cur[1] == u and cur[0] in ("raw", "hat"), f"prologue sees Q {cur}, unit {u}"
                if w == 7:
                    c.qtile[(slot, jb)] = ("hat", u)
                if jb == 1:
                    c.b["QReady"][slot].arrive()
            else:
                st = kcnt % S
                yield c.wait(c.b["KFull"][st], kcnt // S)
                j = g["ke_all"] - (g["r_in"] + jb - 2)
                cur = c.kstage[st]
                assert cur[1] == (g["bh"], j) and cur[0] in ("raw", "hat"), f"prologue sees K {cur}"
                if w == 7:
                    c.kstage[st] = ("hat", cur[1])
                c.b["KReady"][st].arrive()
                kcnt += 1
            yield ("work",)


def s_issuer(c, pv_lag=True, buf_free=True):
    """S issuer: S jobs in stream order; each waits for its buffer's previous P.V (buffer-free) and for
    the tile's P.V job n - 2."""
    S, NB, QS = c.S, c.NB, c.QS
    gS = kc = 0
    scnt = [0, 0]
    for ul in range(len(c.units) + 1):
        slot, ph = ul % QS, ul // QS
        yield c.wait(c.b["Unit"][slot], ph)
        if c.unit_id[slot] == -1:
            break
        u = c.unit_id[slot]
        yield c.wait(c.b["QReady"][slot], ph)
        g = dict(c.unit_geo[slot])
        n_st = g["n"]
        for t in range(2):
            c.q_left[(slot, t)] = sum(has(g, t, g["ke_all"] - i) for i in range(n_st))
        for i in range(n_st):
            j = g["ke_all"] - i
            if i < g["r_in"]:
                pos = kc - g["r_in"] + i
            else:
                pos = kc
                kc += 1
            st = pos % S
            yield c.wait(c.b["KReady"][st], pos // S)
            h1 = has(g, 1, j)
            for t in range(2):
                if not has(g, t, j):
                    continue
                b = gS % NB
                sc = scnt[t]
                if buf_free:
                    yield c.wait(c.b["BufFree"][b], gS // NB - 1)
                if pv_lag and sc >= 2:
                    yield c.wait(c.b["PVDone"][2 * t + (sc & 1)], (sc - 2) >> 1)
                c.jobs[gS] = dict(t=t, n=sc, unit=u, j=j, slot=slot, pos=pos, bh=g["bh"], buf=b,
                                  first=(j == g[f"ke{t}"]))
                c.pipe.append(("S", gS))
                c.pipe.append(("commit", c.b["SFull"][2 * t + (sc & 1)]))
                scnt[t] += 1
                gS += 1
            if i < n_st - g["r_out"]:
                c.pipe.append(("commit", c.b["KFree"][st]))
        if c.q_release:
            c.pipe.append(("commit", c.b["QEmpty"][slot]))
    c.pipe.append(("commit", c.b["Final"][0]))
    yield c.wait(c.b["Final"][0], 0)


def pv_issuer(c, t):
    """P.V issuer of query tile t: observes every key step's V, issues the tile's P.V jobs in order."""
    S, NB, QS = c.S, c.NB, c.QS
    gS = kc = pcnt = 0
    for ul in range(len(c.units) + 1):
        slot, ph = ul % QS, ul // QS
        yield c.wait(c.b["Unit"][slot], ph)
        if c.unit_id[slot] == -1:
            break
        g = dict(c.unit_geo[slot])
        c.b["QEmpty"][slot].arrive()
        n_st = g["n"]
        for i in range(n_st):
            j = g["ke_all"] - i
            h0, h1 = has(g, 0, j), has(g, 1, j)
            gj = gS + (1 if (t == 1 and h0) else 0)
            gS += h0 + h1
            if i < g["r_in"]:
                pos = kc - g["r_in"] + i
            else:
                pos = kc
                kc += 1
            st = pos % S
            release = i < n_st - g["r_out"]
            yield c.wait(c.b["VFull"][st], pos // S)
            if not (h0 if t == 0 else h1):
                if release:
                    c.b["VFree"][st].arrive()
                continue
            k = pcnt
            pcnt += 1
            yield c.wait(c.b["PFull"][2 * t + (k & 1)], k >> 1)
            J = c.jobs[gj]
            assert (J["t"], J["n"]) == (t, k), f"P.V issuer {t} job {k} meets S job {gj} = {J}"
            c.pipe.append(("PV", gj))
            c.pipe.append(("commit", c.b["BufFree"][gj % NB]))
            c.pipe.append(("commit", c.b["PVDone"][2 * t + (k & 1)]))
            if release:
                c.pipe.append(("commit", c.b["VFree"][st]))
    c.pipe.append(("commit", c.b["Final"][1 + t]))
    yield c.wait(c.b["Final"][1 + t], 0)


def softmax(c, t, w):
    QS, NB = c.QS, c.NB
    n = 0
    gS = 0
    for ul in range(len(c.units) + 1):
        slot, ph = ul % QS, ul // QS
        yield c.wait(c.b["Unit"][slot], ph)
        if c.unit_id[slot] == -1:
            return
        u = c.unit_id[slot]
        g = dict(c.unit_geo[slot])
        if c.softmax_release:
            c.b["QEmpty"][slot].arrive()
        for j in range(g["ke_all"], g["kb_all"] - 1, -1):
            h0, h1 = has(g, 0, j), has(g, 1, j)
            gj = gS + (1 if (t == 1 and h0) else 0)
            gS += h0 + h1
            if not has(g, t, j):
                continue
            b = gj % NB
            yield c.wait(c.b["SFull"][2 * t + (n & 1)], n >> 1)
            assert c.buf.get((b, w)) == ("S", gj), f"softmax t{t}.{w} job {gj} reads {c.buf.get((b, w))}"
            J = c.jobs[gj]
            assert (J["t"], J["n"], J["unit"], J["j"]) == (t, n, u, j)
            yield ("work",)
            if j < g[f"ke{t}"] and c.rng.random() < c.rescale_prob:   # O rescale (data dependent)
                yield c.wait(c.b["PVDone"][2 * t + ((n - 1) & 1)], (n - 1) >> 1)
                assert c.o[t] == (u, n - 1), f"rescale of O_{t} at job {n} sees {c.o[t]}"
            assert c.buf.get((b, w)) == ("S", gj), "S overwritten while the softmax reads it"
            c.buf[(b, w)] = ("P", gj)
            c.b["PFull"][2 * t + (n & 1)].arrive()
            n += 1
        if not valid(g, t):
            continue
        # epilogue: every warp reads its own rows of O_t and stores them
        yield c.wait(c.b["PVDone"][2 * t + ((n - 1) & 1)], (n - 1) >> 1)
        assert c.o[t] == (u, n - 1), f"epilogue of O_{t} unit {u} sees {c.o[t]}"
        yield ("work",)
        assert c.o[t] == (u, n - 1), f"O_{t} overwritten while warp {w} reads it"
        c.o_read[t][w] = u


def tensor_pipe(c):
    """Executes the issuing thread's MMAs and commits in order, one per scheduling step."""
    while True:
        if not c.pipe:
            yield ("idle",)
            continue
        op = c.pipe.pop(0)
        if op[0] == "commit":
            op[1].arrive()
        elif op[0] == "S":
            J = c.jobs[op[1]]
            b = J["buf"]
            for w in range(4):
                prev = c.buf.get((b, w))
                assert prev is None or prev[0] == "Pread", f"S job {op[1]} overwrites buffer {b} holding {prev}"
            assert c.qtile[(J["slot"], J["t"])] == ("hat", J["unit"]), "S reads an untransformed Q tile"
            assert c.kstage[J["pos"] % c.S] == ("hat", (J["bh"], J["j"])), "S reads the wrong K stage"
            for w in range(4):
                c.buf[(b, w)] = ("S", op[1])
            key = (J["slot"], J["t"])
            c.q_left[key] -= 1
            if c.q_left[key] == 0:  # the unit's last reader of this Q^ tile
                c.qtile[key] = ("free", J["unit"])
        else:  # P.V
            J = c.jobs[op[1]]
            t, n = J["t"], J["n"]
            for w in range(4):
                got = c.buf.get((J["buf"], w))
                assert got == ("P", op[1]), f"P.V {op[1]} reads buffer {J['buf']} lanes of warp {w}: {got}"
            assert c.vstage[J["pos"] % c.S] == (J["bh"], J["j"]), "P.V reads the wrong V stage"
            if J["first"]:
                if c.o[t] is not None:
                    prev = c.o[t][0]
                    assert all(c.o_read[t].get(w) == prev for w in range(4)), \
                        f"O_{t} restarted before every warp read unit {prev}: {c.o_read[t]}"
            else:
                assert c.o[t] == (J["unit"], n - 1), f"O_{t} accumulation out of order: {c.o[t]}, job {n}"
            c.o[t] = (J["unit"], n)
            for w in range(4):
                c.buf[(J["buf"], w)] = ("Pread", op[1])
        yield ("work",)


def tma_engine(c):
    """Completes TMA loads in a random order."""
    while True:
        if not c.tma:
            yield ("idle",)
            continue
        ld = c.tma.pop(c.rng.randrange(len(c.tma)))
        kind, dst, what, bar = ld
        if kind == "Q":
            c.qtile[dst] = ("raw", what)
        elif kind == "K":
            c.kstage[dst] = ("raw", what)
        else:
            c.vstage[dst] = what
        bar.complete_tx(1)
        yield ("work",)


def run_cta(units, S, NB, QS, seed, max_steps=2_000_000, q_release=True, softmax_release=True, **issuer_flags):
    rng = random.Random(seed)
    c = CTA(units, S, NB, QS, rng, q_release=q_release, softmax_release=softmax_release)
    procs = {"producer": producer(c), "s_issuer": s_issuer(c, **issuer_flags), "pv0": pv_issuer(c, 0),
             "pv1": pv_issuer(c, 1)}
    for w in range(8):
        procs[f"prologue{w}"] = prologue(c, w)
    for t in range(2):
        for w in range(4):
            procs[f"softmax{t}.{w}"] = softmax(c, t, w)
    engines = {"tensor": tensor_pipe(c), "tma": tma_engine(c)}
    pending = {k: None for k in procs}  # the action each process is blocked on
    steps = 0
    while procs:
        steps += 1
        assert steps < max_steps, "model did not finish"
        runnable = []
        for k, act in pending.items():
            if act is None:
                runnable.append(k)
                continue
            _, bar, kph = act
            done = bar.completed
            # exactness: the barrier may be at phase kph (still running) or kph + 1 (done), nothing else
            assert kph <= done <= kph + 1, f"{k}: waits phase {kph} of {bar.name}, which completed {done}"
            if done == kph + 1:
                runnable.append(k)
        busy_engines = [e for e in engines if (e == "tensor" and c.pipe) or (e == "tma" and c.tma)]
        choices = runnable + busy_engines
        if not choices:
            raise Deadlock(f"blocked: {[(k, a[1].name, a[2]) for k, a in pending.items()]}")
        who = rng.choice(choices)
        if who in engines:
            next(engines[who])
            continue
        try:
            act = next(procs[who])
        except StopIteration:
            del procs[who]
            del pending[who]
            continue
        pending[who] = act if act[0] == "wait" else None
    return c


CONFIGS = {64: (4, 3, 2), 128: (2, 2, 1)}  # D -> (ring stages, S/P buffers, Q slots)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("T,window,causal", [(1024, 512, True), (1024, -1, True), (700, 100, True),
                                             (300, -1, False), (513, 0, True), (129, 5, True),
                                             (900, 200, False), (2048, 1024, True)])
def test_protocol_has_no_deadlock_and_exact_waits(D, T, window, causal):
    S, NB, QS = CONFIGS[D]
    B, H = 1, 2
    n_qb = (T + 2 * KT - 1) // (2 * KT)
    n_tickets = B * H * ((n_qb + 1) // 2)
    rnd = random.Random(T + window)
    for trial in range(6):
        tickets = sorted(rnd.sample(range(n_tickets), k=max(1, min(n_tickets, rnd.randint(1, 4)))))
        units = units_for(B, H, T, window, causal, tickets, S)
        c = run_cta(units, S, NB, QS, seed=1000 * trial + T + window)
        assert all(b.completed == 1 for b in c.b["Final"])


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("T,window", [(1024, 512), (1024, 256), (1024, 128), (1500, 300), (2048, 200)])
def test_protocol_with_whole_head_tickets(D, T, window):
    """Tickets of all the blocks of a head (every unit keeps tiles resident for the next; a tile can
    serve three units), mixed with pair tickets of another head."""
    S, NB, QS = CONFIGS[D]
    if window > S * KT:
        pytest.skip("no key tiles shared at this ring depth")
    B, H, n_long = 1, 2, 1
    n_qb = (T + 2 * KT - 1) // (2 * KT)
    n_tickets = n_long + (B * H - n_long) * ((n_qb + 1) // 2)
    rnd = random.Random(T * 3 + window)
    for trial in range(4):
        tickets = [0] + sorted(rnd.sample(range(1, n_tickets), k=min(n_tickets - 1, rnd.randint(0, 3))))
        units = units_for(B, H, T, window, True, tickets, S, n_long)
        assert sum(1 for g in units if g["r_in"] > 0) >= n_qb - 1  # the whole head chains its units
        c = run_cta(units, S, NB, QS, seed=7000 * trial + T + window)
        assert all(b.completed == 1 for b in c.b["Final"])


@pytest.mark.parametrize("flag", ["pv_lag", "buf_free", "q_release", "softmax_release"])
def test_model_catches_removed_rules(flag):
    """Removing any one rule breaks the protocol somewhere: the S issuer waiting for the tile's P.V job
    n - 2 (else the two-slot S-done / P-written / P.V-done waits can fall two phases behind); the S
    issuer waiting for its buffer's previous P.V (else S overwrites P before it is read); the S
    issuer's commit freeing a Q slot after the unit's last S job (else the producer reloads Q^ that S
    jobs still read); and the softmax warps' arrival after reading a slot's unit (else the producer
    publishes the unit two ahead before they have read it)."""
    failures = 0
    for D, T, window, causal in ((64, 300, -1, False), (64, 700, 100, True), (128, 513, 0, True),
                                 (64, 129, 5, True), (64, 600, 0, False)):
        S, NB, QS = CONFIGS[D]
        n_qb = (T + 2 * KT - 1) // (2 * KT)
        units = units_for(1, 3, T, window, causal, list(range(3 * ((n_qb + 1) // 2))), S)
        for seed in range(40):
            try:
                run_cta(units, S, NB, QS, seed=seed, **{flag: False})
            except (Deadlock, AssertionError):
                failures += 1
    assert failures > 0
