"""Host-side model of one CTA of the persistent attention backward kernel, all roles at once (no GPU).

attn_bwd_ws.cuh runs a producer thread (tickets, TMA loads of the K/V slot and the Q ring), one MMA
issuing thread, two softmax warpgroups (the A and B 64-query halves of every iteration) and a dQ
warpgroup (drains dQ^ and writes out a tile's dV, dK^), which hand work to each other through
mbarriers waited by phase parity. This model restates each role's waits, arrivals, loads, MMA issues
and commits in the kernel's order and with its phase arithmetic, as Python generators run under random
interleavings together with an in-order tensor pipe (commits arrive once everything issued before them
has completed) and a TMA engine that completes loads in any order.

Checked on every run:
- exactness: a parity wait only ever sees its barrier at the phase it means or one later;
- data: every TMEM half-buffer, dS^T slot, Q ring stage, K/V slot and the dV / dK^ accumulators hold
  what their reader expects, and nothing is overwritten before its last reader is done;
- progress: every CTA finishes its tiles.
Removing any one of six rules must break it (test_model_catches_removed_rules): the two-slot
dQ-done barrier, the two-slot P-full barrier, the accumulator-free wait, the dQ warps' release of a
B half-buffer only after they have read its dQ^, the Q stage's release after the B half's products,
and the K/V slot's release at a tile's last dQ^ product.
"""
import random

import pytest

from test_pipeline_model import Bar, Deadlock


class CTA:
    def __init__(self, tiles, S, rng, rules):
        self.tiles, self.S, self.rng, self.rules = tiles, S, rng, rules
        b = {}

        def mk(name, count, n=1):
            b[name] = [Bar(f"{name}[{i}]", count) for i in range(n)]

        mk("TileFull", 1, 2); mk("TileEmpty", 1 + 8 + 1, 2); mk("KVFull", 1, 2); mk("KVFree", 1, 2)
        mk("QFull", 1, S); mk("QEmpty", 1, S); mk("Sdp", 1, 3); mk("BufFree", 1, 3)
        mk("PFull", 4, 4); mk("Dq", 1, 2); mk("Final", 1, 2); mk("AccFree", 1, 1)
        self.b = b
        self.tile_id = [None, None]
        self.kv = [None, None]          # K/V slot -> tile index loaded
        self.kv_left = [0, 0]           # reads of the slot's tile still to come
        self.q = [None] * S             # Q ring stage -> iteration loaded
        self.q_left = [0] * S
        self.buf = {}                   # (half-buffer, warp) -> (state, half or iteration)
        self.dsl = {}                   # (dS^T slot, warp) -> (state, half)
        self.acc = None                 # (tile index, products accumulated)
        self.acc_read = -1              # last tile whose accumulators the dQ warps have read
        self.pipe, self.tma = [], []
        self.iter_tile = {}             # iteration N -> (tile index, kv slot)
        self.dq_done = []               # iterations whose dQ^ the dQ warps have read

    @staticmethod
    def wait(bar, k):
        """Parity wait for phase k of `bar` (k = -1: the phase before the first, already done)."""
        return ("wait", bar, k)


def n_iter(c, tl):
    return c.tiles[tl]


def producer(c):
    S = c.S
    N = 0
    for tl in range(len(c.tiles) + 1):
        slot = tl & 1
        if tl >= 2:
            yield c.wait(c.b["TileEmpty"][slot], (tl >> 1) - 1)
        t = tl if tl < len(c.tiles) else -1
        c.tile_id[slot] = t
        c.b["TileFull"][slot].arrive()
        if t < 0:
            return
        if tl >= 2:
            yield c.wait(c.b["KVFree"][slot], (tl >> 1) - 1)
        assert c.kv_left[slot] == 0, f"K/V slot {slot} reloaded with {c.kv_left[slot]} reads of tile {c.kv[slot]} left"
        c.b["KVFull"][slot].arrive(tx=2)
        c.tma += [("K", slot, tl, c.b["KVFull"][slot]), ("V", slot, tl, c.b["KVFull"][slot])]
        for n in range(n_iter(c, tl)):
            s = N % S
            if N >= S:
                yield c.wait(c.b["QEmpty"][s], N // S - 1)
            assert c.q_left[s] == 0, f"Q stage {s} reloaded with {c.q_left[s]} reads of iteration {c.q[s]} left"
            c.b["QFull"][s].arrive(tx=1)
            c.tma.append(("Q", s, N, c.b["QFull"][s]))
            N += 1
            yield ("work",)


def issuer(c):
    S, r = c.S, c.rules
    N = 0
    prev = None  # (kv slot, closes, tile index) of iteration N - 1

    def finish(m, kvs, closes, tl):
        s = m % S
        yield c.wait(c.b["PFull"][2 + ((m & 1) if r["two_slot_pfull"] else 0)],
                     (m >> 1) if r["two_slot_pfull"] else m)
        c.pipe.append(("dvdk", 2 * m + 1, s))
        c.pipe.append(("dQ", m, kvs))
        if r["q_release_late"]:
            c.pipe.append(("commit", c.b["QEmpty"][s]))
        c.pipe.append(("commit", c.b["Dq"][(m & 1) if r["two_slot_dq"] else 0]))
        if closes:
            if r["kv_release_late"]:
                c.pipe.append(("commit", c.b["KVFree"][kvs]))
            c.pipe.append(("commit", c.b["Final"][tl & 1]))

    for tl in range(len(c.tiles) + 1):
        slot = tl & 1
        yield c.wait(c.b["TileFull"][slot], tl >> 1)
        t = c.tile_id[slot]
        c.b["TileEmpty"][slot].arrive()
        if t < 0:
            break
        kvs = tl & 1
        yield c.wait(c.b["KVFull"][kvs], tl >> 1)
        for n in range(n_iter(c, tl)):
            s = N % S
            c.iter_tile[N] = (tl, kvs)
            yield c.wait(c.b["QFull"][s], N // S)
            for half in range(2):
                h = 2 * N + half
                buf = h % 3
                if h >= 3:
                    yield c.wait(c.b["BufFree"][buf], h // 3 - 1)
                c.pipe.append(("sdp", h, s, kvs))
                c.pipe.append(("commit", c.b["Sdp"][buf]))
            if N >= 1:
                if not r["q_release_late"]:  # the rule removed: Q stage freed before the B half's products
                    c.pipe.append(("commit", c.b["QEmpty"][(N - 1) % S]))
                if not r["kv_release_late"] and prev[1]:
                    c.pipe.append(("commit", c.b["KVFree"][prev[0]]))
                yield from finish(N - 1, *prev)
            if n == 0 and tl >= 1 and r["acc_free"]:
                yield c.wait(c.b["AccFree"][0], tl - 1)
            yield c.wait(c.b["PFull"][(N & 1) if r["two_slot_pfull"] else 0],
                         (N >> 1) if r["two_slot_pfull"] else N)
            c.pipe.append(("dvdk", 2 * N, s, n == 0))
            c.pipe.append(("commit", c.b["BufFree"][(2 * N) % 3]))
            prev = (kvs, n == n_iter(c, tl) - 1, tl)
            N += 1
            yield ("work",)
    if N >= 1:
        if not r["q_release_late"]:
            c.pipe.append(("commit", c.b["QEmpty"][(N - 1) % S]))
        if not r["kv_release_late"] and prev[1]:
            c.pipe.append(("commit", c.b["KVFree"][prev[0]]))
        yield from finish(N - 1, *prev)


def softmax(c, half, w):
    S, r = c.S, c.rules
    N = 0
    for tl in range(len(c.tiles) + 1):
        slot = tl & 1
        yield c.wait(c.b["TileFull"][slot], tl >> 1)
        t = c.tile_id[slot]
        c.b["TileEmpty"][slot].arrive()
        if t < 0:
            return
        for n in range(n_iter(c, tl)):
            s, h = N % S, 2 * N + half
            buf = h % 3
            yield c.wait(c.b["QFull"][s], N // S)
            yield c.wait(c.b["Sdp"][buf], h // 3)
            assert c.q[s] == N, f"softmax of half {h} reads lse / delta of iteration {c.q[s]}"
            c.q_left[s] -= 1
            assert c.buf.get((buf, w)) == ("SdP", h), f"softmax {h} warp {w} reads {c.buf.get((buf, w))}"
            yield ("work",)
            assert c.buf.get((buf, w)) == ("SdP", h), f"S^T, dP^T of half {h} overwritten while its softmax ran"
            c.buf[(buf, w)] = ("PdS", h)
            prev = c.dsl.get((h & 3, w))
            assert prev is None or prev in (("read", h - 4), ("free", None)), \
                f"softmax {h} overwrites dS^T slot {h & 3} holding {prev}"
            c.dsl[(h & 3, w)] = ("dS", h)
            c.b["PFull"][2 * half + ((N & 1) if r["two_slot_pfull"] else 0)].arrive()
            N += 1


def dq_warps(c):
    """The dQ warpgroup as its leader (one thread waits and hands the outcome to the others)."""
    r = c.rules
    N = 0
    for tl in range(len(c.tiles) + 1):
        slot = tl & 1
        yield c.wait(c.b["TileFull"][slot], tl >> 1)
        t = c.tile_id[slot]
        c.b["TileEmpty"][slot].arrive()
        if t < 0:
            return
        for n in range(n_iter(c, tl)):
            yield c.wait(c.b["Dq"][(N & 1) if r["two_slot_dq"] else 0], (N >> 1) if r["two_slot_dq"] else N)
            buf = (2 * N + 1) % 3
            for w in range(4):
                assert c.buf.get((buf, w)) == ("dQ", N), f"dQ warps read {c.buf.get((buf, w))} for dQ^ of {N}"
            if not r["b_release"]:  # the rule removed: the half-buffer released before it has been read
                c.b["BufFree"][buf].arrive()
            yield ("work",)  # the TMEM loads of every lane's dQ^ columns
            for w in range(4):
                assert c.buf.get((buf, w)) == ("dQ", N), f"dQ^ of {N} overwritten while the dQ warps read it"
                c.buf[(buf, w)] = ("freed", 2 * N + 1)
            if r["b_release"]:
                c.b["BufFree"][buf].arrive()
            c.dq_done.append(N)
            N += 1
        # write-out of the tile's dV, dK^ (dV staged in the dS^T slot pair of the tile's last iteration)
        yield c.wait(c.b["Final"][tl & 1], tl >> 1)
        assert c.acc == (tl, 2 * n_iter(c, tl)), f"tile {tl} written out with accumulators {c.acc}"
        m = N - 1
        for hh in (2 * m, 2 * m + 1):
            for w in range(4):
                assert c.dsl.get((hh & 3, w)) == ("read", hh), \
                    f"dV staged over dS^T slot {hh & 3} holding {c.dsl.get((hh & 3, w))}"
                c.dsl[(hh & 3, w)] = ("dV", tl)
        yield ("work",)  # TMA stores of dV read the slots; dK^ leaves through the staging buffer
        for hh in (2 * m, 2 * m + 1):
            for w in range(4):
                c.dsl[(hh & 3, w)] = ("free", None)
        c.acc_read = tl
        c.b["AccFree"][0].arrive()


def tensor_pipe(c):
    """Executes the issuing thread's MMAs and commits in order, one per scheduling step."""
    while True:
        if not c.pipe:
            yield ("idle",)
            continue
        op = c.pipe.pop(0)
        kind = op[0]
        if kind == "commit":
            op[1].arrive()
        elif kind == "sdp":
            _, h, s, kvs = op
            N, buf = h // 2, h % 3
            tl = c.iter_tile[N][0]
            for w in range(4):
                prev = c.buf.get((buf, w))
                assert prev is None or prev == ("freed", h - 3), f"S^T/dP^T of half {h} overwrites buffer {buf}: {prev}"
                c.buf[(buf, w)] = ("SdP", h)
            assert c.q[s] == N, f"S^T/dP^T of half {h} reads Q stage {s} holding iteration {c.q[s]}"
            assert c.kv[kvs] == tl, f"S^T/dP^T of half {h} reads K/V slot {kvs} holding tile {c.kv[kvs]}"
            c.q_left[s] -= 1
            c.kv_left[kvs] -= 1
        elif kind == "dvdk":
            h, s = op[1], op[2]
            N, buf = h // 2, h % 3
            tl = c.iter_tile[N][0]
            for w in range(4):
                assert c.buf.get((buf, w)) == ("PdS", h), f"dV/dK^ of half {h} read buffer {buf}: {c.buf.get((buf, w))}"
            assert c.q[s] == N, f"dV/dK^ of half {h} reads Q stage {s} holding iteration {c.q[s]}"
            c.q_left[s] -= 1
            if h % 2 == 0 and op[3]:  # the tile's first product restarts the accumulators
                assert c.acc is None or c.acc_read == c.acc[0], \
                    f"tile {tl} restarts the accumulators before tile {c.acc[0]}'s were read"
                c.acc = (tl, 1)
            else:
                assert c.acc is not None and c.acc[0] == tl, f"dV/dK^ of tile {tl} accumulates onto {c.acc}"
                c.acc = (tl, c.acc[1] + 1)
            if h % 2 == 0:
                for w in range(4):
                    c.buf[(buf, w)] = ("freed", h)
            else:
                for w in range(4):
                    c.buf[(buf, w)] = ("dvdkB", h)
        elif kind == "dQ":
            _, m, kvs = op
            buf = (2 * m + 1) % 3
            tl = c.iter_tile[m][0]
            for w in range(4):
                assert c.buf.get((buf, w)) == ("dvdkB", 2 * m + 1), f"dQ^ of {m} writes buffer {buf}: {c.buf.get((buf, w))}"
                c.buf[(buf, w)] = ("dQ", m)
                for hh in (2 * m, 2 * m + 1):
                    assert c.dsl.get((hh & 3, w)) == ("dS", hh), \
                        f"dQ^ of {m} reads dS^T slot {hh & 3}: {c.dsl.get((hh & 3, w))}"
                    c.dsl[(hh & 3, w)] = ("read", hh)
            assert c.kv[kvs] == tl, f"dQ^ of {m} reads K slot {kvs} holding tile {c.kv[kvs]}"
            c.kv_left[kvs] -= 1
        yield ("work",)


def tma_engine(c):
    """Completes loads in a random order."""
    while True:
        if not c.tma:
            yield ("idle",)
            continue
        kind, dst, what, bar = c.tma.pop(c.rng.randrange(len(c.tma)))
        if kind == "Q":
            c.q[dst] = what
            c.q_left[dst] = 2 + 8 + 2  # S^T/dP^T of both halves, eight softmax warps, dV/dK^ of both halves
        elif kind == "K":
            c.kv[dst] = what
            c.kv_left[dst] = 3 * n_iter(c, what)  # two S^T/dP^T products and one dQ^ product per iteration
        bar.complete_tx(1)
        yield ("work",)


RULES = dict(two_slot_dq=True, two_slot_pfull=True, acc_free=True, b_release=True, q_release_late=True,
             kv_release_late=True)


def run_cta(tiles, S, seed, max_steps=400_000, **flags):
    rng = random.Random(seed)
    c = CTA(tiles, S, rng, dict(RULES, **flags))
    procs = {"producer": producer(c), "issuer": issuer(c), "dq": dq_warps(c)}
    for half in range(2):
        for w in range(4):
            procs[f"softmax{half}.{w}"] = softmax(c, half, w)
    engines = {"tensor": tensor_pipe(c), "tma": tma_engine(c)}
    # how much more often each process is picked: slow dQ warps and fast softmax warps open the
    # windows in which a barrier runs ahead of its waiter
    bias = {k: rng.choice([1, 1, 2, 8]) for k in list(procs) + list(engines)}
    pending = {k: None for k in procs}
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
            assert kph <= done <= kph + 1, f"{k}: waits phase {kph} of {bar.name}, which completed {done}"
            if done == kph + 1:
                runnable.append(k)
        busy = [e for e in engines if (e == "tensor" and c.pipe) or (e == "tma" and c.tma)]
        choices = runnable + busy
        if not choices:
            raise Deadlock(f"blocked: {[(k, a[1].name, a[2]) for k, a in pending.items()]}")
        who = rng.choices(choices, weights=[bias[k] for k in choices])[0]
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
    assert c.dq_done == list(range(sum(tiles))), "not every iteration's dQ^ was drained"
    assert c.acc_read == len(tiles) - 1, "not every tile was written out"
    return c


def tile_lists(seed, n):
    rng = random.Random(seed)
    out = [[1], [2], [3], [1, 1], [1, 2, 1], [5, 1], [1, 1, 1, 1], [2, 3, 1, 4]]
    for _ in range(n):
        out.append([rng.choice([1, 1, 2, 3, 4, 6]) for _ in range(rng.randint(1, 5))])
    return out


@pytest.mark.parametrize("S", [2, 3])  # the Q ring at D = 64 and D = 32
def test_protocol_has_no_deadlock_exact_waits_and_no_hazard(S):
    for i, tiles in enumerate(tile_lists(S, 40)):
        for seed in range(6):
            run_cta(tiles, S, seed=1000 * i + seed + 17 * S)


@pytest.mark.parametrize("flag", sorted(RULES))
def test_model_catches_removed_rules(flag):
    """Each rule is needed: without it some interleaving falls two phases behind a barrier, reads or
    overwrites a buffer at the wrong time, or deadlocks."""
    caught = False
    for i, tiles in enumerate(tile_lists(99, 60)):
        for seed in range(8):
            try:
                run_cta(tiles, 2, seed=7919 * i + seed, **{flag: False})
            except (AssertionError, Deadlock):
                caught = True
                break
        if caught:
            break
    assert caught, f"removing {flag} went unnoticed"
