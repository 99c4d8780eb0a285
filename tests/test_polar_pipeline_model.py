"""Host-side model of one CTA of the persistent Polar Express GEMM kernel (no GPU).

polar.cuh's gemm_kernel runs a producer thread (TMA loads of the K slices of both operands into a
ring of stages), one MMA-issuing thread (a tile's products into one of two TMEM accumulator buffers)
and four epilogue warps (read the accumulator in 64-column chunks, stage each chunk as bf16 in one of
two shared-memory boxes and store it by TMA). This model restates each role's waits, arrivals, loads,
MMA issues, commits and bulk-store waits in the kernel's order and phase arithmetic, as generators run
under random interleavings with an in-order tensor pipe, a TMA engine that completes loads in any
order and bulk stores that read their box some time after they are issued.

Checked: every parity wait is exact (its barrier is at the phase it means or one later), every stage,
accumulator buffer and staging box holds what its reader expects and is not overwritten before its
last reader is done, and every tile's chunks reach the output. Removing any one of four rules breaks it
(test_model_catches_removed_rules): the issuer's wait for the epilogue to free an accumulator buffer,
the epilogue's release only after its last TMEM read of the tile, the stage's release by a commit after
its products, and the epilogue's wait for a box's previous store to have read it.
"""
import random

import pytest

from test_pipeline_model import Bar, Deadlock


class CTA:
    def __init__(self, tiles, S, rng, rules):
        self.tiles, self.S, self.rng, self.rules = tiles, S, rng, rules  # tiles: [(k steps, 64-col chunks)]
        self.b = {"Full": [Bar(f"Full[{i}]", 1) for i in range(S)],
                  "Empty": [Bar(f"Empty[{i}]", 1) for i in range(S)],
                  "AccFull": [Bar(f"AccFull[{i}]", 1) for i in range(2)],
                  "AccEmpty": [Bar(f"AccEmpty[{i}]", 4) for i in range(2)],
                  "Done": [Bar("Done", 1)]}
        self.stage = [None] * S          # stage -> (tile, k step) loaded
        self.stage_readers = [0] * S     # products still to read the stage's load
        self.acc = [None, None]          # accumulator buffer -> (tile, k steps accumulated)
        self.acc_reads = [{}, {}]        # buffer -> warp -> chunks of the current tile read
        self.box = [None, None]          # staging box -> (tile, chunk) staged by all four warps
        self.box_pending = [None, None]  # staging box -> (tile, chunk) whose store has not read it yet
        self.groups = []                 # committed bulk stores, oldest first: box index
        self.stored = set()
        self.pipe, self.tma = [], []

    @staticmethod
    def wait(bar, k):
        return ("wait", bar, k)


def producer(c):
    S = c.S
    g = 0
    for t, (nk, _) in enumerate(c.tiles):
        for kt in range(nk):
            s = g % S
            if g >= S:
                yield c.wait(c.b["Empty"][s], g // S - 1)
            assert c.stage_readers[s] == 0, f"stage {s} reloaded with {c.stage_readers[s]} products left"
            c.b["Full"][s].arrive(tx=1)
            c.tma.append((s, (t, kt), c.b["Full"][s]))
            g += 1
            yield ("work",)


def issuer(c):
    S, r = c.S, c.rules
    g = 0
    for i, (nk, _) in enumerate(c.tiles):
        buf = i & 1
        if i >= 2 and r["acc_empty_wait"]:
            yield c.wait(c.b["AccEmpty"][buf], (i >> 1) - 1)
        for kt in range(nk):
            s = g % S
            yield c.wait(c.b["Full"][s], g // S)
            if not r["empty_after_mma"]:  # the rule removed: the stage released before its products
                c.pipe.append(("commit", c.b["Empty"][s]))
            c.pipe.append(("mma", i, kt, buf, s))
            if r["empty_after_mma"]:
                c.pipe.append(("commit", c.b["Empty"][s]))
            g += 1
            yield ("work",)
        c.pipe.append(("commit", c.b["AccFull"][buf]))
    c.pipe.append(("commit", c.b["Done"][0]))
    yield c.wait(c.b["Done"][0], 0)


def epilogue(c, w):
    """Warp w of the epilogue; warp 0's lane 0 also does the leader's waits (AccFull, bulk reads)."""
    r = c.rules
    cc = 0
    for i, (nk, nvc) in enumerate(c.tiles):
        buf = i & 1
        yield c.wait(c.b["AccFull"][buf], i >> 1)  # the leader's wait, handed to all four warps
        for ch in range(nvc):
            assert c.acc[buf] == (i, nk), f"epilogue of tile {i} reads accumulator {buf}: {c.acc[buf]}"
            yield ("work",)  # the TMEM loads of the chunk
            assert c.acc[buf] == (i, nk), f"accumulator {buf} overwritten while tile {i} was read"
            c.acc_reads[buf][w] = (i, ch)
            last = ch == nvc - 1
            if (last and r["acc_release_late"]) or (ch == 0 and not r["acc_release_late"]):
                c.b["AccEmpty"][buf].arrive()
            sb = cc & 1
            if w == 0 and r["box_read_wait"]:  # at most one store group may still be reading a box
                while len(c.groups) > 1:
                    yield ("idle",)
            yield ("sync", cc, 0)  # the epilogue's named barrier
            assert c.box_pending[sb] is None, f"box {sb} rewritten while the store of {c.box_pending[sb]} reads it"
            c.box[sb] = (i, ch) if w == 0 else c.box[sb]
            yield ("sync", cc, 1)
            if w == 0:
                assert c.box[sb] == (i, ch)
                c.box_pending[sb] = (i, ch)
                c.groups.append(sb)
            cc += 1


def tensor_pipe(c):
    while True:
        if not c.pipe:
            yield ("idle",)
            continue
        op = c.pipe.pop(0)
        if op[0] == "commit":
            op[1].arrive()
        else:
            _, i, kt, buf, s = op
            assert c.stage[s] == (i, kt), f"product ({i}, {kt}) reads stage {s} holding {c.stage[s]}"
            c.stage_readers[s] -= 1
            if kt == 0:
                prev = c.acc[buf]
                if prev is not None:
                    nvc = c.tiles[prev[0]][1]
                    for w in range(4):
                        assert c.acc_reads[buf].get(w) == (prev[0], nvc - 1), \
                            f"tile {i} restarts accumulator {buf} before tile {prev[0]} was read: {c.acc_reads[buf]}"
                c.acc[buf] = (i, 1)
            else:
                assert c.acc[buf] == (i, kt), f"product ({i}, {kt}) accumulates onto {c.acc[buf]}"
                c.acc[buf] = (i, kt + 1)
        yield ("work",)


def tma_engine(c):
    """Completes loads in any order and lets the oldest bulk store read its box."""
    while True:
        if not c.tma and not c.groups:
            yield ("idle",)
            continue
        if c.groups and (not c.tma or c.rng.random() < 0.5):
            sb = c.groups.pop(0)
            c.stored.add(c.box_pending[sb])
            c.box_pending[sb] = None
        else:
            s, what, bar = c.tma.pop(c.rng.randrange(len(c.tma)))
            c.stage[s] = what
            c.stage_readers[s] = 1
            bar.complete_tx(1)
        yield ("work",)


RULES = dict(acc_empty_wait=True, acc_release_late=True, empty_after_mma=True, box_read_wait=True)


def run_cta(tiles, S, seed, max_steps=300_000, **flags):
    rng = random.Random(seed)
    c = CTA(tiles, S, rng, dict(RULES, **flags))
    procs = {"producer": producer(c), "issuer": issuer(c)}
    for w in range(4):
        procs[f"epi{w}"] = epilogue(c, w)
    engines = {"tensor": tensor_pipe(c), "tma": tma_engine(c)}
    bias = {k: rng.choice([1, 1, 2, 8]) for k in list(procs) + list(engines)}
    pending = {k: None for k in procs}
    syncs = {}  # (cc, phase) -> warps arrived at the epilogue's named barrier
    steps = 0
    while procs:
        steps += 1
        assert steps < max_steps, "model did not finish"
        runnable = []
        for k, act in pending.items():
            if act is None or act[0] == "idle":
                runnable.append(k)
            elif act[0] == "sync":
                if len(syncs.get(act[1:], ())) == 4:
                    runnable.append(k)
            else:
                _, bar, kph = act
                done = bar.completed
                assert kph <= done <= kph + 1, f"{k}: waits phase {kph} of {bar.name}, which completed {done}"
                if done == kph + 1:
                    runnable.append(k)
        busy = [e for e in engines if (e == "tensor" and c.pipe) or (e == "tma" and (c.tma or c.groups))]
        choices = runnable + busy
        if not choices:
            raise Deadlock(f"blocked: {pending}")
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
        if act[0] == "sync":
            syncs.setdefault(act[1:], set()).add(who)
        pending[who] = act if act[0] in ("wait", "sync") else None
    want = {(i, ch) for i, (_, nvc) in enumerate(tiles) for ch in range(nvc)}
    assert want <= c.stored | {x for x in c.box_pending if x}, "a chunk never reached its store"
    return c


def tile_lists(seed, n):
    rng = random.Random(seed)
    out = [[(1, 1)], [(2, 2), (1, 4)], [(3, 1)] * 3, [(12, 4)] * 2, [(1, 2)] * 5]
    for _ in range(n):
        out.append([(rng.choice([1, 2, 3, 12]), rng.choice([1, 2, 4])) for _ in range(rng.randint(1, 6))])
    return out


@pytest.mark.parametrize("S", [4, 6])  # ring depth at BN = 256 and BN = 128
def test_protocol_has_no_deadlock_exact_waits_and_no_hazard(S):
    for i, tiles in enumerate(tile_lists(S, 40)):
        for seed in range(5):
            run_cta(tiles, S, seed=100 * i + seed + S)


@pytest.mark.parametrize("flag", sorted(RULES))
def test_model_catches_removed_rules(flag):
    caught = False
    for i, tiles in enumerate(tile_lists(123, 80)):
        for seed in range(8):
            try:
                run_cta(tiles, 4, seed=31 * i + seed, **{flag: False})
            except (AssertionError, Deadlock):
                caught = True
                break
        if caught:
            break
    assert caught, f"removing {flag} went unnoticed"
