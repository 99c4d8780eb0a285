"""Host-side model of the persistent kernel's K/V ring bookkeeping (runs without a GPU).

The kernel hands out tickets of consecutive query blocks of one head: all the blocks of heads
0 .. n_long - 1 (one ticket each), then pairs (qb, qb - 1) of the other heads, heaviest first. It
streams each unit's key tiles downwards and keeps the last R tiles of a unit resident for the next
unit of its ticket (R = ke_all(next) - kb_all(unit) + 1 when 1 <= R <= ring depth). Every role derives the
ring position of a key step with the same arithmetic: the producer and the prologue take fresh
positions in order for the non-resident steps; the MMA issuers and the softmax use position
`kc - r_in + i` for resident step i and the next fresh position otherwise; a stage is released
at the last use of its load. This model restates that arithmetic (attn_fwd_ws.cuh: unit_geom,
shared_steps, the producer's ticket loop, the S and P.V issuers' step loops) and checks, over
shapes, windows, mask modes and random assignments of tickets to CTAs, that
- every consumer's position holds the key tile of its step (same head),
- every load is released exactly once, at its last use,
- no consumer needs a stage whose previous load has not been released yet (no deadlock).
"""
import itertools
import random

import pytest

KT, S = 128, 4  # key tile rows, ring depth


def unit_geom(T, window, causal, bh, qb):
    g = dict(bh=bh, qs0=qb * 2 * KT, r_in=0, r_out=0)
    kb, ke = [0, 0], [0, 0]
    for t in range(2):
        qs = g["qs0"] + KT * t
        if qs < T:
            qe = min(T - 1, qs + KT - 1)
            lo = max(0, qs - window) if window >= 0 else 0
            hi = qe if causal else (min(T - 1, qe + window) if window >= 0 else T - 1)
            kb[t], ke[t] = lo // KT, hi // KT
        else:
            kb[t], ke[t] = 1, 0
    two = kb[1] <= ke[1]
    g["kb_all"] = min(kb) if two else kb[0]
    g["ke_all"] = max(ke) if two else ke[0]
    g["n"] = g["ke_all"] - g["kb_all"] + 1
    return g


def shared_steps(a, nb):
    if a["bh"] != nb["bh"] or nb["qs0"] + 2 * KT != a["qs0"]:
        return 0
    R = nb["ke_all"] - a["kb_all"] + 1
    return R if (1 <= R <= S and R <= a["n"] and R <= nb["n"]) else 0


def ticket_decode(c, n_bh, n_qb, head_group, n_long=0):
    """Ticket c -> (head, highest query block, units): heads below n_long whole, then pairs of the other
    heads in groups of head_group heads, inside a group the heaviest pair of every head first (the
    producer's decode in attn_fwd_ws.cuh)."""
    if c < n_long:
        return c, n_qb - 1, n_qb
    cpb = (n_qb + 1) // 2
    grp, rem = divmod(c - n_long, head_group * cpb)
    gsize = min(head_group, n_bh - n_long - grp * head_group)
    rank, i = divmod(rem, gsize)
    qb = n_qb - 1 - 2 * rank
    return n_long + grp * head_group + i, qb, (2 if qb >= 1 else 1)


def n_long_heads(B, H, T, window, causal, sm_count=148):
    """Heads that run as one ticket each (attn_api.cu, launch_ws): all but about two waves of pair
    tickets, where consecutive blocks can share key tiles (causal, window within the ring's depth)."""
    n_qb = (T + 2 * KT - 1) // (2 * KT)
    cpb = (n_qb + 1) // 2
    tail = 2 * ((sm_count + cpb - 1) // cpb)
    chains = causal and 0 <= window <= S * KT and n_qb > 1
    return B * H - tail if chains and B * H > tail else 0


def n_tickets(B, H, T, n_long):
    n_qb = (T + 2 * KT - 1) // (2 * KT)
    return n_long + (B * H - n_long) * ((n_qb + 1) // 2)


def cta_units(B, H, T, window, causal, tickets, head_group=1 << 20, n_long=0):
    """The units one CTA runs for the given tickets, with r_in / r_out as the producer sets them."""
    n_qb = (T + 2 * KT - 1) // (2 * KT)
    n_bh = B * H
    units = []
    for c in tickets:
        bh, qb, left = ticket_decode(c, n_bh, n_qb, head_group, n_long)
        first, r_prev = True, 0
        while left:
            g = unit_geom(T, window, causal, bh, qb)
            g["r_in"] = 0 if first else r_prev
            first = False
            if left >= 2:
                g["r_out"] = shared_steps(g, unit_geom(T, window, causal, bh, qb - 1))
            r_prev = g["r_out"]
            units.append(g)
            left, qb = left - 1, qb - 1
    return units


def check_ring(units):
    loads = [(g["bh"], g["ke_all"] - i) for g in units for i in range(g["r_in"], g["n"])]
    kc, uses, order = 0, {}, []
    for g in units:
        for i in range(g["n"]):
            if i < g["r_in"]:
                pos = kc - g["r_in"] + i
            else:
                pos, kc = kc, kc + 1
            assert 0 <= pos < len(loads) and loads[pos] == (g["bh"], g["ke_all"] - i)
            release = i < g["n"] - g["r_out"]
            uses.setdefault(pos, []).append(release)
            order.append((pos, release))
    assert kc == len(loads)
    for rel in uses.values():
        assert sum(rel) == 1 and rel[-1]
    released = set()
    for pos, rel in order:
        assert pos < S or pos - S in released
        if rel:
            released.add(pos)
    return sum(g["n"] - g["r_in"] for g in units), sum(g["n"] for g in units)


@pytest.mark.parametrize("B,H,T", [(2, 3, 1024), (1, 2, 513), (1, 1, 2048), (2, 2, 300), (1, 1, 129),
                                   (1, 3, 256), (1, 1, 4096)])
def test_ring_positions_releases_and_order(B, H, T):
    n_qb = (T + 2 * KT - 1) // (2 * KT)
    n_tickets = B * H * ((n_qb + 1) // 2)
    for window, causal in itertools.product([-1, 0, 1, 100, 127, 128, 200, 255, 256, 383, 384, 511, 512, 513,
                                             640, 1000, 1024, 3000], [True, False]):
        rnd = random.Random(T * 7 + window)
        parts = [list(range(n_tickets))]
        for _ in range(3):
            per = {}
            for c in range(n_tickets):
                per.setdefault(rnd.randrange(3), []).append(c)
            parts += list(per.values())
        for tickets in parts:
            for head_group in (1, 2, 5, 1 << 20):
                check_ring(cta_units(B, H, T, window, causal, tickets, head_group))


@pytest.mark.parametrize("n_bh,n_qb,head_group,n_long", [(384, 4, 256, 0), (512, 8, 64, 0), (192, 4, 512, 0),
                                                         (7, 3, 2, 0), (5, 1, 3, 0), (6, 5, 4, 0), (384, 4, 256, 236),
                                                         (40, 8, 16, 21), (9, 3, 2, 4), (6, 5, 4, 5)])
def test_tickets_cover_every_block_once_heaviest_pairs_first(n_bh, n_qb, head_group, n_long):
    n_t = n_long + (n_bh - n_long) * ((n_qb + 1) // 2)
    seen = [ticket_decode(c, n_bh, n_qb, head_group, n_long) for c in range(n_t)]
    blocks = sorted((bh, qb - i) for bh, qb, units in seen for i in range(units))
    assert blocks == sorted((bh, qb) for bh in range(n_bh) for qb in range(n_qb))
    assert all(units == n_qb and qb == n_qb - 1 for bh, qb, units in seen[:n_long])
    pairs = seen[n_long:]
    for c in range(1, len(pairs)):  # inside a group the pairs come heaviest (highest query block) first
        (b0, q0, _), (b1, q1, _) = pairs[c - 1], pairs[c]
        if (b0 - n_long) // head_group == (b1 - n_long) // head_group:
            assert q1 <= q0


def test_reuse_on_the_120m_shape():
    """With pairs alone, S layers (W = 512) load and transform 2/3 of the K tiles their key steps visit
    and L layers 90 %. With whole-head tickets for all but two waves of pairs (148 SMs: 236 of the 384
    heads), S layers load 8 of a head's 18 visited tiles there and 12 in the pair heads."""
    for W, frac in ((512, 2 / 3), (1024, 0.9)):
        fresh, steps = check_ring(cta_units(32, 12, 1024, W, True, list(range(32 * 12 * 2))))
        assert abs(fresh / steps - frac) < 1e-9
    n_long = n_long_heads(32, 12, 1024, 512, True)
    assert n_long == 236 and n_long_heads(32, 12, 1024, 1024, True) == 0
    tickets = list(range(n_tickets(32, 12, 1024, n_long)))
    fresh, steps = check_ring(cta_units(32, 12, 1024, 512, True, tickets, n_long=n_long))
    assert (fresh, steps) == (236 * 8 + 148 * 12, 384 * 18)


@pytest.mark.parametrize("B,H,T", [(2, 80, 1024), (1, 160, 2048), (1, 200, 513), (4, 40, 1024)])
def test_whole_head_tickets_ring_positions_and_releases(B, H, T):
    """Chunks of all the blocks of a head: every unit shares with the next, a key tile can serve three
    units; positions, single releases at the last use and load order still hold under random
    assignments of tickets to CTAs."""
    for window in (0, 100, 127, 128, 255, 256, 383, 384, 511, 512):
        n_long = n_long_heads(B, H, T, window, True)
        assert n_long > 0
        n_t = n_tickets(B, H, T, n_long)
        rnd = random.Random(T + window + H)
        parts = [list(range(n_t))]
        for _ in range(2):
            per = {}
            for c in range(n_t):
                per.setdefault(rnd.randrange(4), []).append(c)
            parts += list(per.values())
        for tickets in parts:
            for head_group in (1, 3, 1 << 20):
                check_ring(cta_units(B, H, T, window, True, tickets, head_group, n_long))
