"""Host-side model of the persistent kernel's K/V ring bookkeeping (runs without a GPU).

The kernel hands out tickets of two query blocks (qb, qb - 1) of one head, heaviest first, streams
each unit's key tiles downwards and keeps the last R tiles of the first unit resident for the
second (R = ke_all(second) - kb_all(first) + 1 when 1 <= R <= ring depth). Every role derives the
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


def ticket_decode(c, n_bh, n_qb, head_group):
    """Ticket c -> (head, highest query block of its pair): groups of head_group heads in turn, inside a
    group the heaviest pair of every head first (the producer's decode in attn_fwd_ws.cuh)."""
    cpb = (n_qb + 1) // 2
    grp, rem = divmod(c, head_group * cpb)
    gsize = min(head_group, n_bh - grp * head_group)
    rank, i = divmod(rem, gsize)
    return grp * head_group + i, n_qb - 1 - 2 * rank


def cta_units(B, H, T, window, causal, tickets, head_group=1 << 20):
    """The units one CTA runs for the given tickets, with r_in / r_out as the producer sets them."""
    n_qb = (T + 2 * KT - 1) // (2 * KT)
    n_bh = B * H
    units = []
    for c in tickets:
        bh, qb = ticket_decode(c, n_bh, n_qb, head_group)
        left, r_prev = (2 if qb >= 1 else 1), 0
        while left:
            g = unit_geom(T, window, causal, bh, qb)
            g["r_in"] = r_prev if left == 1 else 0
            if left == 2:
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


@pytest.mark.parametrize("n_bh,n_qb,head_group", [(384, 4, 256), (512, 8, 64), (192, 4, 512), (7, 3, 2),
                                                  (5, 1, 3), (6, 5, 4)])
def test_tickets_cover_every_pair_once_heaviest_first_in_a_group(n_bh, n_qb, head_group):
    n_tickets = n_bh * ((n_qb + 1) // 2)
    seen = [ticket_decode(c, n_bh, n_qb, head_group) for c in range(n_tickets)]
    assert sorted(seen) == sorted((bh, n_qb - 1 - 2 * r) for bh in range(n_bh) for r in range((n_qb + 1) // 2))
    for c in range(1, n_tickets):  # inside a group the pairs come heaviest (highest query block) first
        (b0, q0), (b1, q1) = seen[c - 1], seen[c]
        if b0 // head_group == b1 // head_group:
            assert q1 <= q0


def test_reuse_on_the_120m_shape():
    """S layers (W = 512) load and transform 2/3 of the K tiles their key steps visit, L layers 90 %."""
    for W, frac in ((512, 2 / 3), (1024, 0.9)):
        fresh, steps = check_ring(cta_units(32, 12, 1024, W, True, list(range(32 * 12 * 2))))
        assert abs(fresh / steps - frac) < 1e-9
