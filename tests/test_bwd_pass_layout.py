"""Host-side model of the backward's staged prologue and finalize passes (runs without a GPU).

Both passes hand out groups of rows to warps in strides of the grid's warp count; each warp stages a
group's rows in shared memory with cp.async and then computes from there. This model restates the
passes' index arithmetic (attn_bwd.cuh: PrepCfg, prep_pos, prep_issue and the prologue's compute loop;
FinCfg, fin_gpos, fin_xpos, fin_issue and the finalize's compute loop; attn_bwd.cu's grid sizes) and
checks, over ragged shapes, grouped K/V heads and D = 32, 64, 128, that
- every global read stays inside its tensor and every staged chunk inside its warp's stage,
- each stage chunk is written once per fill, and every lane reads only chunks its group staged,
- every q^, k^, delta / -lse row, every cleared dq^ element and every dq, dk row is written once,
- the strided assignment visits every group exactly once,
- each shared-memory read instruction takes the minimum number of wavefronts (no bank conflicts
  beyond the bytes it moves).
"""
import itertools
import math

import pytest

SMEM_PER_CTA = 232448  # bytes of dynamic shared memory one CTA may use


def prep_cfg(D):
    arr = 16 * 2 * D  # 16 bf16 rows
    stage = 3 * arr + 16 * 4
    return dict(warps=8, stages=2, q_rows=16, k_rows=48, arr=arr, stage=stage, smem=8 * 2 * stage)


def fin_cfg(D):
    rows = 512 // D
    g, x = rows * 4 * D, rows * 2 * D
    return dict(warps=8, stages=2, rows=rows, g=g, x=x, stage=g + x, smem=8 * 2 * (g + x))


def prep_pos(D, r, c):
    sw = ((r >> 1) & 3) if D == 32 else (r & 7)
    assert 0 <= (c ^ sw) < D // 8
    return r * 2 * D + 16 * (c ^ sw)


def fin_swap(D, r):
    return ((r >> 1) & 1) if D == 32 else (r & 1)


def fin_gpos(D, r, u):
    return r * 4 * D + 16 * (u ^ ((r & 1) * (D // 8)))


def fin_xpos(D, r, j):
    return r * 2 * D + 8 * (j ^ (fin_swap(D, r) * (D // 8)))


def strided_cover(groups, warps_total):
    seen = [0] * groups
    for gw in range(warps_total):
        g = gw
        while g < groups:
            seen[g] += 1
            g += warps_total
    return all(s == 1 for s in seen)


def model_prep(B, T, H, Hkv, D, ctas):
    C = prep_cfg(D)
    NC = D // 8
    assert C["smem"] <= SMEM_PER_CTA and C["stage"] % 16 == 0
    nq, nk = B * T * H, B * T * Hkv
    nqg, nkg = -(-nq // 16), -(-nk // 48)
    groups = nqg + nkg
    grid = min(-(-groups // C["warps"]), ctas)
    assert strided_cover(groups, grid * C["warps"])
    qh, kh, dlt = [0] * nq, [0] * nk, [0] * nq
    dq0 = [0] * (nq * D // 4)
    for grp in range(groups):
        staged = set()
        if grp < nqg:
            row0 = grp * 16
            for i in range(16 * NC):
                r, c = divmod(i, NC)
                row = row0 + r
                off = (row if row < nq else 0) * D + 8 * c
                assert off + 8 <= nq * D
                for a in range(3):  # q, out, dout
                    pos = a * C["arr"] + prep_pos(D, r, c)
                    assert pos % 16 == 0 and pos + 16 <= 3 * C["arr"] and pos not in staged
                    staged.add(pos)
            for lane in range(16):
                row = row0 + lane
                if row < nq:
                    bt = row // H
                    h, t, b = row - bt * H, bt % T, bt // T
                    assert 0 <= (b * H + h) * T + t < B * H * T
                    assert 3 * C["arr"] + 4 * lane + 4 <= C["stage"]
            for lane in range(32):
                e, rl = lane & 1, lane >> 1
                row = row0 + rl
                for c in range(NC):
                    for a in range(3):
                        p = a * C["arr"] + prep_pos(D, rl, c) + 8 * e
                        assert p - p % 16 in staged
                assert 0 <= (row // H) % T < T
                if row < nq and e == 0:
                    qh[row] += 1
                    dlt[row] += 1
            for i in range(16 * D // 4):
                if row0 + i // (D // 4) < nq:
                    dq0[row0 * D // 4 + i] += 1
        else:
            row0 = (grp - nqg) * 48
            for i in range(48 * NC):
                r, c = divmod(i, NC)
                row = row0 + r
                assert (row if row < nk else 0) * D + 8 * c + 8 <= nk * D
                pos = prep_pos(D, r, c)
                assert pos + 16 <= 3 * C["arr"] and pos not in staged
                staged.add(pos)
            for s in range(3):
                for lane in range(32):
                    e, rl = lane & 1, lane >> 1
                    rr = 16 * s + rl
                    row = row0 + rr
                    for c in range(NC):
                        p = prep_pos(D, rr, c) + 8 * e
                        assert p - p % 16 in staged
                    assert 0 <= (row // Hkv) % T < T
                    if row < nk and e == 0:
                        kh[row] += 1
    assert all(x == 1 for x in qh) and all(x == 1 for x in kh) and all(x == 1 for x in dlt)
    assert all(x == 1 for x in dq0)


def model_fin(B, T, H, Hkv, D, ctas):
    C = fin_cfg(D)
    NC, NU, RPW, R = D // 8, D // 4, 32 // (D // 8), fin_cfg(D)["rows"]
    assert C["smem"] <= SMEM_PER_CTA
    nq, nk = B * T * H, B * T * Hkv
    nqg, nkg = -(-nq // R), -(-nk // R)
    grid = min(-(-(nqg + nkg) // C["warps"]), ctas)
    assert strided_cover(nqg + nkg, grid * C["warps"])
    out_q, out_k = [0] * nq, [0] * nk
    for grp in range(nqg + nkg):
        isq = grp < nqg
        row0, n = (grp if isq else grp - nqg) * R, (nq if isq else nk)
        gs, xs = set(), set()
        for i in range(R * NU):
            r, u = divmod(i, NU)
            row = row0 + r
            assert (row if row < n else 0) * D + 4 * u + 4 <= n * D
            pos = fin_gpos(D, r, u)
            assert pos % 16 == 0 and pos + 16 <= C["g"] and pos not in gs
            gs.add(pos)
        for i in range(R * NC):
            r, k = divmod(i, NC)
            row = row0 + r
            assert (row if row < n else 0) * D + 8 * k + 8 <= n * D
            pos = fin_xpos(D, r, 2 * k)
            assert fin_xpos(D, r, 2 * k + 1) == pos + 8  # a 16-byte chunk keeps its two halves adjacent
            assert pos % 16 == 0 and pos + 16 <= C["x"] and pos not in xs
            xs.add(pos)
        for s in range(R // RPW):
            for lane in range(32):
                c, sub = lane % NC, lane // NC
                rr = s * RPW + sub
                row = row0 + rr
                assert fin_gpos(D, rr, c) in gs and fin_gpos(D, rr, c + NC) in gs
                for j in (c, c + NC):
                    p = fin_xpos(D, rr, j)
                    assert p - p % 16 in xs
                assert 2 * c + 1 < D // 4  # the two table entries of the lane's pairs
                for off in (1 << b for b in range(int(math.log2(NC)))):
                    assert (lane ^ off) // NC == sub  # row sums stay within the row's lanes
                if row < n and c == 0:
                    (out_q if isq else out_k)[row] += 1
    assert all(x == 1 for x in out_q) and all(x == 1 for x in out_k)


def wavefronts(addrs, width):
    """Shared-memory wavefronts of one warp-wide access: the largest number of distinct 4-byte words
    that fall into one bank."""
    banks = {}
    for a in addrs:
        for w in range(width // 4):
            word = a // 4 + w
            banks.setdefault(word % 32, set()).add(word)
    return max(len(v) for v in banks.values())


SHAPES = [(1, 1, 1, 1), (1, 7, 3, 1), (2, 9, 3, 3), (1, 130, 4, 2), (3, 17, 6, 2), (2, 300, 5, 5), (1, 64, 16, 4),
          (1, 37, 3, 1), (3, 45, 3, 3)]


@pytest.mark.parametrize("D", [32, 64, 128])
def test_prologue_pass_layout(D):
    for (B, T, H, Hkv), ctas in itertools.product(SHAPES, (2, 5)):
        model_prep(B, T, H, Hkv, D, ctas)


@pytest.mark.parametrize("D", [32, 64, 128])
def test_finalize_pass_layout(D):
    for (B, T, H, Hkv), ctas in itertools.product(SHAPES, (2, 7)):
        model_fin(B, T, H, Hkv, D, ctas)


@pytest.mark.parametrize("D", [32, 64, 128])
def test_staged_reads_take_minimum_wavefronts(D):
    NC, RPW = D // 8, 32 // (D // 8)
    # prologue: 16 rows x 2 lanes x 8 bytes = 256 bytes -> 2 wavefronts
    for c, base in itertools.product(range(NC), (0, 16, 32)):
        addrs = [prep_pos(D, base + (lane >> 1), c) + 8 * (lane & 1) for lane in range(32)]
        assert wavefronts(addrs, 8) == 2
    # finalize: fp32 halves 512 bytes -> 4 wavefronts; bf16 halves 256 bytes -> 2
    for s, half in itertools.product(range(16 // RPW), (0, 1)):
        rows = [s * RPW + lane // NC for lane in range(32)]
        cols = [lane % NC + half * NC for lane in range(32)]
        assert wavefronts([fin_gpos(D, r, u) for r, u in zip(rows, cols)], 16) == 4
        assert wavefronts([fin_xpos(D, r, j) for r, j in zip(rows, cols)], 8) == 2


def test_pass_shared_memory_fits():
    for D in (32, 64, 128):
        assert prep_cfg(D)["smem"] <= SMEM_PER_CTA and fin_cfg(D)["smem"] <= SMEM_PER_CTA
        assert fin_cfg(D)["stage"] == 3072  # 3 KB stages: four CTAs (32 warps) per SM
