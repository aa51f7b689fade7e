"""The balanced split's work assignment, replayed on the host for many length
mixes: the tiles of all (sequence, kv head) segments, each charged a fixed
piece set-up cost, laid end to end and cut into equal warp ranges.  The
replay follows the decode kernel's piece walk and record addressing step for
step (its constants are read from the kernel source) and checks what the
kernels rely on: every tile is attended exactly once, a segment cut into
several pieces has its records at the addresses the merge reads, in tile
order, and no two pieces share a record slot."""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = open(os.path.join(ROOT, "paged_kv_cache_227_gb300", "csrc", "decode.cu")).read()
MIN_PER = int(re.search(r"constexpr int kLeanMinBlocks = (\d+);", SRC).group(1))
COST = int(re.search(r"constexpr int kLeanPieceCost = (\d+);", SRC).group(1))


def prefix(lens, cost):
    nb = [-(-int(L) // 16) for L in lens]
    pfx = [0]
    for n in nb:
        pfx.append(pfx[-1] + (n + cost if n else 0))
    return pfx


def per_of(pfx, Hkv, units):
    T = Hkv * pfx[-1]
    return max(-(-T // units), MIN_PER)


def pieces_of_warp(u, pfx, Hkv, units, cost):
    """The pieces warp u attends: (i, h, j0, j1, final, record)."""
    B = len(pfx) - 1
    T = Hkv * pfx[-1]
    per = per_of(pfx, Hkv, units)
    cur, end = per * u, min(per * u + per, T)
    out = []
    if cur >= end:
        return out
    li = max(i for i in range(B) if Hkv * pfx[i] <= cur)
    cnt = pfx[li + 1] - pfx[li]
    lh = (cur - Hkv * pfx[li]) // cnt
    first = True
    while cur < end:
        cnt = pfx[li + 1] - pfx[li]
        seg_start = Hkv * pfx[li] + lh * cnt
        rs, seg_end = seg_start + cost, seg_start + cnt
        if end <= rs:
            break
        frm, pend = max(cur, rs), min(end, seg_end)
        out.append((li, lh, frm - rs, pend - rs, frm == rs and pend == seg_end, 2 * u + (0 if first else 1)))
        first = False
        cur = pend
        if cur == seg_end:
            lh += 1
            if lh == Hkv:
                lh = 0
                li += 1
                while li < B and pfx[li + 1] == pfx[li]:
                    li += 1
    return out


def segment_records(i, h, pfx, Hkv, units, cost):
    """(count, addresses) of a segment's records, as the merge computes them."""
    per = per_of(pfx, Hkv, units)
    cnt = pfx[i + 1] - pfx[i]
    nb = cnt - cost
    s0 = Hkv * pfx[i] + h * cnt
    rs = s0 + cost
    c0 = rs // per
    count = (rs + nb - 1) // per - c0 + 1
    at = [2 * (c0 + k) + (1 if (k == 0 and s0 > c0 * per) else 0) for k in range(count)]
    return count, at


def check(lens, Hkv, units, cost=COST):
    pfx = prefix(lens, cost)
    nb = [-(-int(L) // 16) for L in lens]
    seen = {}
    recs = {}
    for u in range(units):
        for (i, h, j0, j1, final, rec) in pieces_of_warp(u, pfx, Hkv, units, cost):
            assert 0 <= j0 < j1 <= nb[i]
            for j in range(j0, j1):
                assert (i, h, j) not in seen, "a tile attended twice"
                seen[(i, h, j)] = u
            if not final:
                assert rec not in recs, "two pieces share a record slot"
                assert rec < 2 * units
                recs[rec] = (i, h, j0)
    assert len(seen) == sum(nb) * Hkv, "a tile never attended"
    by_seg = {}
    for rec, (i, h, j0) in recs.items():
        by_seg.setdefault((i, h), []).append((j0, rec))
    for (i, h), lst in by_seg.items():
        count, at = segment_records(i, h, pfx, Hkv, units, cost)
        assert count >= 2
        assert [rec for _, rec in sorted(lst)] == at, (i, h)


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("Hkv,units", [(8, 1216), (2, 1216), (40, 1216), (8, 304), (1, 7), (3, 1)])
def test_random_length_mixes(seed, Hkv, units):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 80))
    kind = seed % 4
    if kind == 0:
        lens = rng.integers(0, 5000, B)
    elif kind == 1:
        lens = np.clip(np.round(np.exp(np.log(600) + 0.8 * rng.standard_normal(B))), 16, 8192)
    elif kind == 2:
        lens = rng.choice([0, 1, 15, 16, 17, 31, 32, 33], B)
    else:
        lens = rng.integers(20000, 40000, max(1, B // 16))
    if lens.sum() == 0:
        lens[0] = 1
    check(lens.astype(int).tolist(), Hkv, units)


def test_bench_workloads():
    from workloads import CONFIGS, context_lengths
    for key in (2, 3, 5):
        cfg = CONFIGS[key]
        lens = (context_lengths(cfg) + 1).tolist()
        check(lens, cfg.n_kv_heads, 152 * 4 * 2)


def test_ranges_no_larger_than_needed_and_the_minimum():
    pfx = prefix([16] * 3, COST)          # 3 segments of 1 tile + cost
    assert per_of(pfx, 1, 1216) == MIN_PER
    pfx = prefix([16 * 1000], COST)
    assert per_of(pfx, 1, 10) == -(-(1000 + COST) // 10)
