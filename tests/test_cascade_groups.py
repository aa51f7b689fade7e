"""Host-side grouping for the shared-prefix (cascade) decode (pa_cascade_groups,
no GPU): sequences whose tables start with the same block, in order of first
appearance, cut into groups of at most 8/G members, each group's prefix the
run of full blocks all its members share.  Checked against the rule written
out plainly here and against the properties the cascade kernels rely on."""
import numpy as np
import pytest

import paged_kv_cache_227_gb300 as pa
from workloads import CONFIGS, build_tables, make_case


def rule(tables, lens, max_members):
    """The documented rule, step by step."""
    order, by_first = [], {}
    for i, L in enumerate(lens):
        if L < 16:
            continue
        b = int(tables[i, 0])
        if b not in by_first:
            order.append(b)
            by_first[b] = []
        by_first[b].append(i)
    out = []
    for b in order:
        seqs = by_first[b]
        for c in range(0, len(seqs), max_members):
            grp = seqs[c:c + max_members]
            if len(grp) < 2:
                continue
            lim = min(min(int(lens[i]) // 16 for i in grp), tables.shape[1])
            P = 0
            while P < lim and all(tables[i, P] == tables[grp[0], P] for i in grp):
                P += 1
            if P >= 1:
                out.append((grp, P))
    return out


def groups_of(tables, lens, Hq, Hkv):
    gs, mem, pre = pa.cascade_groups(tables, lens, Hq, Hkv)
    return [(mem[gs[k]:gs[k + 1]].tolist(), int(pre[k])) for k in range(len(pre))]


def random_history(seed, n_seqs=24, num_blocks=2000):
    """Tables from the library's allocator: fresh sequences and forks of
    earlier ones at random lengths, then more tokens (copy-on-write)."""
    rng = np.random.default_rng(seed)
    alloc = pa.BlockAllocator(num_blocks, 16, rng.permutation(num_blocks).tolist())
    for i in range(n_seqs):
        if i and rng.random() < 0.6:
            alloc.fork(int(rng.integers(0, i)), i)
        else:
            alloc.seq_add(i)
        for _ in range(int(rng.integers(0, 70))):
            alloc.append_slot(i)
    tabs = [alloc.table(i) for i in range(n_seqs)]
    W = max(1, max(len(t) for t in tabs))
    tables = np.full((n_seqs, W), -1, np.int32)
    for i, t in enumerate(tabs):
        tables[i, :len(t)] = t
    lens = np.array([alloc.seq_len(i) for i in range(n_seqs)], np.int32)
    return tables, lens


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("Hq,Hkv", [(40, 40), (32, 8), (12, 2), (8, 1)])
def test_matches_the_rule_and_the_kernels_assumptions(seed, Hq, Hkv):
    tables, lens = random_history(seed)
    got = groups_of(tables, lens, Hq, Hkv)
    assert got == rule(tables, lens, 8 // (Hq // Hkv))
    seen = set()
    for grp, P in got:
        assert 2 <= len(grp) <= 8 // (Hq // Hkv)
        assert not seen & set(grp)
        seen |= set(grp)
        for i in grp:
            assert 16 * P <= lens[i]
            assert (tables[i, :P] == tables[grp[0], :P]).all()


def test_shared_prefix_workload():
    """Llama-2-13B MHA: the 8 forks of the 2,048-token parent are one group
    over its 128 blocks; with G = 4 the same forks make 4 groups of two."""
    case = make_case(CONFIGS[4])
    alloc = pa.BlockAllocator(case.num_blocks, 16, case.free_order.tolist())
    tables, _, _, lens = build_tables(case, alloc)
    assert groups_of(tables, lens, 40, 40) == [(list(range(8)), 128)]
    four = groups_of(tables, lens, 32, 8)
    assert [g for g, _ in four] == [[0, 1], [2, 3], [4, 5], [6, 7]]
    assert all(P == 128 for _, P in four)


def test_short_and_lonely_sequences_form_no_group():
    tables = np.array([[3, 4], [3, 5], [9, 1], [7, 2]], np.int32)
    lens = np.array([15, 32, 20, 17], np.int32)     # sequence 0 has no full block
    assert groups_of(tables, lens, 8, 8) == []
    lens = np.array([16, 32, 20, 17], np.int32)
    assert groups_of(tables, lens, 8, 8) == [([0, 1], 1)]
    tables[1, 0] = 8                                 # nothing shared any more
    assert groups_of(tables, lens, 8, 8) == []
