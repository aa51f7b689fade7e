"""The library's C++ host allocator reproduces the oracle's reference allocator
bit for bit (tables, slots, copy-on-write pairs, reference counts, free list
size) on random histories of add / fork / append / free."""
import random

import numpy as np
import pytest

from oracle.allocator import ReferenceAllocator


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_227_gb300 as pa
    return pa


@pytest.mark.parametrize("seed", range(12))
def test_matches_reference_on_random_histories(pa, seed):
    rnd = random.Random(seed)
    N = rnd.choice([8, 32, 100])
    order = rnd.sample(range(N), N)
    ref = ReferenceAllocator(N, 16, order)
    lib = pa.BlockAllocator(N, 16, order)
    live, nxt = [], 0
    for _ in range(600):
        op = rnd.random()
        if op < 0.08 or not live:
            ref.seq_add(nxt); lib.seq_add(nxt); live.append(nxt); nxt += 1
        elif op < 0.16:
            p = rnd.choice(live)
            ref.fork(p, nxt); lib.fork(p, nxt); live.append(nxt); nxt += 1
        elif op < 0.22:
            s = rnd.choice(live)
            ref.seq_free(s); lib.seq_free(s); live.remove(s)
        else:
            s = rnd.choice(live)
            try:
                want = ref.append_slot(s)
            except MemoryError:
                with pytest.raises(MemoryError):
                    lib.append_slot(s)
                continue
            assert lib.append_slot(s) == want
        assert lib.num_free() == ref.num_free()
    for s in live:
        assert lib.table(s) == ref.table(s)
        assert lib.seq_len(s) == ref.lengths[s]
    assert [lib.refcount(b) for b in range(N)] == ref.refcount


def test_extend_equals_repeated_append(pa):
    ref = ReferenceAllocator(40, 16, list(range(39, -1, -1)))
    lib = pa.BlockAllocator(40, 16, list(range(39, -1, -1)))
    ref.seq_add(0); lib.seq_add(0)
    for _ in range(20):
        ref.append_slot(0)
    lib.extend(0, 20)
    ref.fork(0, 1); lib.fork(0, 1)
    want = [ref.append_slot(1) for _ in range(30)]
    slots, cow = lib.extend(1, 30)
    assert slots.tolist() == [w[0] for w in want]
    assert cow == (want[0][1], want[0][2]) and cow[0] >= 0
    assert lib.table(1) == ref.table(1)


def test_errors(pa):
    a = pa.BlockAllocator(2, 16)
    a.seq_add(0)
    with pytest.raises(pa.PagedAttentionError):
        a.seq_add(0)
    with pytest.raises(pa.PagedAttentionError):
        a.fork(5, 6)
    a.extend(0, 32)
    with pytest.raises(MemoryError):
        a.append_slot(0)
    assert a.seq_len(0) == 32 and a.num_free() == 0
    with pytest.raises(pa.PagedAttentionError):
        pa.BlockAllocator(3, 16, [0, 0, 1])
