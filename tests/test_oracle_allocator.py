"""Pins for the reference allocator: invariants of paging with shared blocks
("Serving" 23.4: blocks handed out as a sequence grows, shared by sequences
with a common prefix; "Paged Attention" teaser: copy-on-write)."""
import random

import pytest

from oracle.allocator import ReferenceAllocator

BS = 16


def check_invariants(a):
    counts = [0] * a.num_blocks
    for t in a.tables.values():
        for b in t:
            counts[b] += 1
    assert counts == a.refcount, "refcount = number of tables holding the block"
    free = list(a.free)
    assert len(set(free)) == len(free)
    assert all(a.refcount[b] == 0 for b in free)
    assert len(free) + sum(1 for c in counts if c > 0) == a.num_blocks
    for s, t in a.tables.items():
        L = a.lengths[s]
        assert len(t) == -(-L // BS), "blocks allocated only as the sequence grows"
        assert len(t) * BS - L <= BS - 1, "waste is under one block per sequence"


def test_random_histories_keep_invariants():
    rnd = random.Random(0)
    for trial in range(30):
        a = ReferenceAllocator(64, BS, free_order=rnd.sample(range(64), 64))
        live, nxt = [], 0
        for step in range(400):
            op = rnd.random()
            try:
                if op < 0.1 or not live:
                    a.seq_add(nxt); live.append(nxt); nxt += 1
                elif op < 0.2:
                    a.fork(rnd.choice(live), nxt); live.append(nxt); nxt += 1
                elif op < 0.3:
                    s = rnd.choice(live); a.seq_free(s); live.remove(s)
                else:
                    a.append_slot(rnd.choice(live))
            except MemoryError:
                pass
            check_invariants(a)


def test_slot_points_into_the_table_at_the_position():
    a = ReferenceAllocator(10, BS, free_order=[3, 9, 1, 0, 2, 4, 5, 6, 7, 8])
    a.seq_add(0)
    for p in range(40):
        slot, cs, cd = a.append_slot(0)
        assert (cs, cd) == (-1, -1)
        assert slot // BS == a.table(0)[p // BS] and slot % BS == p % BS
    assert a.table(0) == [3, 9, 1]


def test_copy_on_write_only_for_a_shared_partial_block():
    a = ReferenceAllocator(8, BS)
    a.seq_add(0)
    for _ in range(20):          # 20 tokens: block 0 full, block 1 holds 4
        a.append_slot(0)
    a.fork(0, 1)
    parent_table = a.table(0)
    assert a.refcount[0] == 2 and a.refcount[1] == 2
    slot, cs, cd = a.append_slot(1)
    assert (cs, cd) == (1, 2) and slot == 2 * BS + 4
    assert a.table(0) == parent_table, "the parent is untouched"
    assert a.table(1) == [0, 2] and a.refcount[1] == 1 and a.refcount[2] == 1
    # a second append to the child no longer copies
    assert a.append_slot(1)[1:] == (-1, -1)
    # the parent now owns block 1 alone: no copy either
    assert a.append_slot(0)[1:] == (-1, -1)


def test_block_aligned_fork_never_copies():
    a = ReferenceAllocator(8, BS)
    a.seq_add(0)
    for _ in range(32):
        a.append_slot(0)
    a.fork(0, 1)
    slot, cs, cd = a.append_slot(1)
    assert (cs, cd) == (-1, -1) and a.table(1)[:2] == a.table(0)


def test_out_of_blocks_changes_nothing():
    a = ReferenceAllocator(2, BS)
    a.seq_add(0)
    for _ in range(32):
        a.append_slot(0)
    before = (list(a.free), list(a.refcount), a.table(0), a.lengths[0])
    with pytest.raises(MemoryError):
        a.append_slot(0)
    assert (list(a.free), list(a.refcount), a.table(0), a.lengths[0]) == before


def test_free_returns_blocks_fifo_in_table_order():
    a = ReferenceAllocator(6, BS, free_order=[5, 4, 3, 2, 1, 0])
    a.seq_add(0)
    for _ in range(40):
        a.append_slot(0)
    assert a.table(0) == [5, 4, 3]
    a.seq_free(0)
    assert list(a.free) == [2, 1, 0, 5, 4, 3]
