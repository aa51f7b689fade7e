"""Pins for the reference prefix cache (prefix caching by block hashes,
"Paged Attention" teaser on the inference-serving tag page; hash chains and
the one-changed-character rule, posts on the pagedattention tag)."""
import random

import pytest

import oracle.prefix_cache as pc
from oracle.prefix_cache import PrefixCacheAllocator, block_hash, fnv1a64

BS = 16


def test_fnv1a64_published_vectors():
    # test vectors of the FNV-1a 64-bit reference
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


def test_block_hash_byte_layout():
    # parent as 8 little-endian bytes, then each id as 4 little-endian bytes
    toks = [1, -2, 65536] + [0] * 13
    data = (0x0102030405060708).to_bytes(8, "little") + bytes([1, 0, 0, 0, 0xFE, 0xFF, 0xFF, 0xFF, 0, 0, 1, 0]) + bytes(52)
    assert block_hash(0x0102030405060708, toks) == fnv1a64(data)


def chain(prompt):
    hs, parent = [], 0
    for k in range(len(prompt) // BS):
        parent = block_hash(parent, prompt[k * BS:(k + 1) * BS])
        hs.append(parent)
    return hs


def test_one_changed_token_changes_every_later_hash():
    rnd = random.Random(1)
    prompt = [rnd.randrange(50000) for _ in range(10 * BS)]
    base = chain(prompt)
    for p in (0, 5, 17, 63, 64, 100, 159):
        q = list(prompt)
        q[p] += 1
        h = chain(q)
        k = p // BS
        assert h[:k] == base[:k] and all(a != b for a, b in zip(h[k:], base[k:]))


def run(a, seq, prompt, extra=0):
    """A request: cached prefix, then the rest of the prompt and `extra`
    generated tokens appended with ids.  Returns the cached token count."""
    n = a.seq_add_cached(seq, prompt)
    for t in prompt[n:]:
        a.append_token(seq, t)
    for k in range(extra):
        a.append_token(seq, 900000 + k)
    return n


def check_invariants(a):
    counts = [0] * a.num_blocks
    for t in a.tables.values():
        for b in t:
            counts[b] += 1
    assert counts == a.refcount
    assert len(set(a.free)) == len(a.free) and all(a.refcount[b] == 0 for b in a.free)
    assert len(a.free) + sum(c > 0 for c in counts) == a.num_blocks
    for h, (b, parent, toks) in a.index.items():
        assert a.key_of[b] == h and block_hash(parent, toks) == h
    for s, toks in a.tokens.items():
        if toks is not None:
            assert chain(toks) == a.chain[s]
            for k, h in enumerate(a.chain[s]):
                if h in a.index and a.index[h][0] == a.tables[s][k]:
                    assert a.index[h][2] == tuple(toks[k * BS:(k + 1) * BS])


def test_same_prompt_reuses_every_full_block_and_never_the_partial_one():
    a = PrefixCacheAllocator(64)
    prompt = list(range(5 * BS + 7))
    assert run(a, 0, prompt) == 0
    t0 = a.table(0)
    a.seq_free(0)
    assert run(a, 1, prompt) == 5 * BS
    assert a.table(1)[:5] == t0[:5] and a.table(1)[5] != t0[5]
    check_invariants(a)


def test_changed_token_hits_only_the_blocks_before_it():
    a = PrefixCacheAllocator(128)
    prompt = list(range(1000, 1000 + 8 * BS))
    run(a, 0, prompt)
    for s, p in enumerate((0, 3, 16, 40, 127), start=1):
        q = list(prompt)
        q[p] = -q[p]
        assert run(a, s, q) == (p // BS) * BS
        check_invariants(a)


def test_live_sequences_share_cached_blocks():
    a = PrefixCacheAllocator(64)
    prompt = list(range(3 * BS))
    run(a, 0, prompt)
    assert run(a, 1, prompt + [5, 6]) == 3 * BS
    assert all(a.refcount[b] == 2 for b in a.table(0))
    check_invariants(a)


def test_freed_blocks_stay_cached_until_the_free_list_reuses_them():
    a = PrefixCacheAllocator(8)
    prompt = list(range(4 * BS))
    run(a, 0, prompt)
    a.seq_free(0)               # free list: 4 untouched blocks, then the 4 cached ones
    run(a, 1, [7] * (5 * BS))   # takes the 4 untouched and the first cached block
    assert a.seq_add_cached(2, prompt) == 0, "block 0 of the chain was evicted, so nothing after it hits"
    assert a.hits == 0
    check_invariants(a)


def test_hash_collision_is_a_miss(monkeypatch):
    a = PrefixCacheAllocator(32)
    run(a, 0, list(range(2 * BS)))
    monkeypatch.setattr(pc, "block_hash", lambda parent, toks: 42)  # every block collides
    a2 = PrefixCacheAllocator(32)
    run(a2, 0, list(range(2 * BS)))
    assert run(a2, 1, list(range(100, 100 + 2 * BS))) == 0
    assert run(a2, 2, list(range(2 * BS))) == BS, "first block verified; the second's entry belongs to nobody"


def test_cached_prefix_equals_brute_force_longest_common_prefix():
    rnd = random.Random(7)
    a = PrefixCacheAllocator(4096)
    done = []
    base = [rnd.randrange(1000) for _ in range(40 * BS)]
    for s in range(60):
        if done and rnd.random() < 0.7:
            src = rnd.choice(done)
            cut = rnd.randrange(len(src) + 1)
            prompt = src[:cut] + [rnd.randrange(1000) for _ in range(rnd.randrange(3 * BS))]
        else:
            prompt = base[:rnd.randrange(len(base))]
        expect = 0
        for d in done:
            lcp = 0
            while lcp < min(len(d), len(prompt)) and d[lcp] == prompt[lcp]:
                lcp += 1
            expect = max(expect, (lcp // BS) * BS)
        assert run(a, s, prompt) == expect
        done.append(prompt)
        if rnd.random() < 0.5:
            a.seq_free(s)
        check_invariants(a)


def test_untracked_sequences_are_not_hashed():
    a = PrefixCacheAllocator(16)
    a.seq_add(0)
    for _ in range(2 * BS):
        a.append_slot(0)
    assert a.index == {}
    a.seq_free(0)
    assert a.seq_add_cached(1, list(range(2 * BS))) == 0


def test_out_of_blocks_raises():
    a = PrefixCacheAllocator(1)
    with pytest.raises(MemoryError):
        run(a, 0, list(range(BS + 1)))
