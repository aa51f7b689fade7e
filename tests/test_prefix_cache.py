"""The library's prefix cache (pa_alloc_seq_add_cached / pa_alloc_append_token)
against the reference prefix cache, bit for bit, on random request histories
(host code: runs without a GPU)."""
import random

import pytest

from oracle.prefix_cache import PrefixCacheAllocator, block_hash

BS = 16


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_227_gb300 as pa
    return pa


def both(fn_ref, fn_lib):
    """Calls both; they must agree on the result or both run out of blocks."""
    try:
        r = fn_ref()
    except MemoryError:
        with pytest.raises(MemoryError):
            fn_lib()
        return None
    assert fn_lib() == r
    return r


def same_state(lib_a, ref, seqs):
    assert lib_a.num_free() == len(ref.free)
    for b in range(ref.num_blocks):
        assert lib_a.refcount(b) == ref.refcount[b]
        assert lib_a.block_hash(b) == ref.key_of.get(b)
    for s in seqs:
        assert lib_a.table(s) == ref.table(s)
        assert lib_a.seq_len(s) == ref.lengths[s]
    q, h, c = lib_a.prefix_stats()
    assert (q, h, c) == (ref.queries, ref.hits, len(ref.index))


def test_hash_of_a_block_matches_the_reference(pa):
    a = pa.BlockAllocator(4)
    a.seq_add_cached(0, [])
    toks = [3, -1, 70000, 5] * 4
    for t in toks:
        a.append_token(0, t)
    assert a.block_hash(a.table(0)[0]) == block_hash(0, toks)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_random_histories_match_the_reference(pa, seed):
    rnd = random.Random(seed)
    N = 96
    order = rnd.sample(range(N), N)
    a, ref = pa.BlockAllocator(N, BS, order), PrefixCacheAllocator(N, BS, order)
    live, done, nxt = [], [], 0
    base = [rnd.randrange(500) for _ in range(12 * BS)]
    for step in range(250):
        op = rnd.random()
        if op < 0.25 or not live:      # a request whose prompt may share a prefix
            if done and rnd.random() < 0.6:
                src = rnd.choice(done)
                cut = rnd.randrange(len(src) + 1)
                prompt = src[:cut] + [rnd.randrange(500) for _ in range(rnd.randrange(2 * BS))]
            else:
                prompt = base[:rnd.randrange(len(base))]
            n_ref = ref.seq_add_cached(nxt, prompt)
            assert a.seq_add_cached(nxt, prompt) == n_ref
            live.append(nxt)
            done.append(prompt)
            for t in prompt[n_ref:]:
                if both(lambda: ref.append_token(nxt, t), lambda: a.append_token(nxt, t)) is None:
                    break
            nxt += 1
        elif op < 0.35:
            p = rnd.choice(live)
            ref.fork(p, nxt)
            a.fork(p, nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.5:
            s = rnd.choice(live)
            ref.seq_free(s)
            a.seq_free(s)
            live.remove(s)
        elif op < 0.55:
            s = rnd.choice(live)
            both(lambda: ref.append_slot(s), lambda: a.append_slot(s))
        else:
            s = rnd.choice(live)
            t = rnd.randrange(500)
            both(lambda: ref.append_token(s, t), lambda: a.append_token(s, t))
        same_state(a, ref, live)


def test_one_changed_token_voids_every_later_block(pa):
    a = pa.BlockAllocator(64)
    prompt = list(range(7 * BS))
    a.seq_add_cached(0, [])
    for t in prompt:
        a.append_token(0, t)
    for s, p in enumerate((0, 15, 16, 50, 111), start=1):
        q = list(prompt)
        q[p] = 10 ** 6
        assert a.seq_add_cached(s, q) == (p // BS) * BS
        a.seq_free(s)
