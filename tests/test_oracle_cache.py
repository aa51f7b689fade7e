"""Pins for the oracle's cache-write and block-copy models and the KV-size
closed form."""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle.allocator import ReferenceAllocator
from tests._util import BS, bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_cache_sizes.txt")


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, *nums, src = line.split()
            rows.append((name, [int(x) for x in nums], src))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_kv_cache_bytes_match_the_pages(row):
    """The closed form of "Serving" 23.1 against every size the pages print."""
    name, (layers, kvh, d, L, B, nbytes, expect), src = row
    assert oracle.cache.kv_cache_bytes(layers, kvh, d, L, B, nbytes) == expect


def test_kv_cache_bytes_printed_rounding():
    """The pages' rounded figures: 2 GiB is about 2.15 GB; 64 GiB about 68.7 GB;
    LLaMA-3 8B at 8,192 tokens is 1.0 GiB (twice the context of LLaMA-2 7B in
    half the cache)."""
    kb = oracle.cache.kv_cache_bytes
    assert round(kb(32, 32, 128, 4096, 1, 2) / 1e9, 2) == 2.15
    assert round(kb(32, 32, 128, 4096, 32, 2) / 1e9, 1) == 68.7
    l7 = kb(32, 32, 128, 4096, 1, 2)
    l8 = kb(32, 8, 128, 8192, 1, 2)
    assert l8 * 2 == l7 and l8 == 2 ** 30
    assert oracle.cache.kv_bytes_per_token(28, 2, 128, 2) == 28 * 1024
    assert oracle.cache.kv_bytes_per_token(40, 40, 128, 2) == 800 * 1024


def _pool(seed, N, Hkv, d=128):
    g = torch.Generator().manual_seed(seed)
    return (bits(torch.randn(N, Hkv, BS, d, generator=g).half()),
            bits(torch.randn(N, Hkv, BS, d, generator=g).half()))


def test_append_writes_exactly_the_named_rows():
    """Slot s is row s of the pool seen as [N*16] token rows per head (numpy
    reshape, not the model's own divmod); every other byte is unchanged and
    negative slots write nothing."""
    N, Hkv, d = 6, 3, 128
    kp, vp = _pool(1, N, Hkv)
    g = torch.Generator().manual_seed(2)
    kn = bits(torch.randn(5, Hkv, d, generator=g).half())
    vn = bits(torch.randn(5, Hkv, d, generator=g).half())
    slots = np.array([0, 17, -1, 95, 40], np.int64)
    k2, v2 = oracle.cache.append(kp, vp, kn, vn, slots)
    rows_k = k2.transpose(0, 2, 1, 3).reshape(N * BS, Hkv, d)
    rows_v = v2.transpose(0, 2, 1, 3).reshape(N * BS, Hkv, d)
    old_k = kp.transpose(0, 2, 1, 3).reshape(N * BS, Hkv, d)
    for t, s in enumerate(slots):
        if s >= 0:
            assert np.array_equal(rows_k[s], kn[t]) and np.array_equal(rows_v[s], vn[t])
    untouched = np.setdiff1d(np.arange(N * BS), slots[slots >= 0])
    assert np.array_equal(rows_k[untouched], old_k[untouched])
    assert not np.shares_memory(k2, kp)


def test_append_then_gather_is_the_dense_sequence():
    """Tokens written one by one at the reference allocator's slots are what
    the decode oracle attends over: the result equals torch SDPA on the dense
    tokens, which ties the slot encoding to the table lookup."""
    Hkv, Hq, d, L = 2, 6, 128, 53
    N = 8
    alloc = ReferenceAllocator(N, BS, free_order=[5, 2, 7, 0, 1, 3, 4, 6])
    alloc.seq_add(0)
    g = torch.Generator().manual_seed(3)
    K = torch.randn(L, Hkv, d, generator=g).half()
    V = torch.randn(L, Hkv, d, generator=g).half()
    q = torch.randn(1, Hq, d, generator=g).half()
    kp = np.zeros((N, Hkv, BS, d), np.uint16); vp = kp.copy()
    slots = np.array([alloc.append_slot(0)[0] for _ in range(L)], np.int64)
    kp, vp = oracle.cache.append(kp, vp, bits(K), bits(V), slots)
    table = np.array([alloc.table(0)], np.int32)
    got = oracle.paged_decode(bits(q), kp, vp, 0, table, np.array([L], np.int32), 0.125)
    ref = F.scaled_dot_product_attention(q.double()[:, :, None, :], K.double().permute(1, 0, 2)[None],
                                         V.double().permute(1, 0, 2)[None], scale=0.125, enable_gqa=True)
    np.testing.assert_allclose(got[0], ref[0, :, 0, :].numpy(), rtol=0, atol=1e-12)


def test_copy_blocks_copies_whole_blocks_only():
    N, Hkv = 7, 2
    kp, vp = _pool(4, N, Hkv)
    k2, v2 = oracle.cache.copy_blocks(kp, vp, [1, 4], [6, 0])
    assert np.array_equal(k2[6], kp[1]) and np.array_equal(v2[0], vp[4])
    for b in (1, 2, 3, 4, 5):
        assert np.array_equal(k2[b], kp[b]) and np.array_equal(v2[b], vp[b])
