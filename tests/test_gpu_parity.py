"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Bar: bit-exact for the cache write and block copy; attention within
max |err| <= 2e-3 absolute and <= 1e-2 of the largest output magnitude with
fp32 output, and within 1 ulp of the rounded oracle with native 16-bit output.
Every unused pool slot holds NaN, so a read outside a sequence shows up."""
import numpy as np
import pytest
import torch

from tests._gpu import GpuCase, assert_close, assert_within_one_ulp16, bits, from_bits, NAN_BITS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_227_gb300 as pa
    torch.cuda.set_device(0)
    return pa


def _check_ok(pa, pool):
    code, detail = pa.pa_check(pool)
    assert code == pa.PA_OK, (pa.strerror(code), detail)


def test_append_bit_exact(pa):
    c = GpuCase(1)
    pool = c.pool()
    rng = np.random.default_rng(0)
    n_tok = 40
    slots = rng.choice(c.case.num_blocks * 16, size=n_tok, replace=False).astype(np.int64)
    slots[[3, 17]] = -1
    g = torch.Generator().manual_seed(1)
    kn = torch.randn(n_tok, c.cfg.n_kv_heads, 128, generator=g).half()
    vn = torch.randn(n_tok, c.cfg.n_kv_heads, 128, generator=g).half()
    pa.pa_cache_append(pool, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    _check_ok(pa, pool)
    import oracle
    k_ref, v_ref = oracle.cache.append(c.kp, c.vp, bits(kn), bits(vn), slots)
    assert np.array_equal(bits(pool.k), k_ref)
    assert np.array_equal(bits(pool.v), v_ref)


def test_append_out_of_range_slot_is_skipped_and_reported(pa):
    c = GpuCase(1)
    pool = c.pool()
    kn = torch.ones(2, c.cfg.n_kv_heads, 128, dtype=torch.float16, device="cuda")
    slots = torch.tensor([5, c.case.num_blocks * 16], dtype=torch.int64, device="cuda")
    pa.pa_cache_append(pool, kn, kn, slots)
    code, detail = pa.pa_check(pool)
    assert code == pa.PA_ERR_DEVICE_CHECK and detail == c.case.num_blocks * 16
    k = bits(pool.k)
    assert (k[0, :, 5, :] == 0x3C00).all()          # the valid row was written
    assert pa.pa_check(pool)[0] == pa.PA_OK          # the error word was cleared


def test_copy_blocks_bit_exact(pa):
    import oracle
    c = GpuCase(1)
    pool = c.pool()
    src = np.array([3, 10, 0], np.int32)
    dst = np.array([60, 61, 63], np.int32)
    pa.pa_copy_blocks(pool, torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda())
    _check_ok(pa, pool)
    k_ref, v_ref = oracle.cache.copy_blocks(c.kp, c.vp, src, dst)
    assert np.array_equal(bits(pool.k), k_ref) and np.array_equal(bits(pool.v), v_ref)


def _run(pa, c, mode, pool, out_dtype=torch.float32, partition=0, after_append=True):
    q = c.dev("q")
    out = torch.empty(q.shape, dtype=out_dtype, device="cuda")
    bt = c.tables_dev()
    if mode == "fused":
        pa.pa_append_decode(pool, q, c.dev("k_new"), c.dev("v_new"), bt, c.lens_dev("dec"),
                            c.case.scale, out, partition_blocks=partition)
    else:
        if after_append:
            pa.pa_cache_append(pool, c.dev("k_new"), c.dev("v_new"), c.slots_dev())
        lens = c.lens_dev("dec" if after_append else "ctx")
        if mode == "segment":
            pa.pa_decode(pool, q, bt, lens, c.case.scale, out)
        else:
            pa.pa_decode_split(pool, q, bt, lens, c.case.scale, out, partition_blocks=partition)
    _check_ok(pa, pool)
    return out


MODES = [("segment", 0), ("split", 0), ("split", 1), ("split", 3), ("split", 16), ("fused", 0), ("fused", 2)]


@pytest.mark.parametrize("mode,partition", MODES, ids=[f"{m}-{p}" for m, p in MODES])
def test_tiny_config_all_paths(pa, mode, partition):
    """Qwen2.5-1.5B layout, fp16, lengths 17/100/256/513 plus one append each."""
    c = GpuCase(1)
    ref = c.reference(after_append=True)
    pool = c.pool()
    out = _run(pa, c, mode, pool, partition=partition)
    assert_close(out, ref, f"config 1 {mode}/{partition}")
    if mode == "fused":
        k_ref, v_ref = c.appended_pools()
        assert np.array_equal(bits(pool.k), k_ref) and np.array_equal(bits(pool.v), v_ref)


def test_tiny_config_before_append(pa):
    c = GpuCase(1)
    ref = c.reference(after_append=False)
    for mode in ("segment", "split"):
        out = _run(pa, c, mode, c.pool(), after_append=False)
        assert_close(out, ref, f"config 1 before append {mode}")


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_native_16bit_output_within_one_ulp(pa, out_dtype):
    c = GpuCase(1)
    ref = c.reference()
    out = _run(pa, c, "split", c.pool(), out_dtype=out_dtype)
    assert_within_one_ulp16(out, ref, out_dtype, "config 1 native output", vmax=c.vmax())


def test_fused_never_reads_the_new_slot(pa):
    """The new token's slot holds NaN before the fused call; the result must
    come from k_new/v_new, and the slot must hold them afterwards."""
    c = GpuCase(3, lens=[15, 16, 31, 200, 1000, 17, 1, 64])
    nan = np.uint16(NAN_BITS[c.dtype])
    for s in c.slots.tolist():
        c.kp[s // 16, :, s % 16, :] = nan
        c.vp[s // 16, :, s % 16, :] = nan
    ref = c.reference()
    pool = c.pool()
    out = _run(pa, c, "fused", pool)
    assert_close(out, ref, "fused with NaN slots")
    k_ref, v_ref = c.appended_pools()
    assert np.array_equal(bits(pool.k), k_ref) and np.array_equal(bits(pool.v), v_ref)


FULL = [(2, "split", 0), (2, "segment", 0), (3, "fused", 0), (3, "split", 0), (3, "segment", 0),
        (3, "split", 8), (4, "split", 0), (4, "segment", 0), (5, "fused", 0), (5, "fused", 64),
        (5, "fused", 32), (5, "fused", 128)]


@pytest.mark.parametrize("cfg,mode,partition", FULL, ids=[f"cfg{a}-{b}-{p}" for a, b, p in FULL])
def test_full_size_configs(pa, cfg, mode, partition):
    """Every config at its full size, every output row against the oracle.
    (cfg 3, fused, 0) is the launch the benchmark times."""
    c = GpuCase(cfg)
    ref = c.reference()
    pool = c.pool()
    out = _run(pa, c, mode, pool, partition=partition)
    assert_close(out, ref, f"config {cfg} {mode}/{partition}")
    if mode == "fused":
        k_ref, v_ref = c.appended_pools()
        assert np.array_equal(bits(pool.k), k_ref)
    pool.close()


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8])
def test_every_group_size(pa, G):
    from workloads import Config
    Hkv = 2
    cfg = Config(90 + G, f"group{G}", G * Hkv, Hkv, "bf16", 6, ("fixed", [0, 1, 15, 16, 17, 300]))
    c = GpuCase(cfg)
    ref = c.reference()
    for mode, part in (("segment", 0), ("split", 0), ("fused", 1)):
        out = _run(pa, c, mode, c.pool(), partition=part)
        assert_close(out, ref, f"G={G} {mode}")


def test_empty_sequences_give_zero_rows(pa):
    from workloads import Config
    cfg = Config(80, "empties", 8, 2, "fp16", 3, ("fixed", [40, 7, 90]))
    c = GpuCase(cfg)
    lens = c.dec_lens.copy()
    lens[1] = 0
    ref_lens = lens
    import oracle
    kp, vp = c.appended_pools()
    ref = oracle.paged_decode(c.q, kp, vp, c.code, c.tables, ref_lens, c.case.scale)
    for split in (False, True):
        pool = c.pool()
        pa.pa_cache_append(pool, c.dev("k_new"), c.dev("v_new"), c.slots_dev())
        out = torch.full((3, 8, 128), 7.0, device="cuda")
        fn = pa.pa_decode_split if split else pa.pa_decode
        fn(pool, c.dev("q"), c.tables_dev(), torch.from_numpy(lens).cuda(), c.case.scale, out)
        _check_ok(pa, pool)
        assert (out[1] == 0).all()
        assert_close(out, ref, f"empty rows split={split}")


def test_block_permutation_gives_bit_identical_output(pa):
    c = GpuCase(3, lens=[33, 700, 5, 1200, 64, 250])
    out1 = _run(pa, c, "split", c.pool())
    pi = np.random.default_rng(3).permutation(c.case.num_blocks).astype(np.int32)
    kp2 = np.empty_like(c.kp); vp2 = np.empty_like(c.vp)
    kp2[pi] = c.kp; vp2[pi] = c.vp
    c.kp, c.vp = kp2, vp2
    c.tables = np.where(c.tables >= 0, pi[np.maximum(c.tables, 0)], -1).astype(np.int32)
    c.slots = (pi[c.slots // 16].astype(np.int64) * 16 + c.slots % 16)
    out2 = _run(pa, c, "split", c.pool())
    assert torch.equal(out1, out2)


def test_block_ids_past_4_GiB_offsets(pa):
    """The same sequences placed in the top blocks of a 140,000-block pool
    (4.6 GB per K or V array, so byte offsets pass 2^32): the cache write puts
    the new rows at the same bits, the block copy moves whole blocks, and every
    decode path gives bit-identical output to the small pool's."""
    c = GpuCase(3, lens=[33, 700, 5, 1200, 64])
    ref = c.reference(after_append=True)
    small = {m: _run(pa, c, m, c.pool()) for m in ("fused", "split", "segment")}
    assert_close(small["split"], ref, "small pool")
    n_big = 140_000
    top = (n_big - 1 - np.arange(c.case.num_blocks)).astype(np.int64)   # block b -> n_big-1-b
    big_k, big_v = c.kp, c.vp
    k_ref, v_ref = c.appended_pools()          # the small pool after the append
    c.tables = np.where(c.tables >= 0, top[np.maximum(c.tables, 0)], -1).astype(np.int32)
    c.slots = top[c.slots // 16] * 16 + c.slots % 16
    for m in ("fused", "split", "segment"):
        pool = pa.Pool(n_big, c.cfg.n_kv_heads, c.dtype)
        idx = torch.from_numpy(top).cuda()
        pool.k[idx] = from_bits(big_k, c.dtype)
        pool.v[idx] = from_bits(big_v, c.dtype)
        out = _run(pa, c, m, pool)
        assert torch.equal(out, small[m]), m
        assert np.array_equal(bits(pool.k[idx]), k_ref) and np.array_equal(bits(pool.v[idx]), v_ref)
    src = torch.tensor([n_big - 1, n_big - 5], dtype=torch.int32, device="cuda")
    dst = torch.tensor([3, n_big - 2000], dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(pool, src, dst)
    _check_ok(pa, pool)
    assert torch.equal(pool.k[dst.long()], pool.k[src.long()]) and torch.equal(pool.v[dst.long()], pool.v[src.long()])
    del pool


def test_largest_split_batch(pa):
    """4,096 sequences (the split schedules' limit: their prefix lives in
    shared memory) of 1 to 81 tokens after the append, on every path; one
    sequence more is refused by the split schedules."""
    from workloads import Config
    cfg = Config(90, "max-batch-8q-2kv-bf16", 8, 2, "bf16", 4096, ("uniform", 0, 80))
    c = GpuCase(cfg)
    ref = c.reference(after_append=True)
    for mode in ("fused", "split", "segment"):
        assert_close(_run(pa, c, mode, c.pool()), ref, f"batch 4096 {mode}")
    pool = pa.Pool(4, 2, torch.bfloat16)
    q = torch.zeros(4097, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(4097, 8, 128, device="cuda")
    bt = torch.full((4097, 1), -1, dtype=torch.int32, device="cuda")
    sl = torch.zeros(4097, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PagedAttentionError):
        pa.pa_decode_split(pool, q, bt, sl, 0.1, out)
    pa.pa_decode(pool, q, bt, sl, 0.1, out)          # the segment schedule has no such limit
    _check_ok(pa, pool)
    assert (out == 0).all()


def unshare(c):
    """Host side of the shared-prefix test: every sequence after the first gets
    private copies (appended to the pool) of the blocks it shares."""
    shared = {b for b in range(c.case.num_blocks) if c.alloc.refcount[b] > 1}
    assert shared, "config 4 must share blocks"
    tables = c.tables.copy()
    extra_k, extra_v = [], []
    n = c.case.num_blocks
    for i in range(1, len(c.dec_lens)):
        for j, b in enumerate(tables[i].tolist()):
            if b in shared:
                extra_k.append(c.kp[b]); extra_v.append(c.vp[b])
                tables[i, j] = n
                n += 1
    kp = np.concatenate([c.kp, np.stack(extra_k)])
    vp = np.concatenate([c.vp, np.stack(extra_v)])
    return kp, vp, tables, n


def test_shared_prefix_equals_unshared_copy(pa):
    """Sequences sharing prefix blocks give bit-identical results to the same
    sequences with private copies of those blocks."""
    c = GpuCase(4, lens=[2100, 2500, 2048, 3000, 2200, 2600])
    out_shared = _run(pa, c, "split", c.pool())
    kp, vp, tables, n = unshare(c)
    c.kp, c.vp, c.tables = kp, vp, tables
    c.case.num_blocks = n
    out_copy = _run(pa, c, "split", c.pool())
    assert torch.equal(out_shared, out_copy)


def test_copy_on_write_flow(pa):
    """Fork at an unaligned length, append to the child: the allocator asks for
    a copy, pa_copy_blocks makes it, the pool matches the oracle's byte model
    of the same writes, the parent's rows are untouched and both outputs
    match the oracle."""
    import oracle
    from oracle.allocator import ReferenceAllocator
    d, Hkv, Hq = 128, 2, 8
    N = 12
    alloc = pa.BlockAllocator(N, 16, list(range(N)))
    ref_alloc = ReferenceAllocator(N, 16, list(range(N)))
    g = torch.Generator().manual_seed(9)
    pool = pa.Pool(N, Hkv, torch.bfloat16)          # zero-filled by pa_pool_create
    kp = np.zeros((N, Hkv, 16, d), np.uint16); vp = kp.copy()
    K = torch.randn(40, Hkv, d, generator=g).bfloat16()
    V = torch.randn(40, Hkv, d, generator=g).bfloat16()
    alloc.seq_add(0); ref_alloc.seq_add(0)
    slots = [alloc.append_slot(0)[0] for _ in range(35)]
    assert slots == [ref_alloc.append_slot(0)[0] for _ in range(35)]
    pa.pa_cache_append(pool, K[:35].cuda(), V[:35].cuda(), torch.tensor(slots, device="cuda"))
    kp, vp = oracle.cache.append(kp, vp, bits(K[:35]), bits(V[:35]), slots)
    alloc.fork(0, 1); ref_alloc.fork(0, 1)
    slot, cs, cd = alloc.append_slot(1)
    assert (slot, cs, cd) == ref_alloc.append_slot(1) and cs >= 0
    pa.pa_copy_blocks(pool, torch.tensor([cs], dtype=torch.int32, device="cuda"),
                      torch.tensor([cd], dtype=torch.int32, device="cuda"))
    kp, vp = oracle.cache.copy_blocks(kp, vp, [cs], [cd])
    pa.pa_cache_append(pool, K[35:36].cuda(), V[35:36].cuda(), torch.tensor([slot], device="cuda"))
    kp, vp = oracle.cache.append(kp, vp, bits(K[35:36]), bits(V[35:36]), [slot])
    _check_ok(pa, pool)
    assert np.array_equal(bits(pool.k), kp) and np.array_equal(bits(pool.v), vp)
    q = torch.randn(2, Hq, d, generator=g).bfloat16()
    tables = np.array([alloc.table(0), alloc.table(1)], np.int32)
    assert tables[0, 2] == cs and tables[1, 2] == cd
    lens = np.array([35, 36], np.int32)
    out = torch.empty(2, Hq, d, device="cuda")
    pa.pa_decode(pool, q.cuda(), torch.from_numpy(tables).cuda(), torch.from_numpy(lens).cuda(), 0.09, out)
    _check_ok(pa, pool)
    ref = oracle.paged_decode(bits(q), kp, vp, 1, tables, lens, 0.09)
    assert_close(out, ref, "copy-on-write")
    # the parent's last block still holds exactly its own three tokens
    kb = bits(pool.k)
    assert np.array_equal(kb[cs, :, :3], bits(K[32:35]).transpose(1, 0, 2))
    assert not kb[cs, :, 3:].any()


def test_out_of_range_table_entry_is_reported_not_read(pa):
    c = GpuCase(1)
    pool = c.pool()
    bad = c.tables.copy()
    bad[2, 3] = c.case.num_blocks + 5
    out = torch.empty(4, 12, 128, device="cuda")
    pa.pa_decode_split(pool, c.dev("q"), torch.from_numpy(bad).cuda(), c.lens_dev("ctx"), c.case.scale, out)
    code, detail = pa.pa_check(pool)
    assert code == pa.PA_ERR_DEVICE_CHECK and detail == c.case.num_blocks + 5
    # the other sequences are still right
    ref = c.reference(after_append=False)
    assert_close(out[[0, 1, 3]], ref[[0, 1, 3]], "rows without the bad entry")


def test_too_long_sequence_is_clamped_and_reported(pa):
    c = GpuCase(1)
    pool = c.pool()
    lens = c.ctx_lens.copy()
    lens[0] = 16 * c.tables.shape[1] + 100
    out = torch.empty(4, 12, 128, device="cuda")
    pa.pa_decode(pool, c.dev("q"), c.tables_dev(), torch.from_numpy(lens).cuda(), c.case.scale, out)
    code, _ = pa.pa_check(pool)
    assert code == pa.PA_ERR_DEVICE_CHECK


def test_host_side_errors(pa):
    c = GpuCase(1)
    pool = c.pool()
    q = c.dev("q")
    out = torch.empty(4, 12, 128, device="cuda")
    bt, sl = c.tables_dev(), c.lens_dev()
    call = pa.lib.pa_decode
    assert call(pool.handle, q.data_ptr(), bt.data_ptr(), 0, sl.data_ptr(), 4, 12, 0.1,
                out.data_ptr(), 2, None) == pa.PA_ERR_INVALID          # no table columns
    assert call(pool.handle, q.data_ptr(), bt.data_ptr(), bt.shape[1], sl.data_ptr(), 4, 7, 0.1,
                out.data_ptr(), 2, None) == pa.PA_ERR_INVALID          # 7 q heads over 2 kv heads
    assert call(pool.handle, q.data_ptr(), bt.data_ptr(), bt.shape[1], sl.data_ptr(), 4, 12, 0.1,
                out.data_ptr(), 5, None) == pa.PA_ERR_INVALID          # bad output type
    assert call(pool.handle, q.data_ptr(), bt.data_ptr(), bt.shape[1], sl.data_ptr(), 4, 36, 0.1,
                out.data_ptr(), 2, None) == pa.PA_ERR_UNSUPPORTED      # group 18 > 8
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedAttentionError):
        pa.pa_decode_split(pool, q, bt, sl, 0.1, out, workspace=small)
    # table rows addressed by 32-bit element offsets: 4096 x 2^20 entries is refused
    assert pa.lib.pa_decode_cascade_workspace_bytes(pool.handle, 4096, 12, 1 << 20, 1) == 0
    assert pa.lib.pa_decode_multi_workspace_bytes(pool.handle, 4096, 4096, 12, 1 << 20) == 0
    assert pa.lib.pa_decode_multi_workspace_bytes(pool.handle, 8, 4, 12, 64) > 0
