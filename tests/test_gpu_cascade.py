"""Shared-prefix (cascade) decode against the fp64 decode oracle: the cascade
is an exact rearrangement of attention, so the oracle is the plain definition.
Covers the Llama-2-13B MHA workload with its 2,048-token shared prefix, GQA
groups of two, members whose whole cache is the shared prefix, sequences in
no group, no groups at all, a group that breaks the rules, and repeated calls (the
prefix pass overlaps the suffix pass as a dependent launch: every call must
give the same bits)."""
import numpy as np
import pytest
import torch

import oracle

from ._gpu import ORACLE_THREADS, GpuCase, assert_close, assert_within_one_ulp16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_227_gb300 as pa
    return pa


def cascade(pa, c, tables, lens, groups=None, out_dtype=torch.float32):
    gs, mem, pre = groups if groups is not None else pa.cascade_groups(tables, lens, c.cfg.n_q_heads,
                                                                        c.cfg.n_kv_heads)
    pool = c.pool()
    q = c.dev("q")
    out = torch.full(q.shape, float("nan"), dtype=out_dtype, device="cuda")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    pa.pa_decode_cascade(pool, q, dev(tables), dev(lens), c.case.scale, out, dev(gs), dev(mem), dev(pre))
    torch.cuda.synchronize()
    code, _ = pa.pa_check(pool)
    return out, code, (gs, mem, pre)


def reference(c, tables, lens, rows=None):
    return oracle.paged_decode(c.q, c.kp, c.vp, c.code, tables, lens, c.case.scale, rows=rows,
                               threads=ORACLE_THREADS)


def test_mha_shared_prefix_workload(pa):
    c = GpuCase(4)
    out, code, (gs, mem, pre) = cascade(pa, c, c.tables, c.dec_lens)
    assert code == 0
    assert len(pre) == 1 and pre[0] == 128 and len(mem) == 8, "one group: the 8 forks of the 2,048-token parent"
    assert_close(out, reference(c, c.tables, c.dec_lens), "cascade MHA")


def share(tables, members, P):
    """A copy of host tables in which `members` use the first member's first
    P blocks."""
    t = tables.copy()
    for i in members[1:]:
        t[i, :P] = t[members[0], :P]
    return t


def test_gqa_groups_of_two(pa):
    c = GpuCase(3, lens=[63, 95, 300, 47, 160, 160, 31, 200])
    t = share(c.tables, [0, 3], 3)        # groups of at most 2 members for G = 4
    t = share(t, [1, 2], 5)
    t = share(t, [4, 5], 10)
    lens = c.dec_lens.copy()
    lens[3] = 48                          # whole cache = the shared 3 blocks
    out, code, (gs, mem, pre) = cascade(pa, c, t, lens)
    assert code == 0 and list(pre) == [3, 5, 10]
    assert_close(out, reference(c, t, lens), "cascade GQA")


def test_no_groups_is_plain_decode(pa):
    c = GpuCase(3, lens=[10, 700, 33])
    out, code, (gs, mem, pre) = cascade(pa, c, c.tables, c.dec_lens)
    assert code == 0 and len(pre) == 0
    assert_close(out, reference(c, c.tables, c.dec_lens), "cascade without groups")


def test_native_16bit_output(pa):
    c = GpuCase(4, lens=[2100, 2500, 2048, 3000, 2200, 2600])
    out, code, _ = cascade(pa, c, c.tables, c.dec_lens, out_dtype=torch.float16)
    assert code == 0
    assert_within_one_ulp16(out.cpu(), reference(c, c.tables, c.dec_lens), torch.float16, "cascade fp16 out",
                            vmax=c.vmax())


def test_a_group_that_shares_nothing_is_reported_and_ignored(pa):
    c = GpuCase(3, lens=[64, 64, 64])
    ref = reference(c, c.tables, c.dec_lens)
    for pre in (2, 9):   # 2 blocks that differ between the members; more blocks than they hold
        groups = (np.array([0, 2]), np.array([0, 1]), np.array([pre]))
        out, code, _ = cascade(pa, c, c.tables, c.dec_lens, groups=groups)
        assert code == pa.PA_ERR_DEVICE_CHECK
        assert_close(out, ref, "members decoded without their broken group")


def test_repeated_calls_give_the_same_bits(pa):
    """Back-to-back calls on one stream, with a plain decode between some of
    them: the overlapped passes and their merges always see complete inputs."""
    c = GpuCase(4, lens=[2100, 2500, 2048, 3000, 2200, 2600])
    pool = c.pool()
    q = c.dev("q")
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    bt, sl = dev(c.tables), dev(c.dec_lens)
    gs, mem, pre = (dev(x) for x in pa.cascade_groups(c.tables, c.dec_lens, c.cfg.n_q_heads, c.cfg.n_kv_heads))
    outs = [torch.full(q.shape, float("nan"), device="cuda") for _ in range(12)]
    plain = torch.empty(q.shape, device="cuda")
    for k, out in enumerate(outs):
        pa.pa_decode_cascade(pool, q, bt, sl, c.case.scale, out, gs, mem, pre)
        if k % 3 == 1:
            pa.pa_decode_split(pool, q, bt, sl, c.case.scale, plain)
    torch.cuda.synchronize()
    assert pa.pa_check(pool)[0] == pa.PA_OK
    for out in outs[1:]:
        assert torch.equal(out, outs[0])
    assert_close(outs[0], reference(c, c.tables, c.dec_lens), "cascade, repeated")
