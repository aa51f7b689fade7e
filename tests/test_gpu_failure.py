"""Failure detection without a GPU fault: the kernels' bounded mbarrier wait
runs out on a barrier that nothing arrives at, the host reads PA_ERR_TIMEOUT
through pa_check, and the context keeps working (a decode right after it is
still correct)."""
import time

import pytest
import torch

import oracle

from ._gpu import ORACLE_THREADS, GpuCase, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_227_gb300 as pa
    return pa


def test_bounded_wait_times_out_and_the_context_survives(pa):
    c = GpuCase(3, lens=[40, 300, 7])
    pool = c.pool()
    t0 = time.perf_counter()
    assert pa.pa_selftest_wait_timeout(pool, 20_000_000, None) == pa.PA_OK   # 20 ms
    code, detail = pa.pa_check(pool)
    assert (code, detail) == (pa.PA_ERR_TIMEOUT, 9), "the wait site is reported"
    assert time.perf_counter() - t0 < 5.0
    assert pa.pa_check(pool)[0] == pa.PA_OK, "pa_check clears the error word"
    out = torch.full(c.dev("q").shape, float("nan"), dtype=torch.float32, device="cuda")
    pa.pa_decode_split(pool, c.dev("q"), c.tables_dev(), c.lens_dev(), c.case.scale, out)
    torch.cuda.synchronize()
    assert pa.pa_check(pool)[0] == pa.PA_OK
    ref = oracle.paged_decode(c.q, c.kp, c.vp, c.code, c.tables, c.dec_lens, c.case.scale,
                              threads=ORACLE_THREADS)
    assert_close(out, ref, "decode after a timed-out wait")


def test_selftest_rejects_limits_out_of_range(pa):
    pool = pa.Pool(4, 1, torch.float16)
    for limit in (0, -5, 2_000_000_000):
        assert pa.pa_selftest_wait_timeout(pool, limit, None) == pa.PA_ERR_INVALID
    assert pa.pa_check(pool)[0] == pa.PA_OK
