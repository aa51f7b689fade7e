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


def test_a_call_from_another_device_is_refused_before_any_launch(pa):
    """Every launching entry point checks that the current device is the
    pool's.  With one GPU the test makes the pool claim another device (the
    handle's device field, found next to the shape it reports) and expects
    PA_ERR_INVALID from each call; nothing is launched, so no kernel touches
    memory it should not."""
    import ctypes
    c = GpuCase(1)
    pool = c.pool()
    base = ctypes.cast(pool.handle, ctypes.c_void_p).value
    ints = (ctypes.c_int * 4).from_address(base + 128)  # after the 128-byte tensor map
    if (ints[0], ints[1], ints[3]) != (c.case.num_blocks, c.cfg.n_kv_heads, torch.cuda.current_device()):
        pytest.skip("pool handle layout differs")
    q, bt, sl = c.dev("q"), c.tables_dev(), c.lens_dev()
    out = torch.zeros(q.shape, dtype=torch.float32, device="cuda")
    ints[3] = ints[3] + 1
    try:
        assert pa.lib.pa_decode(pool.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(bt.data_ptr()),
                                bt.shape[1], ctypes.c_void_p(sl.data_ptr()), q.shape[0], q.shape[1],
                                ctypes.c_float(0.1), ctypes.c_void_p(out.data_ptr()), pa.PA_FP32,
                                None) == pa.PA_ERR_INVALID
        ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
        assert pa.lib.pa_decode_split(pool.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(bt.data_ptr()),
                                      bt.shape[1], ctypes.c_void_p(sl.data_ptr()), q.shape[0], q.shape[1],
                                      ctypes.c_float(0.1), ctypes.c_void_p(out.data_ptr()), pa.PA_FP32, 0,
                                      ctypes.c_void_p(ws.data_ptr()), ws.numel(), None) == pa.PA_ERR_INVALID
        assert pa.lib.pa_decode_split_static(pool.handle, ctypes.c_void_p(q.data_ptr()),
                                             ctypes.c_void_p(bt.data_ptr()), bt.shape[1],
                                             ctypes.c_void_p(sl.data_ptr()), q.shape[0], q.shape[1],
                                             ctypes.c_float(0.1), ctypes.c_void_p(out.data_ptr()), pa.PA_FP32, 0,
                                             None) == pa.PA_ERR_INVALID
        kn = c.dev("k_new")
        slots = c.slots_dev()
        assert pa.lib.pa_cache_append(pool.handle, ctypes.c_void_p(kn.data_ptr()), ctypes.c_void_p(kn.data_ptr()),
                                      ctypes.c_void_p(slots.data_ptr()), kn.shape[0], None) == pa.PA_ERR_INVALID
        assert pa.lib.pa_selftest_wait_timeout(pool.handle, 1000, None) == pa.PA_ERR_INVALID
    finally:
        ints[3] = ints[3] - 1
    torch.cuda.synchronize()
    assert pa.pa_check(pool)[0] == pa.PA_OK
    pool.close()
