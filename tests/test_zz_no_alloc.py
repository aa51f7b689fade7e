"""The decode entry point that allocates nothing.

Some callers of this library cannot allocate device memory at the moment they
decode - for example a serving loop whose device memory is budgeted once at
start-up, or a host program that links this library without an allocator of
its own - so they cannot pass the workspace pa_decode_split needs.
pa_decode_split_static uses a static device array inside the library
instead.  These tests call it through the C ABI, twice in a row (the array
keeps the previous call's contents): it must give exactly pa_decode_split's
bits (same kernels, same schedule), agree with the fp64 oracle, leave the
device's free memory unchanged, and refuse what does not fit."""
import ctypes

import pytest
import torch

from tests._gpu import GpuCase, assert_close
from workloads import Config

pytestmark = pytest.mark.gpu

# group 8 (16 query heads over 2 kv heads): the balanced split's records come
# closest to the array's size
GROUP8 = Config(9, "group8-bf16", 16, 2, "bf16", 6, ("fixed", [40, 300, 1000, 1500, 2049, 4000]))


def _call_static(pa, pool, q, bt, sl, scale, out, partition_blocks=0):
    return pa.lib.pa_decode_split_static(
        pool.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(bt.data_ptr()), bt.shape[1],
        ctypes.c_void_p(sl.data_ptr()), q.shape[0], q.shape[1], ctypes.c_float(scale),
        ctypes.c_void_p(out.data_ptr()), pa._DTYPE_CODE[out.dtype], partition_blocks,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("cfg,partition", [(3, 0), (1, 2), (GROUP8, 0)])
def test_static_scratch_gives_the_workspace_entrys_bits_twice(cfg, partition):
    import paged_kv_cache_227_gb300 as pa
    torch.cuda.set_device(0)
    c = GpuCase(cfg)
    pool = c.pool()
    q, bt, sl = c.dev("q"), c.tables_dev(), c.lens_dev("ctx")
    need = pa.pa_decode_workspace_bytes(pool, q.shape[0], q.shape[1], bt.shape[1], partition)
    assert 0 < need <= pa.PA_STATIC_SCRATCH_BYTES
    ref = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    pa.pa_decode_split(pool, q, bt, sl, c.case.scale, ref, partition_blocks=partition)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _call_static(pa, pool, q, bt, sl, c.case.scale, out, partition) == pa.PA_OK
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before, "the call allocated device memory"
        code, detail = pa.pa_check(pool)
        assert code == pa.PA_OK, (pa.strerror(code), detail)
        assert torch.equal(out, ref), f"call {call + 1}: not pa_decode_split's bits"
    assert_close(out, c.reference(after_append=False), "static scratch vs the fp64 oracle")
    pool.close()


def test_static_scratch_rejects_oversized_requests():
    import paged_kv_cache_227_gb300 as pa
    torch.cuda.set_device(0)
    c = GpuCase(1)
    pool = c.pool()
    B, Hq = 4096, 12
    q = torch.zeros(B, Hq, 128, dtype=torch.float16, device="cuda")
    bt = torch.zeros(B, 64, dtype=torch.int32, device="cuda")
    sl = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.zeros(B, Hq, 128, dtype=torch.float32, device="cuda")
    need = pa.pa_decode_workspace_bytes(pool, B, Hq, 64, 1)
    assert need > pa.PA_STATIC_SCRATCH_BYTES
    assert _call_static(pa, pool, q, bt, sl, 0.1, out, 1) == pa.PA_ERR_SCRATCH_LIMIT
    assert pa.strerror(pa.PA_ERR_SCRATCH_LIMIT).startswith("the call needs more workspace")
    pool.close()
