"""The decode entry point that allocates nothing.

Some callers of this library cannot allocate device memory at the moment they
decode - for example code that is being captured into a CUDA graph, or a
serving loop whose memory is budgeted once at start-up - so they cannot pass
the workspace pa_decode_split needs.  pa_decode_split_static uses a static
device array inside the library instead.  These tests call it through the C
ABI, twice in a row (the array keeps the previous call's contents), and
compare its output with pa_decode_split's under the parity tolerance."""
import ctypes

import numpy as np
import pytest
import torch

from tests._gpu import ABS_TOL, REL_TOL, GpuCase

pytestmark = pytest.mark.gpu


def _call_static(pa, pool, q, bt, sl, scale, out, partition_blocks=0):
    return pa.lib.pa_decode_split_static(
        pool.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(bt.data_ptr()), bt.shape[1],
        ctypes.c_void_p(sl.data_ptr()), q.shape[0], q.shape[1], ctypes.c_float(scale),
        ctypes.c_void_p(out.data_ptr()), pa._DTYPE_CODE[out.dtype], partition_blocks,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _close(a, b, what):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    err = np.abs(a - b).max()
    bound = min(ABS_TOL, REL_TOL * np.abs(b).max())
    assert err <= bound, f"{what}: max |diff| {err:.3e} > {bound:.3e}"


@pytest.mark.parametrize("cfg,partition", [(3, 0), (1, 2)])
def test_static_scratch_matches_the_workspace_entry_twice(cfg, partition):
    import paged_kv_cache_227_gb300 as pa
    torch.cuda.set_device(0)
    c = GpuCase(cfg)
    pool = c.pool()
    q, bt, sl = c.dev("q"), c.tables_dev(), c.lens_dev("ctx")
    ref = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    pa.pa_decode_split(pool, q, bt, sl, c.case.scale, ref, partition_blocks=partition)
    for call in range(2):
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        assert _call_static(pa, pool, q, bt, sl, c.case.scale, out, partition) == pa.PA_OK
        code, detail = pa.pa_check(pool)
        assert code == pa.PA_OK, (pa.strerror(code), detail)
        _close(out, ref, f"config {cfg}, call {call + 1}")
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
