"""The Python binding only marshals arguments: on host tensors it refuses to
run (there is no CPU path), and non-tensors are refused before anything
reaches the library.  No GPU needed: a stand-in pool object carries
the attributes the binding reads."""
import types

import pytest
import torch

import paged_kv_cache_227_gb300 as pa


def fake_pool(dtype=torch.bfloat16, n_kv_heads=2):
    return types.SimpleNamespace(handle=None, dtype=dtype, n_kv_heads=n_kv_heads)


def host_args(B=2, Hq=4, W=3, dtype=torch.bfloat16):
    return (torch.zeros(B, Hq, 128, dtype=dtype), torch.zeros(B, W, dtype=torch.int32),
            torch.ones(B, dtype=torch.int32), torch.zeros(B, Hq, 128, dtype=torch.float32))


@pytest.mark.parametrize("call", ["pa_decode", "pa_decode_split", "pa_decode_split_static"])
def test_host_tensors_are_refused(call):
    q, bt, sl, out = host_args()
    with pytest.raises(ValueError, match="must be on the GPU"):
        getattr(pa, call)(fake_pool(), q, bt, sl, 0.1, out)


def test_append_and_fused_step_refuse_host_tensors():
    q, bt, sl, out = host_args()
    kn = torch.zeros(2, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="must be on the GPU"):
        pa.pa_cache_append(fake_pool(), kn, kn, torch.zeros(2, dtype=torch.int64))
    with pytest.raises(ValueError, match="must be on the GPU"):
        pa.pa_append_decode(fake_pool(), q, kn, kn, bt, sl, 0.1, out)
    with pytest.raises(ValueError, match="must be on the GPU"):
        pa.pa_decode_multi(fake_pool(), q, torch.zeros(3, dtype=torch.int32), bt, sl, 0.1, out)


def test_non_tensors_are_refused_before_the_library():
    q, bt, sl, out = host_args()
    with pytest.raises(TypeError, match="must be a torch.Tensor"):
        pa.pa_decode(fake_pool(), [1, 2], bt, sl, 0.1, out)
    with pytest.raises(TypeError, match="must be a torch.Tensor"):
        pa.pa_cache_append(fake_pool(), None, None, torch.zeros(1, dtype=torch.int64))
