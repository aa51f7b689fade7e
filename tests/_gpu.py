"""Helpers for the GPU parity tests: case construction with NaN sentinels,
oracle references, tolerance checks."""
import os

import numpy as np
import torch

import oracle
from oracle.allocator import ReferenceAllocator
from workloads import CONFIGS, build_tables, make_case

NAN_BITS = {torch.float16: 0x7E00, torch.bfloat16: 0x7FC0}
ORACLE_THREADS = max(1, len(os.sched_getaffinity(0)))
ABS_TOL, REL_TOL = 2e-3, 1e-2


def bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a, dtype, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype).to(device)


def used_slots(tables, lens, num_blocks):
    """[N][16] mask of slots holding one of the first lens[i] tokens."""
    used = np.zeros((num_blocks, 16), dtype=bool)
    for i, L in enumerate(np.asarray(lens).tolist()):
        if L <= 0:
            continue
        nb = -(-L // 16)
        used[tables[i, :nb - 1]] = True
        used[tables[i, nb - 1], :L - 16 * (nb - 1)] = True
    return used


class GpuCase:
    """One config's inputs on host (bit patterns) and device.  Every pool slot
    that holds no token of the step (after its append) is set to NaN."""

    def __init__(self, cfg, seed=None, lens=None, sentinel=True, device="cuda"):
        cfg = CONFIGS[cfg] if isinstance(cfg, int) else cfg
        self.cfg = cfg
        self.case = make_case(cfg, seed=seed, lens=lens)
        c = self.case
        self.dtype = cfg.torch_dtype
        self.code = 0 if self.dtype == torch.float16 else 1
        self.alloc = ReferenceAllocator(c.num_blocks, 16, c.free_order)
        self.tables, self.slots, self.cows, self.dec_lens = build_tables(c, self.alloc)
        self.ctx_lens = (self.dec_lens - 1).astype(np.int32)
        self.kp, self.vp = bits(c.k_pool), bits(c.v_pool)
        if sentinel:
            unused = ~used_slots(self.tables, self.dec_lens, c.num_blocks)
            nan = np.uint16(NAN_BITS[self.dtype])
            self.kp.transpose(0, 2, 1, 3)[unused] = nan
            self.vp.transpose(0, 2, 1, 3)[unused] = nan
        self.q, self.kn, self.vn = bits(c.q), bits(c.k_new), bits(c.v_new)
        self.device = torch.device(device)

    # device tensors
    def pool(self):
        import paged_kv_cache_227_gb300 as pa
        p = pa.Pool(self.case.num_blocks, self.cfg.n_kv_heads, self.dtype)
        p.k.copy_(from_bits(self.kp, self.dtype))
        p.v.copy_(from_bits(self.vp, self.dtype))
        return p

    def dev(self, name):
        arr = {"q": self.q, "k_new": self.kn, "v_new": self.vn}[name]
        return from_bits(arr, self.dtype)

    def tables_dev(self):
        return torch.from_numpy(self.tables).to(self.device)

    def lens_dev(self, which="dec"):
        return torch.from_numpy(self.dec_lens if which == "dec" else self.ctx_lens).to(self.device)

    def slots_dev(self):
        return torch.from_numpy(self.slots).to(self.device)

    # oracle references
    def appended_pools(self):
        return oracle.cache.append(self.kp, self.vp, self.kn, self.vn, self.slots)

    def vmax(self):
        """max |v| over the V values the step attends (pool after the append;
        the NaN sentinels of unused slots excluded)."""
        _, vp = self.appended_pools()
        v = torch.from_numpy(np.ascontiguousarray(vp).view(np.int16)).view(self.dtype).float().abs()
        v = v[torch.isfinite(v)]
        return float(v.max()) if v.numel() else 0.0

    def reference(self, after_append=True, rows=None):
        if after_append:
            kp, vp = self.appended_pools()
            lens = self.dec_lens
        else:
            kp, vp, lens = self.kp, self.vp, self.ctx_lens
        return oracle.paged_decode(self.q, kp, vp, self.code, self.tables, lens, self.case.scale,
                                   rows=rows, threads=ORACLE_THREADS)


def assert_close(out, ref, what=""):
    """The parity bar: max |err| <= 2e-3 absolute and <= 1e-2 * max |ref|."""
    got = out.detach().float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref).max()
    bound = min(ABS_TOL, REL_TOL * np.abs(ref).max()) if ref.size else ABS_TOL
    assert err <= bound, f"{what}: max |err| {err:.3e} > {bound:.3e}"
    return err


def fp32_floor(vmax):
    """Absolute error floor of the native 16-bit check: the fp32 arithmetic
    (2e-6), plus the value product's weights, which the tensor-core path
    carries as a high and a low 16-bit half, i.e. to 2^-18 relative: summed
    with weights that add up to 1 over values |v| <= vmax, that is at most
    2^-18 * vmax per output."""
    return 2e-6 + 2.0 ** -18 * float(vmax)


def assert_within_one_ulp16(out16, ref, dtype, what="", vmax=None):
    """Native 16-bit output: |out - RN16(ref)| <= 1 ulp of RN16(ref) + fp32_floor(vmax).
    The absolute term covers outputs so small that one 16-bit ulp (down to
    2^-24 for fp16) is below the kernel's own error (fp32 accumulation and
    17-bit weights on the tensor-core value path).  vmax: max |v| of the
    attended values (required)."""
    assert vmax is not None, "pass the case's max |v| (GpuCase.vmax())"
    r16 = torch.from_numpy(ref).to(torch.float32).to(dtype).to(torch.float64).numpy()
    got = out16.detach().cpu().to(torch.float64).numpy().reshape(ref.shape)
    mant = 7 if dtype == torch.bfloat16 else 10
    min_exp = -126 if dtype == torch.bfloat16 else -14
    e = np.floor(np.log2(np.maximum(np.abs(r16), 2.0 ** min_exp)))
    ulp = 2.0 ** (e - mant)
    bad = np.abs(got - r16) > ulp + fp32_floor(vmax)
    assert not bad.any(), f"{what}: {bad.sum()} elements more than 1 ulp from RN16(ref)"
