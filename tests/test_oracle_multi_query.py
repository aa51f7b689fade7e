"""Pins for the fp64 multi-token-query oracle (several new tokens per
sequence, causal within them): torch fp64 SDPA with an explicit causal mask on
the un-paged cache, the single-token decode oracle, exact decoding, a closed
form and a pure-Python brute force."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle.multi_query import decode16, paged_multi_query

from ._util import BS, bits, dtype_code, pool_from_dense, to_bits

DTYPES = [torch.float16, torch.bfloat16]


def make(seed, lens, news, Hq, Hkv, dt, d=128, extra=3):
    g = torch.Generator().manual_seed(seed)
    q_start = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    q = torch.randn(int(q_start[-1]), Hq, d, generator=g).to(dt)
    dk = [torch.randn(Hkv, L, d, generator=g).to(dt) for L in lens]
    dv = [torch.randn(Hkv, L, d, generator=g).to(dt) for L in lens]
    nbs = [max(1, -(-L // BS)) for L in lens]
    N = sum(nbs) + extra
    perm = torch.randperm(N, generator=g).numpy()
    kp, tables = pool_from_dense([x.double().numpy() for x in dk], nbs, N, perm)
    vp, _ = pool_from_dense([x.double().numpy() for x in dv], nbs, N, perm)
    _, kb = to_bits(kp, dt)
    _, vb = to_bits(vp, dt)
    return dict(q=q, dk=dk, dv=dv, kp=kb, vp=vb, tables=tables, lens=np.array(lens, np.int32), q_start=q_start)


def test_decode16_matches_the_c_decoders_on_every_pattern():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    lib = oracle.attention._load()
    sample = pats[::97]
    for code, fn in ((0, lib.oracle_fp16_to_double), (1, lib.oracle_bf16_to_double)):
        got = decode16(sample, code)
        ref = np.array([fn(int(p)) for p in sample])
        same = (got == ref) | (np.isnan(got) & np.isnan(ref))
        assert same.all()


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("Hq,Hkv", [(12, 2), (32, 8), (4, 4)])
def test_matches_torch_sdpa_with_causal_mask(dt, Hq, Hkv):
    lens, news = [5, 16, 40, 100, 33], [5, 3, 16, 1, 7]
    c = make(11 + Hq, lens, news, Hq, Hkv, dt)
    scale = 1 / math.sqrt(128)
    got = paged_multi_query(bits(c["q"]), c["kp"], c["vp"], dtype_code(dt), c["tables"], c["lens"], c["q_start"],
                            scale)
    for i, (L, T) in enumerate(zip(lens, news)):
        r0 = c["q_start"][i]
        qi = c["q"][r0:r0 + T].double().permute(1, 0, 2)[None]      # [1][Hq][T][d]
        ki = c["dk"][i].double()[None]                               # [1][Hkv][L][d]
        vi = c["dv"][i].double()[None]
        mask = torch.arange(L)[None, :] <= (L - T + torch.arange(T))[:, None]   # [T][L]
        ref = F.scaled_dot_product_attention(qi, ki, vi, attn_mask=mask, scale=scale, enable_gqa=True)
        np.testing.assert_allclose(got[r0:r0 + T], ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_one_new_token_is_the_decode_oracle():
    dt = torch.bfloat16
    lens = [1, 17, 64, 300]
    c = make(5, lens, [1] * len(lens), 32, 8, dt)
    scale = 0.09
    got = paged_multi_query(bits(c["q"]), c["kp"], c["vp"], 1, c["tables"], c["lens"], c["q_start"], scale)
    ref = oracle.paged_decode(bits(c["q"]), c["kp"], c["vp"], 1, c["tables"], c["lens"], scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


def test_first_token_of_a_fresh_sequence_returns_its_value():
    dt = torch.float16
    c = make(2, [20], [20], 4, 2, dt)
    got = paged_multi_query(bits(c["q"]), c["kp"], c["vp"], 0, c["tables"], c["lens"], c["q_start"], 0.3)
    v0 = c["dv"][0][:, 0, :].double().numpy()           # [Hkv][d]
    np.testing.assert_array_equal(got[0], np.repeat(v0, 2, axis=0))


def test_brute_force_tiny():
    # pure-Python loops: 2 sequences, width 8, block 4 (pool laid out by hand)
    rng = np.random.default_rng(1)
    bs, d, Hq, Hkv = 4, 8, 2, 1
    lens, news = [6, 3], [2, 3]
    tables = np.array([[2, 0], [1, -1]], np.int32)
    kp = rng.standard_normal((3, Hkv, bs, d)).astype(np.float16)
    vp = rng.standard_normal((3, Hkv, bs, d)).astype(np.float16)
    q = rng.standard_normal((5, Hq, d)).astype(np.float16)
    q_start = np.array([0, 2, 5], np.int32)
    got = paged_multi_query(q.view(np.uint16), kp.view(np.uint16), vp.view(np.uint16), 0, tables,
                            np.array(lens, np.int32), q_start, 0.5)
    for i in range(2):
        for t in range(news[i]):
            r = q_start[i] + t
            p = lens[i] - news[i] + t
            for h in range(Hq):
                s = []
                for j in range(p + 1):
                    kk = kp[tables[i][j // bs], 0, j % bs].astype(float)
                    s.append(0.5 * sum(float(q[r, h, x]) * kk[x] for x in range(d)))
                m = max(s)
                w = [math.exp(x - m) for x in s]
                o = [sum(w[j] * float(vp[tables[i][j // bs], 0, j % bs, x]) for j in range(p + 1)) / sum(w)
                     for x in range(d)]
                np.testing.assert_allclose(got[r, h], o, rtol=0, atol=1e-12)
